// TTT-linear forward (page "fla/ops/ttt/fused_chunk.py": fused_chunk_ttt_linear_fwd_kernel, then the
// norm_residual step of fused_chunk_ttt_linear) on CUDA cores in fp32.
//
// Per (sequence, head) the inner model is h [D][D], hb [D]; each mini-batch (chunk) of BT rows takes one
// gradient step of the loss 1/2 |LN(k h + hb) * w + b + k - v|^2 per row, in the dual form:
//   kh_i = k_i h + hb, xhat_i = LN(kh_i), g_i = (xhat_i w + b + k_i - v_i) w,
//   v2_i = rstd_i / D (D g_i - sum g_i - xhat_i sum(g_i xhat_i))                 (gradient wrt kh_i)
//   o_i  = scale q_i h + hb - eta_i sum_{j<=i} (scale q_i . k_j + 1) v2_j;  o_i += LN(o_i) w + b
//   h   -= eta_last sum_j k_j^T v2_j,  hb -= eta_last sum_j v2_j
// Rows past the end of a sequence do not take part (the page's kernel also sums the zero-padded rows of
// a partial last chunk into the hb update; here they do not exist).  One CTA per (sequence, head), the
// state in shared memory, serial over chunks like the page's kernel.
#include "gla_internal.h"
#include "io.cuh"

namespace gla {

namespace {

constexpr int NTT = 256;

template <int D, int BT>
struct TttSmem {
    static constexpr int S = 0;                 // [D][D] state
    static constexpr int HB = S + D * D;        // [D]
    static constexpr int Q = HB + D;            // [BT][D] q (scaled)
    static constexpr int K = Q + BT * D;        // [BT][D]
    static constexpr int VV = K + BT * D;       // [BT][D] v
    static constexpr int KH = VV + BT * D;      // [BT][D] k h + hb, later the outputs before the norm
    static constexpr int V2 = KH + BT * D;      // [BT][D] gradients wrt kh
    static constexpr int A = V2 + BT * D;       // [BT][BT] scale q k^T (masked) + 1
    static constexpr int E = A + BT * BT;       // [BT] eta
    static constexpr int W = E + BT;            // [D] LN weight
    static constexpr int B = W + D;             // [D] LN bias
    static constexpr int FLOATS = B + D;
};

// mean and 1/sqrt(var + eps) of x[0..D) with one warp (D / 32 values per lane)
template <int D>
__device__ __forceinline__ void warp_ln_stats(const float *x, float eps, float &mean, float &rstd)
{
    const int lane = threadIdx.x & 31;
    float s = 0.f;
#pragma unroll
    for (int c = lane; c < D; c += 32)
        s += x[c];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        s += __shfl_xor_sync(0xffffffffu, s, o);
    mean = s / D;
    float v = 0.f;
#pragma unroll
    for (int c = lane; c < D; c += 32)
        v = fmaf(x[c] - mean, x[c] - mean, v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    rstd = rsqrtf(v / D + eps);
}

template <typename Tin, int D, int BT>
__global__ void __launch_bounds__(NTT, 1) ttt_linear_fwd(TttArgs a)
{
    using L = TttSmem<D, BT>;
    extern __shared__ __align__(16) float sm[];
    float *S = sm + L::S, *HB = sm + L::HB, *Qs = sm + L::Q, *Ks = sm + L::K, *Vs = sm + L::VV;
    float *KH = sm + L::KH, *V2 = sm + L::V2, *As = sm + L::A, *Es = sm + L::E, *Ws = sm + L::W, *Bs = sm + L::B;
    const int nh = blockIdx.x, n = nh / a.H, h = nh - n * a.H, H = a.H, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    int bos, eos;
    if (a.cu) {
        bos = a.cu[n];
        eos = a.cu[n + 1];
        if (bos < 0 || eos < bos || eos > a.T) {   // bad offsets: report, leave this sequence untouched
            if (tid == 0 && h == 0)
                report(a.status, GLA_ERR_INVALID_ARG);
            return;
        }
    } else {
        bos = n * a.T;
        eos = bos + a.T;
    }
    const Tin *q = static_cast<const Tin *>(a.q), *k = static_cast<const Tin *>(a.k);
    const Tin *v = static_cast<const Tin *>(a.v);
    const size_t st = (size_t)n * H + h;
    for (int e = tid; e < D * D; e += NTT)
        S[e] = a.h0 ? a.h0[st * D * D + e] : 0.f;
    for (int c = tid; c < D; c += NTT) {
        HB[c] = a.hb0 ? a.hb0[st * D + c] : 0.f;
        Ws[c] = a.w[(size_t)h * D + c];
        Bs[c] = a.b[(size_t)h * D + c];
    }
    // thread mapping of the [BT][D] products: row i = tid / (NTT / BT), columns c = col0 + 32*m
    constexpr int TPR = NTT / BT, CPT = D / TPR;   // threads per row, columns per thread
    const int ri = tid / TPR, col0 = tid % TPR;
    __syncthreads();
    for (int r0 = bos; r0 < eos; r0 += BT) {
        const int len = min(BT, eos - r0);
        // ---- load the chunk (q scaled), eta
        for (int e = tid; e < BT * D / 4; e += NTT) {
            const int i = e / (D / 4), c4 = (e - i * (D / 4)) * 4;
            const size_t o = ((size_t)(r0 + i) * H + h) * D + c4;
            const bool in = i < len;
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            float4 x = in ? IO<Tin>::load4(q + o) : z;
            x.x *= a.scale;
            x.y *= a.scale;
            x.z *= a.scale;
            x.w *= a.scale;
            *reinterpret_cast<float4 *>(Qs + i * D + c4) = x;
            *reinterpret_cast<float4 *>(Ks + i * D + c4) = in ? IO<Tin>::load4(k + o) : z;
            *reinterpret_cast<float4 *>(Vs + i * D + c4) = in ? IO<Tin>::load4(v + o) : z;
        }
        if (tid < BT)
            Es[tid] = tid < len ? a.eta[(size_t)(r0 + tid) * H + h] : 0.f;
        __syncthreads();
        // ---- KH = k h + hb and the query readout q h + hb (the latter into V2 for now)
        {
            float acck[CPT], accq[CPT];
#pragma unroll
            for (int m = 0; m < CPT; ++m)
                acck[m] = accq[m] = HB[col0 + TPR * m];
            for (int kk = 0; kk < D; ++kk) {
                const float kv = Ks[ri * D + kk], qv = Qs[ri * D + kk];
#pragma unroll
                for (int m = 0; m < CPT; ++m) {
                    const float s = S[kk * D + col0 + TPR * m];
                    acck[m] = fmaf(kv, s, acck[m]);
                    accq[m] = fmaf(qv, s, accq[m]);
                }
            }
#pragma unroll
            for (int m = 0; m < CPT; ++m) {
                KH[ri * D + col0 + TPR * m] = acck[m];
                V2[ri * D + col0 + TPR * m] = accq[m];
            }
        }
        // ---- A = scale q k^T + 1 on and below the diagonal
        for (int e = tid; e < BT * BT; e += NTT) {
            const int i = e / BT, j = e - i * BT;
            float s = 0.f;
            if (j <= i)
                for (int kk = 0; kk < D; ++kk)
                    s = fmaf(Qs[i * D + kk], Ks[j * D + kk], s);
            As[e] = j <= i ? s + 1.f : 0.f;
        }
        __syncthreads();
        // ---- per row (one warp each): the gradient v2 of the inner loss wrt kh; the readout moves to KH
        for (int i = warp; i < BT; i += NTT / 32) {
            float *x = KH + i * D;
            float mean, rstd;
            warp_ln_stats<D>(x, a.eps, mean, rstd);
            float sg = 0.f, sgx = 0.f;
            float gv[D / 32], xh[D / 32];
#pragma unroll
            for (int m = 0; m < D / 32; ++m) {
                const int c = lane + 32 * m;
                xh[m] = (x[c] - mean) * rstd;
                gv[m] = i < len ? (xh[m] * Ws[c] + Bs[c] + Ks[i * D + c] - Vs[i * D + c]) * Ws[c] : 0.f;
                sg += gv[m];
                sgx = fmaf(gv[m], xh[m], sgx);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sg += __shfl_xor_sync(0xffffffffu, sg, o);
                sgx += __shfl_xor_sync(0xffffffffu, sgx, o);
            }
            __syncwarp();
#pragma unroll
            for (int m = 0; m < D / 32; ++m) {
                const int c = lane + 32 * m;
                const float readout = V2[i * D + c];
                x[c] = readout;   // KH row i now holds scale q_i h + hb
                V2[i * D + c] = rstd / D * (D * gv[m] - sg - xh[m] * sgx);
            }
        }
        __syncthreads();
        // ---- outputs: o_i = readout_i - eta_i sum_{j<=i} A_ij v2_j, then o_i += LN(o_i) w + b
        {
            float acc[CPT];
#pragma unroll
            for (int m = 0; m < CPT; ++m)
                acc[m] = 0.f;
            for (int j = 0; j <= ri; ++j) {
                const float aij = As[ri * BT + j];
#pragma unroll
                for (int m = 0; m < CPT; ++m)
                    acc[m] = fmaf(aij, V2[j * D + col0 + TPR * m], acc[m]);
            }
            const float ei = Es[ri];
            __syncthreads();   // every thread has read V2 rows it needs before KH is rewritten
#pragma unroll
            for (int m = 0; m < CPT; ++m)
                KH[ri * D + col0 + TPR * m] = fmaf(-ei, acc[m], KH[ri * D + col0 + TPR * m]);
        }
        __syncthreads();
        for (int i = warp; i < len; i += NTT / 32) {
            const float *x = KH + i * D;
            float mean, rstd;
            warp_ln_stats<D>(x, a.eps, mean, rstd);
            float *orow = a.o + ((size_t)(r0 + i) * H + h) * D;
#pragma unroll
            for (int m = 0; m < D / 32; ++m) {
                const int c = lane + 32 * m;
                orow[c] = x[c] + (x[c] - mean) * rstd * Ws[c] + Bs[c];
            }
        }
        // ---- state update with the last valid row's learning rate
        {
            const float el = Es[len - 1];
            for (int e = tid; e < D * D; e += NTT) {
                const int kk = e / D, c = e - kk * D;
                float s = 0.f;
                for (int j = 0; j < len; ++j)
                    s = fmaf(Ks[j * D + kk], V2[j * D + c], s);
                S[e] = fmaf(-el, s, S[e]);
            }
            for (int c = tid; c < D; c += NTT) {
                float s = 0.f;
                for (int j = 0; j < len; ++j)
                    s += V2[j * D + c];
                HB[c] = fmaf(-el, s, HB[c]);
            }
        }
        __syncthreads();
    }
    if (a.ht)
        for (int e = tid; e < D * D; e += NTT)
            a.ht[st * D * D + e] = S[e];
    if (a.hbt)
        for (int c = tid; c < D; c += NTT)
            a.hbt[st * D + c] = HB[c];
}

template <typename Tin, int D, int BT>
cudaError_t launch_t(const TttArgs &a, cudaStream_t s)
{
    const size_t bytes = sizeof(float) * TttSmem<D, BT>::FLOATS;
    auto f = ttt_linear_fwd<Tin, D, BT>;
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess)
        return e;
    f<<<a.N * a.H, NTT, bytes, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_tin(const TttArgs &a, cudaStream_t s)
{
    if (a.D == 64)
        return a.BT == 16 ? launch_t<Tin, 64, 16>(a, s) : launch_t<Tin, 64, 32>(a, s);
    return a.BT == 16 ? launch_t<Tin, 128, 16>(a, s) : launch_t<Tin, 128, 32>(a, s);
}

}  // namespace

cudaError_t launch_ttt_linear_fwd(const TttArgs &a, int dtype, cudaStream_t s)
{
    if (dtype == GLA_F32)
        return launch_tin<float>(a, s);
    if (dtype == GLA_F16)
        return launch_tin<__half>(a, s);
    return launch_tin<__nv_bfloat16>(a, s);
}

}  // namespace gla
