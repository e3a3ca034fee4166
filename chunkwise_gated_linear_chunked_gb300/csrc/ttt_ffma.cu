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
// a partial last chunk into the hb update; here they do not exist).
//
// GB300 layout of the work: one thread-block cluster of CL = D / 16 CTAs per (sequence, head).  CTA r of
// the cluster owns value columns [16 r, 16 r + 16) of h and hb, held in registers (thread (c, g) keeps
// h[g KG .. g KG + KG)[c]), so the products k h, q h and the update k^T v2 need no state traffic at all.
// What couples the columns is per row: the LayerNorm statistics of k h + hb and of the outputs, and the two
// sums of the loss gradient.  Each CTA reduces its 16 columns and pushes (mean, M2) or the two sums into
// every CTA of the cluster with distributed shared-memory stores; the row statistics are merged with the
// pairwise (Chan) update, in the same order in every CTA.  The scores A = scale q k^T are split by rows
// across the cluster the same way.  The pushes are asynchronous remote stores that complete transaction
// bytes on an mbarrier of the receiving CTA (one per exchanged quantity, one phase per mini-batch), so a
// CTA waits only for the data it reads, with no cluster-wide barrier or fence on the path.  Buffer reuse
// needs no extra handshake: a CTA can only push mini-batch t+1's values after it has received every CTA's
// last push of mini-batch t, which each CTA sends after a CTA-wide barrier that follows its reads of the
// buffers of t (the scores, read after that barrier, alternate between two buffers instead).  The next mini-batch's
// q, k, v are loaded into registers a whole mini-batch ahead and parked in a second shared-memory buffer.
#include "gla_internal.h"
#include "io.cuh"
#include "tc_ptx.cuh"

namespace gla {

namespace {

constexpr int NTT = 256;    // threads per CTA
constexpr int NCOL = 16;    // value columns of the inner model per CTA

template <int D, int BT>
struct TttLayout {
    static constexpr int CL = D / NCOL;             // CTAs per (sequence, head)
    static constexpr int KG = D / 16;               // rows of h per thread
    static constexpr int DP = D + 4;                // padded row of the q / k tiles
    static constexpr int RA = BT / CL;              // rows of A each CTA computes
    static constexpr int KSTR = 16 * NCOL + 16;     // reduction buffer: one kind (k h or q h) of one warp,
                                                    // one 16-row block at a time
    static constexpr int MB = 0;                    // 4 mbarriers (X1, X2, X3, AX), 8 floats
    static constexpr int QB = 8;                    // [2][BT][DP] q (scaled)
    static constexpr int KB = QB + 2 * BT * DP;     // [2][BT][DP] k
    static constexpr int VB = KB + 2 * BT * DP;     // [2][BT][NCOL] v (own columns)
    static constexpr int EB = VB + 2 * BT * NCOL;   // [2][BT] eta (0 past the end)
    static constexpr int RED = EB + 2 * BT;         // [8 warps][2 kinds][KSTR] partial products
    static constexpr int V2 = RED + 16 * KSTR;      // [BT][NCOL] gradient wrt k h + hb
    static constexpr int AX = V2 + BT * NCOL;       // [2][BT][BT] scale q k^T (rows from every CTA), by parity
    static constexpr int X1 = AX + 2 * BT * BT;       // [CL][BT] float2: (mean, M2) of k h + hb per CTA
    static constexpr int X2 = X1 + 2 * CL * BT;     // [CL][BT] float2: (sum g, sum g xhat) per CTA
    static constexpr int X3 = X2 + 2 * CL * BT;     // [CL][BT] float2: (mean, M2) of the outputs per CTA
    static constexpr int FLOATS = X3 + 2 * CL * BT;
    static_assert(BT % 16 == 0 && BT % CL == 0, "tile shape");
    static_assert((BT * D / 4) % NTT == 0, "prefetch split");
    static_assert(NTT % (RA * BT) == 0, "score split");
};

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t remote(const void *p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(tc::smem_u32(p)), "r"(rank));
    return r;
}

// asynchronous store to the same shared-memory offset in CTA `rank`, completing 4 (8) transaction bytes on
// that CTA's mbarrier `bar`
__device__ __forceinline__ void push(float *p, uint64_t *bar, uint32_t rank, float x)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(remote(p, rank)),
                 "r"(__float_as_uint(x)), "r"(remote(bar, rank))
                 : "memory");
}

__device__ __forceinline__ void push2(float *p, uint64_t *bar, uint32_t rank, float x, float y)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
                     remote(p, rank)),
                 "f"(x), "f"(y), "r"(remote(bar, rank))
                 : "memory");
}

// Wait for phase `parity` of the local mbarrier `bar` (fed by remote pushes: acquire at cluster scope).
// Bounded: after about tc::kWaitNs the CTA-wide abort word is set and every later wait returns at once, so
// the CTA runs its remaining mini-batches without waiting (its results are void) and reaches the end.
__device__ __forceinline__ void wait_push(uint64_t *bar, uint32_t parity, volatile int *abort)
{
    auto try_once = [&]() {
        uint32_t ok;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}\n"
                     : "=r"(ok)
                     : "r"(tc::smem_u32(bar)), "r"(parity), "r"(100000u)
                     : "memory");
        return ok != 0;
    };
    if (try_once())
        return;
    const unsigned long long t0 = tc::global_ns();
    while (!try_once()) {
        if (*abort)
            return;
        if (tc::global_ns() - t0 > tc::kWaitNs) {
            *abort = 1;
            return;
        }
    }
}

// two fp32 fused multiply-adds in one instruction (each rounded like fmaf)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// sum over the 16 lanes of a half warp
__device__ __forceinline__ float hsum(float x)
{
#pragma unroll
    for (int o = 8; o > 0; o >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Row mean and 1/sqrt(var + eps) from the (mean, M2) pairs of CL column groups of NCOL columns each.
template <int CL, int BT>
__device__ __forceinline__ void merge_stats(const float *xs, int i, float inv_d, float eps, float &mean, float &rstd)
{
    float m = 0.f;
#pragma unroll
    for (int r = 0; r < CL; ++r)
        m += xs[2 * (r * BT + i)];
    m *= 1.f / CL;
    float m2 = 0.f;
#pragma unroll
    for (int r = 0; r < CL; ++r) {
        const float d = xs[2 * (r * BT + i)] - m;
        m2 += fmaf((float)NCOL * d, d, xs[2 * (r * BT + i) + 1]);
    }
    mean = m;
    rstd = rsqrtf(fmaf(m2, inv_d, eps));
}

// The next mini-batch in registers: q (scaled), k as float4 units; v (own columns) and eta per row slot.
template <int D, int BT>
struct Prefetch {
    static constexpr int NPF = BT * D / 4 / NTT;
    float4 q[NPF], k[NPF];
    float v[BT / 16];
    float e;
};

template <typename Tin, int D, int BT>
__device__ __forceinline__ void prefetch(Prefetch<D, BT> &pf, const TttArgs &a, int r0, int nlen, int h, int c0)
{
    const int tid = threadIdx.x, H = a.H;
    const Tin *q = static_cast<const Tin *>(a.q), *k = static_cast<const Tin *>(a.k);
    const Tin *v = static_cast<const Tin *>(a.v);
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < Prefetch<D, BT>::NPF; ++m) {
        const int u = tid + NTT * m, i = u / (D / 4), c4 = (u - i * (D / 4)) * 4;
        const size_t o = ((size_t)(r0 + i) * H + h) * D + c4;
        const bool in = i < nlen;
        pf.q[m] = in ? IO<Tin>::load4(q + o) : z;
        pf.k[m] = in ? IO<Tin>::load4(k + o) : z;
    }
#pragma unroll
    for (int r = 0; r < BT / 16; ++r) {
        const int i = (tid >> 4) + 16 * r;
        pf.v[r] = i < nlen ? IO<Tin>::load1(v + ((size_t)(r0 + i) * H + h) * D + c0 + (tid & 15)) : 0.f;
    }
    pf.e = tid < nlen ? a.eta[(size_t)(r0 + tid) * H + h] : 0.f;
}

template <int D, int BT>
__device__ __forceinline__ void park(const Prefetch<D, BT> &pf, float *sm, int buf, float scale)
{
    using L = TttLayout<D, BT>;
    const int tid = threadIdx.x;
    float *Qs = sm + L::QB + buf * BT * L::DP, *Ks = sm + L::KB + buf * BT * L::DP;
#pragma unroll
    for (int m = 0; m < Prefetch<D, BT>::NPF; ++m) {
        const int u = tid + NTT * m, i = u / (D / 4), c4 = (u - i * (D / 4)) * 4;
        float4 x = pf.q[m];
        x.x *= scale;
        x.y *= scale;
        x.z *= scale;
        x.w *= scale;
        *reinterpret_cast<float4 *>(Qs + i * L::DP + c4) = x;
        *reinterpret_cast<float4 *>(Ks + i * L::DP + c4) = pf.k[m];
    }
#pragma unroll
    for (int r = 0; r < BT / 16; ++r)
        sm[L::VB + buf * BT * NCOL + ((tid >> 4) + 16 * r) * NCOL + (tid & 15)] = pf.v[r];
    if (tid < BT)
        sm[L::EB + buf * BT + tid] = pf.e;
}

template <typename Tin, int D, int BT>
__global__ void __launch_bounds__(NTT, 2) ttt_linear_fwd(TttArgs a)
{
    using L = TttLayout<D, BT>;
    constexpr int CL = L::CL, KG = L::KG, DP = L::DP, RA = L::RA, NR = BT / 16;
    constexpr uint32_t XBYTES = CL * BT * 8, ABYTES = BT * BT * 4;   // transaction bytes per phase
    extern __shared__ __align__(16) float sm[];
    __shared__ int abort_word;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, c = tid & 15, g = tid >> 4;
    const uint32_t rank = cluster_rank();
    const int nh = blockIdx.x / CL, n = nh / a.H, h = nh - n * a.H, H = a.H, c0 = (int)rank * NCOL;
    int bos, eos;
    if (a.cu) {
        bos = a.cu[n];
        eos = a.cu[n + 1];
        if (bos < 0 || eos < bos || eos > a.T) {   // bad offsets: report, leave this sequence untouched
            if (tid == 0 && h == 0 && rank == 0)
                report(a.status, GLA_ERR_INVALID_ARG);
            return;                                  // the whole cluster leaves here, before any exchange
        }
    } else {
        bos = n * a.T;
        eos = bos + a.T;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::MB);
    uint64_t *B1 = bars, *B2 = bars + 1, *B3 = bars + 2, *BA = bars + 3;
    volatile int *abort = &abort_word;
    if (tid == 0) {
        abort_word = 0;
        for (int i = 0; i < 4; ++i)
            tc::bar_init(bars + i, 1);
        tc::bar_fence_init();
        tc::bar_expect_tx(B1, XBYTES);
        tc::bar_expect_tx(B2, XBYTES);
        tc::bar_expect_tx(B3, XBYTES);
        tc::bar_expect_tx(BA, ABYTES);
    }
    const size_t st = (size_t)n * H + h;
    float hs[KG];                                    // h[g KG + u][c0 + c]
#pragma unroll
    for (int u = 0; u < KG; ++u)
        hs[u] = a.h0 ? a.h0[(st * D + g * KG + u) * D + c0 + c] : 0.f;
    float hb = a.hb0 ? a.hb0[st * D + c0 + c] : 0.f;
    const float wc = a.w[(size_t)h * D + c0 + c], bc = a.b[(size_t)h * D + c0 + c];
    const float inv_d = 1.f / D;
    Prefetch<D, BT> pf;
    if (bos < eos) {
        prefetch<Tin, D, BT>(pf, a, bos, min(BT, eos - bos), h, c0);
        park<D, BT>(pf, sm, 0, a.scale);
    }
    cluster_arrive();   // every CTA of the cluster is running, its mbarriers armed, the first mini-batch parked
    cluster_wait();
    float *RED = sm + L::RED, *V2 = sm + L::V2, *AX = sm + L::AX;
    float *X1 = sm + L::X1, *X2 = sm + L::X2, *X3 = sm + L::X3;
    int buf = 0;
    uint32_t par = 0;
    for (int r0 = bos; r0 < eos; r0 += BT, buf ^= 1, par ^= 1) {
        const int len = min(BT, eos - r0), nlen = min(BT, eos - r0 - BT);
        if (nlen > 0)
            prefetch<Tin, D, BT>(pf, a, r0 + BT, nlen, h, c0);
        const float *Qs = sm + L::QB + buf * BT * DP, *Ks = sm + L::KB + buf * BT * DP;
        const float *Vs = sm + L::VB + buf * BT * NCOL, *Es = sm + L::EB + buf * BT;
        // ---- this CTA's RA rows of A = scale q k^T, pushed to every CTA of the cluster
        {
            constexpr int SL = NTT / (RA * BT), NA = D / (4 * SL);
            const int sl = tid % SL, pr = tid / SL, ia = (int)rank * RA + pr % RA, j = pr / RA;
            float s = 0.f;
#pragma unroll
            for (int m = 0; m < NA; ++m) {
                const int kk = 4 * sl + 4 * SL * m;
                const float4 q4 = *reinterpret_cast<const float4 *>(Qs + ia * DP + kk);
                const float4 k4 = *reinterpret_cast<const float4 *>(Ks + j * DP + kk);
                s = fmaf(q4.x, k4.x, s);
                s = fmaf(q4.y, k4.y, s);
                s = fmaf(q4.z, k4.z, s);
                s = fmaf(q4.w, k4.w, s);
            }
#pragma unroll
            for (int o = SL / 2; o > 0; o >>= 1)
                s += __shfl_xor_sync(0xffffffffu, s, o);
            for (int dst = sl; dst < CL; dst += SL)
                push(AX + par * BT * BT + ia * BT + j, BA, dst, s);
        }
        // ---- per 16-row block: partial k h and q h over this thread's KG rows of h (the pair in one packed
        //      fma); the two lanes of a column pair split the kinds, the 8 warps are summed in shared memory;
        //      then rows (thread (i, c)): k h + hb, q h + hb and the local LayerNorm statistics of k h + hb
        float kh[NR], ro[NR];
#pragma unroll
        for (int rb = 0; rb < NR; ++rb) {
            if (rb > 0)
                __syncthreads();   // every thread has read the previous block's partial sums
            float2 acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float *kr = Ks + (rb * 16 + i) * DP + g * KG, *qr = Qs + (rb * 16 + i) * DP + g * KG;
                float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int u4 = 0; u4 < KG; u4 += 4) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(kr + u4);
                    const float4 q4 = *reinterpret_cast<const float4 *>(qr + u4);
                    s2 = ffma2(make_float2(k4.x, q4.x), make_float2(hs[u4], hs[u4]), s2);
                    s2 = ffma2(make_float2(k4.y, q4.y), make_float2(hs[u4 + 1], hs[u4 + 1]), s2);
                    s2 = ffma2(make_float2(k4.z, q4.z), make_float2(hs[u4 + 2], hs[u4 + 2]), s2);
                    s2 = ffma2(make_float2(k4.w, q4.w), make_float2(hs[u4 + 3], hs[u4 + 3]), s2);
                }
                acc[i] = s2;
            }
            const bool lo = lane < 16;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float keep = lo ? acc[i].x : acc[i].y, send = lo ? acc[i].y : acc[i].x;
                RED[(2 * warp + (lane >> 4)) * L::KSTR + i * NCOL + c] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
            }
            __syncthreads();
            const int il = tid >> 4, i = il + 16 * rb;
            float sk = hb, sq = hb;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                sk += RED[(2 * w) * L::KSTR + il * NCOL + c];
                sq += RED[(2 * w + 1) * L::KSTR + il * NCOL + c];
            }
            kh[rb] = sk;
            ro[rb] = sq;
            const float ml = hsum(sk) * (1.f / NCOL), d = sk - ml, m2 = hsum(d * d);
            if (c < CL)
                push2(X1 + 2 * ((int)rank * BT + i), B1, c, ml, m2);
        }
        if (nlen > 0)
            park<D, BT>(pf, sm, buf ^ 1, a.scale);
        wait_push(B1, par, abort);
        if (tid == 0)
            tc::bar_expect_tx(B1, XBYTES);
        // ---- gradient of the inner loss (needs the row sums of g and g xhat over all columns)
        float xh[NR], gv[NR], rs[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const int i = (tid >> 4) + 16 * r;
            float mean;
            merge_stats<CL, BT>(X1, i, inv_d, a.eps, mean, rs[r]);
            xh[r] = (kh[r] - mean) * rs[r];
            gv[r] = i < len ? (fmaf(xh[r], wc, bc) + Ks[i * DP + c0 + c] - Vs[i * NCOL + c]) * wc : 0.f;
            const float sg = hsum(gv[r]), sgx = hsum(gv[r] * xh[r]);
            if (c < CL)
                push2(X2 + 2 * ((int)rank * BT + i), B2, c, sg, sgx);
        }
        wait_push(B2, par, abort);
        if (tid == 0)
            tc::bar_expect_tx(B2, XBYTES);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const int i = (tid >> 4) + 16 * r;
            float sg = 0.f, sgx = 0.f;
#pragma unroll
            for (int q = 0; q < CL; ++q) {
                sg += X2[2 * (q * BT + i)];
                sgx += X2[2 * (q * BT + i) + 1];
            }
            V2[i * NCOL + c] = rs[r] * inv_d * (D * gv[r] - sg - xh[r] * sgx);
        }
        wait_push(BA, par, abort);   // before the barrier: no thread can still wait here when the next
        if (tid == 0)                // mini-batch's scores start arriving
            tc::bar_expect_tx(BA, ABYTES);
        __syncthreads();
        // ---- outputs before the norm: q h + hb - eta_i sum_{j<=i} (A_ij + 1) v2_j; local statistics
        const float *Ac = AX + par * BT * BT;
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const int i = (tid >> 4) + 16 * r;
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < BT; ++j)
                acc = fmaf(j <= i ? Ac[i * BT + j] + 1.f : 0.f, V2[j * NCOL + c], acc);
            ro[r] = fmaf(-Es[i], acc, ro[r]);
            const float ml = hsum(ro[r]) * (1.f / NCOL), d = ro[r] - ml, m2 = hsum(d * d);
            if (c < CL)
                push2(X3 + 2 * ((int)rank * BT + i), B3, c, ml, m2);
        }
        // ---- state update with the last valid row's learning rate (while the output statistics travel)
        {
            const float el = Es[len - 1];
            float2 acc[KG / 2];
            float sv = 0.f;
#pragma unroll
            for (int u = 0; u < KG / 2; ++u)
                acc[u] = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < BT; ++i) {
                const float v2 = V2[i * NCOL + c];
                const float *kr = Ks + i * DP + g * KG;
#pragma unroll
                for (int u4 = 0; u4 < KG; u4 += 4) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(kr + u4);
                    acc[u4 / 2] = ffma2(make_float2(k4.x, k4.y), make_float2(v2, v2), acc[u4 / 2]);
                    acc[u4 / 2 + 1] = ffma2(make_float2(k4.z, k4.w), make_float2(v2, v2), acc[u4 / 2 + 1]);
                }
                sv += v2;
            }
#pragma unroll
            for (int u = 0; u < KG / 2; ++u) {
                hs[2 * u] = fmaf(-el, acc[u].x, hs[2 * u]);
                hs[2 * u + 1] = fmaf(-el, acc[u].y, hs[2 * u + 1]);
            }
            hb = fmaf(-el, sv, hb);
        }
        wait_push(B3, par, abort);
        if (tid == 0)
            tc::bar_expect_tx(B3, XBYTES);
        // ---- o = x + LN(x) w + b
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const int i = (tid >> 4) + 16 * r;
            float mean, rstd;
            merge_stats<CL, BT>(X3, i, inv_d, a.eps, mean, rstd);
            if (i < len)
                a.o[((size_t)(r0 + i) * H + h) * D + c0 + c] = ro[r] + fmaf((ro[r] - mean) * rstd, wc, bc);
        }
    }
    if (*abort && (tid & 31) == 0)
        report(a.status, GLA_ERR_TIMEOUT);
    if (a.ht)
#pragma unroll
        for (int u = 0; u < KG; ++u)
            a.ht[(st * D + g * KG + u) * D + c0 + c] = hs[u];
    if (a.hbt && g == 0)
        a.hbt[st * D + c0 + c] = hb;
    cluster_arrive();   // no CTA leaves while a peer may still push into it
    cluster_wait();
}

template <typename Tin, int D, int BT>
cudaError_t launch_t(const TttArgs &a, cudaStream_t s)
{
    using L = TttLayout<D, BT>;
    const size_t bytes = sizeof(float) * L::FLOATS;
    auto f = ttt_linear_fwd<Tin, D, BT>;
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.N * a.H * L::CL));
    cfg.blockDim = dim3(NTT);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = L::CL;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, f, a);
    return e != cudaSuccess ? e : cudaGetLastError();
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
