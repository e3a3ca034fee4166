// WY representation forward of the gated delta rule (page
// "fla/ops/gated_delta_rule/backends/triton_ascend/wy_fast.py": recompute_w_u_fwd_kernel_npu, launched by
// recompute_w_u_fwd_npu) on CUDA cores in fp32.  Per chunk of BT rows (chunks start at each sequence's
// first row) and value head hv, with key head hv / (HV / H):
//     u = A (v * beta),   w = A (k * beta * 2^g)
// where A is the chunk's BT x BT matrix, stored row by row in A [rows, HV, BT] and used as a full square.
//
// One CTA per (chunk, value head).  The chunk's A goes to shared memory transposed (A^T[s][t], so that a
// warp's rows are broadcast loads); the operand block X = [k*beta*2^g | v*beta] (K + V columns) streams in
// stages of 16 rows: raw k | v rows arrive by asynchronous 16-byte copies two stages ahead, and each stage is
// scaled into fp32 just before it is multiplied.  Each warp owns BT / 4
// rows and half of the columns, each lane the columns {l + 32 q} of it: a thread accumulates its rows x
// columns over the BT columns of A with packed two-wide fmas (two rows at a time) and stores straight from
// registers (a warp writes contiguous row segments of w and u).  Rows past the end of a sequence are
// zero in X and in A^T, so they add nothing, and they are not stored.
#include <atomic>

#include "gla_internal.h"
#include "io.cuh"

namespace gla {

namespace {

constexpr int NTW = 256;   // threads per CTA (8 warps)

template <typename Tin, int BT, int KV>
struct WySmem {
    static constexpr int SB = 16;                   // rows of X per pipeline stage
    static constexpr int ATP = BT + 4;              // padded row of A^T
    static constexpr int EPF = 4 / sizeof(Tin);     // input elements per float of raw storage
    static constexpr int AT = 0;                    // [BT][ATP] A^T (fp32)
    static constexpr int X = AT + BT * ATP;         // [SB][KV] gated operands of the current stage (fp32)
    static constexpr int F = X + SB * KV;           // [2][BT] row factors: beta 2^g (k part), beta (v part)
    static constexpr int RA = F + 2 * BT;           // [BT][BT] raw A (input type)
    static constexpr int RX = RA + BT * BT / EPF;   // [2][SB][KV] raw k | v rows of two stages (input type)
    static constexpr int FLOATS = RX + 2 * SB * KV / EPF;
};

// 16-byte asynchronous global -> shared copy (no registers involved); groups complete in commit order
__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T>
__device__ __forceinline__ float widen1(T x);
template <>
__device__ __forceinline__ float widen1<float>(float x)
{
    return x;
}
template <>
__device__ __forceinline__ float widen1<__nv_bfloat16>(__nv_bfloat16 x)
{
    return __bfloat162float(x);
}
template <>
__device__ __forceinline__ float widen1<__half>(__half x)
{
    return __half2float(x);
}

// Packed pairs of fp32 in one 64-bit register: d = a * b + d lane-wise, each half rounded like fmaf.
__device__ __forceinline__ void ffma2(unsigned long long &d, unsigned long long a, unsigned long long b)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

__device__ __forceinline__ unsigned long long pack2(float x, float y)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}

__device__ __forceinline__ float2 unpack2(unsigned long long r)
{
    float2 x;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x.x), "=f"(x.y) : "l"(r));
    return x;
}

template <typename T>
__device__ __forceinline__ T to_out(float x);

template <>
__device__ __forceinline__ float to_out<float>(float x)
{
    return x;
}

template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float x)
{
    return __float2bfloat16_rn(x);
}

template <typename Tin, typename Tout, int BT, int K, int V>
__global__ void __launch_bounds__(NTW, 2) wy_fwd_ffma(WyArgs a)
{
    constexpr int KV = K + V;
    using L = WySmem<Tin, BT, KV>;
    constexpr int SB = L::SB, NS = BT / SB, EPC = 16 / (int)sizeof(Tin);   // elements per 16-byte copy
    extern __shared__ __align__(16) float sm[];
    float *At = sm + L::AT, *X = sm + L::X, *F = sm + L::F;
    Tin *RA = reinterpret_cast<Tin *>(sm + L::RA), *RX = reinterpret_cast<Tin *>(sm + L::RX);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hv = blockIdx.x, j = blockIdx.y, HV = a.HV, hk = hv / (HV / a.H);
    int bos, eos;
    if (a.table) {
        const int4 e = a.table[j];
        if (e.x < 0)
            return;
        bos = e.z;
        eos = e.w;
    } else {
        const int n = j / a.NT, p = j - n * a.NT;
        bos = n * a.T + p * BT;
        eos = min(bos + BT, n * a.T + a.T);
    }
    const int m = eos - bos;
    if (m <= 0)
        return;
    const Tin *A = static_cast<const Tin *>(a.A), *beta = static_cast<const Tin *>(a.beta);
    const Tin *k = static_cast<const Tin *>(a.k), *v = static_cast<const Tin *>(a.v);
    // ---- asynchronous copies of the raw rows: A's valid rows (group 0), then the k | v rows of stages 0 and
    //      1 (one group each); rows past the end of the sequence are not copied (they become zeros below)
    for (int e = tid; e < BT * (BT / EPC); e += NTW) {
        const int t = e / (BT / EPC), c = (e - t * (BT / EPC)) * EPC;
        if (t < m)
            cp_async16(RA + t * BT + c, A + ((size_t)(bos + t) * HV + hv) * BT + c);
    }
    cp_commit();
    auto copy_stage = [&](int st, int buf) {
        constexpr int UK = K / EPC, UR = KV / EPC;   // copies per row: k part, whole row
        for (int e = tid; e < SB * UR; e += NTW) {
            const int r = e / UR, uc = e - r * UR, s = st * SB + r;
            if (s < m) {
                const size_t row = (size_t)(bos + s);
                Tin *dst = RX + (buf * SB + r) * KV + uc * EPC;
                if (uc < UK)
                    cp_async16(dst, k + (row * a.H + hk) * K + uc * EPC);
                else
                    cp_async16(dst, v + (row * HV + hv) * V + (uc - UK) * EPC);
            }
        }
        cp_commit();
    };
    copy_stage(0, 0);
    if (NS > 1)
        copy_stage(1, 1);
    // row factors (plain loads while the copies fly)
    if (tid < BT) {
        float fb = 0.f, fg = 0.f;
        if (tid < m) {
            const size_t row = (size_t)(bos + tid);
            fb = IO<Tin>::load1(beta + row * HV + hv);
            fg = a.g ? fb * exp2f(a.g[row * HV + hv]) : fb;
        }
        F[tid] = fg;
        F[BT + tid] = fb;
    }
    if (NS > 1)
        cp_wait<1>();   // A and stage 0
    else
        cp_wait<0>();
    __syncthreads();
    for (int e = tid; e < BT * BT; e += NTW) {   // A^T[s][t] = A[t][s] for valid t and s, zero elsewhere
        const int s = e / BT, t = e - s * BT;
        At[s * L::ATP + t] = (t < m && s < m) ? widen1<Tin>(RA[t * BT + s]) : 0.f;
    }
    // ---- (A X)[t][c]: warp w computes rows [WR (w % 4), WR (w % 4) + WR) and the column half w / 4; lane l
    //      the columns {l + 32 q} of that half, two rows per packed fma.  X = [k * beta * 2^g | v * beta]
    //      one stage of SB rows at a time, scaled from the raw copies while stage st + 2's copies fly.
    constexpr int WR = BT / 4;                       // rows per warp
    constexpr int CPW = KV / 2, CQ = CPW / 32;       // columns per warp, columns per lane
    unsigned long long acc[WR / 2][CQ];   // rows (2 r, 2 r + 1) of column q, packed
#pragma unroll
    for (int r = 0; r < WR / 2; ++r)
#pragma unroll
        for (int q = 0; q < CQ; ++q)
            acc[r][q] = 0ull;
    const int t0 = (warp & 3) * WR, cw = (warp >> 2) * CPW;
    for (int st = 0; st < NS; ++st) {
        if (st > 0) {   // stage st's copies: all groups but the most recent one if a later stage is in flight
            if (st + 1 < NS)
                cp_wait<1>();
            else
                cp_wait<0>();
        }
        __syncthreads();   // copies visible; every warp done with the previous stage's X (and A^T written)
        const Tin *R = RX + (st & 1) * SB * KV;
        for (int e = tid; e < SB * KV; e += NTW) {   // X = raw row * factor, zero past the end
            const int r = e / KV, c = e - r * KV, s = st * SB + r;
            X[e] = s < m ? widen1<Tin>(R[e]) * F[(c < K ? 0 : BT) + s] : 0.f;
        }
        __syncthreads();
        if (st + 2 < NS)
            copy_stage(st + 2, st & 1);   // the raw buffer of stage st is free again
#pragma unroll 2
        for (int sl = 0; sl < SB; ++sl) {
            const int s = st * SB + sl;
            unsigned long long av[WR / 2];   // A^T[s][t0 + 2 r], A^T[s][t0 + 2 r + 1]
#pragma unroll
            for (int r = 0; r < WR; r += 4) {
                const ulonglong2 x4 = *reinterpret_cast<const ulonglong2 *>(At + s * L::ATP + t0 + r);
                av[r / 2] = x4.x;
                av[r / 2 + 1] = x4.y;
            }
            unsigned long long xq[CQ];
#pragma unroll
            for (int q = 0; q < CQ; ++q) {
                const float x = X[sl * KV + cw + lane + 32 * q];
                xq[q] = pack2(x, x);
            }
#pragma unroll
            for (int r = 0; r < WR / 2; ++r)
#pragma unroll
                for (int q = 0; q < CQ; ++q)
                    ffma2(acc[r][q], av[r], xq[q]);
        }
    }
    // ---- store valid rows: columns < K go to w, the rest to u
    Tout *w = static_cast<Tout *>(a.w), *u = static_cast<Tout *>(a.u);
#pragma unroll
    for (int r = 0; r < WR; ++r) {
        const int t = t0 + r;
        if (t >= m)
            continue;
        const size_t row = (size_t)(bos + t);
#pragma unroll
        for (int q = 0; q < CQ; ++q) {
            const int c = cw + lane + 32 * q;
            const float2 pr = unpack2(acc[r / 2][q]);
            const float x = (r & 1) ? pr.y : pr.x;
            if (c < K)
                w[(row * HV + hv) * K + c] = to_out<Tout>(x);
            else
                u[(row * HV + hv) * V + (c - K)] = to_out<Tout>(x);
        }
    }
}

template <typename Tin, typename Tout, int BT, int K, int V>
cudaError_t launch_wy_t(const WyArgs &a, int J, cudaStream_t s)
{
    const size_t bytes = sizeof(float) * WySmem<Tin, BT, K + V>::FLOATS;
    auto f = wy_fwd_ffma<Tin, Tout, BT, K, V>;
    static std::atomic<uint64_t> ready{0};   // per-device shared-memory opt-in, done once
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (!(ready.load(std::memory_order_acquire) & (1ull << (dev & 63)))) {
        if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes)) != cudaSuccess)
            return e;
        ready.fetch_or(1ull << (dev & 63), std::memory_order_release);
    }
    f<<<dim3(a.HV, J), NTW, bytes, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, typename Tout, int BT>
cudaError_t launch_wy_bt(const WyArgs &a, int J, cudaStream_t s)
{
    if (a.K == 64)
        return a.V == 64 ? launch_wy_t<Tin, Tout, BT, 64, 64>(a, J, s) : launch_wy_t<Tin, Tout, BT, 64, 128>(a, J, s);
    return a.V == 64 ? launch_wy_t<Tin, Tout, BT, 128, 64>(a, J, s) : launch_wy_t<Tin, Tout, BT, 128, 128>(a, J, s);
}

template <typename Tin, typename Tout>
cudaError_t launch_wy_io(const WyArgs &a, int J, cudaStream_t s)
{
    if (a.BT == 16)
        return launch_wy_bt<Tin, Tout, 16>(a, J, s);
    if (a.BT == 32)
        return launch_wy_bt<Tin, Tout, 32>(a, J, s);
    return launch_wy_bt<Tin, Tout, 64>(a, J, s);
}

}  // namespace

bool wy_supported(int dtype, int K, int V, int BT)
{
    return (dtype == GLA_F32 || dtype == GLA_BF16 || dtype == GLA_BF16_OBF16 || dtype == GLA_F16) &&
           (K == 64 || K == 128) && (V == 64 || V == 128) && (BT == 16 || BT == 32 || BT == 64);
}

cudaError_t launch_wy_fwd(const WyArgs &a, int J, int dtype, cudaStream_t s)
{
    if (dtype == GLA_F32)
        return launch_wy_io<float, float>(a, J, s);
    if (dtype == GLA_F16)
        return launch_wy_io<__half, float>(a, J, s);
    if (dtype == GLA_BF16_OBF16)
        return launch_wy_io<__nv_bfloat16, __nv_bfloat16>(a, J, s);
    return launch_wy_io<__nv_bfloat16, float>(a, J, s);
}

}  // namespace gla
