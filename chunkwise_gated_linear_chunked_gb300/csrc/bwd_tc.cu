// Backward chunk sums on the tensor cores (bf16 inputs, K = 128; page "fla/ops/gla/fused_chunk.py":
// fused_chunk_gla_bwd_kernel, whose state and adjoint carries these sums feed):
//     dS = sum_t (k_t e^{G_l - G_t})^T v_t,    dR = scale sum_t (q_t e^{G_t})^T do_t,    G_l
// per chunk of C = 64 rows and head, with G the chunk-local inclusive cumsum of the gates (natural log).
//
// One CTA per (chunk, head).  Both products are D[k][v] = sum_t A[k][t] B[v][t] with tcgen05 kind::f16 MMAs
// (bf16 operands, fp32 accumulation in TMEM): M = 128 keys, N = V, K = the chunk's 64 rows in steps of 16.
// The A operands (k e^{G_l - G} and q e^{G}, fp32 on chip) are split into three bf16 terms x = x1 + x2 + x3
// (exact to fp32 rounding) and written transposed into 128-byte-swizzled K-major tiles; the B operands
// (v and do, bf16 already) are written transposed into one tile each.  Every input row of the chunk arrives
// first by 16-byte asynchronous copies (q, k, v, do, g: one memory latency per CTA); a thread owns one key,
// takes its cumsum from the staged gates and forms both gated operands.  dS is formed first; its tiles are
// reused for dR once the first MMA group has completed.  Rows past the end of a chunk are zero in every
// tile.  The epilogue reads TMEM (lane = key) and stores rows of dS and dR (fp32, [slot][H][K][V]).
#include <atomic>

#include "gla_internal.h"
#include "io.cuh"
#include "tc_ptx.cuh"

namespace gla {

namespace {

constexpr int CT = kChunk;   // 64 rows per chunk
constexpr int KT = 128;      // keys
constexpr int NTS = 256;     // threads per CTA

template <typename Tg, int V>
struct SumsSmem {
    static constexpr int AT = 0;                   // [3 terms] A^T tiles, 128 rows x 128 bytes each
    static constexpr int BT = AT + 3 * 16384;      // B^T tile, V rows x 128 bytes
    static constexpr int RQ = BT + V * 128;        // raw rows of the chunk: q [64][128] bf16
    static constexpr int RK = RQ + CT * KT * 2;    // k [64][128] bf16
    static constexpr int RV = RK + CT * KT * 2;    // v [64][V] bf16
    static constexpr int RD = RV + CT * V * 2;     // do [64][V] bf16
    static constexpr int RG = RD + CT * V * 2;     // g [64][128] (Tg)
    static constexpr int BAR = RG + CT * KT * (int)sizeof(Tg);
    static constexpr int TSLOT = BAR + 8;
    static constexpr int BYTES = TSLOT + 8;
};

__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}

template <typename T>
__device__ __forceinline__ float wide(T x);
template <>
__device__ __forceinline__ float wide<float>(float x)
{
    return x;
}
template <>
__device__ __forceinline__ float wide<__nv_bfloat16>(__nv_bfloat16 x)
{
    return __bfloat162float(x);
}

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// x (8 values of one key, rows 8j .. 8j+7) -> three bf16 terms, each stored as one 16-byte swizzled chunk
__device__ __forceinline__ void split3_store(unsigned char *tiles, int key, int j, const float (&x)[8])
{
    uint32_t p1[4], p2[4], p3[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 xx = make_float2(x[2 * q], x[2 * q + 1]);
        const __nv_bfloat162 x1 = __float22bfloat162_rn(xx);
        const float2 y1 = __bfloat1622float2(x1);
        const float2 r1 = make_float2(xx.x - y1.x, xx.y - y1.y);
        const __nv_bfloat162 x2 = __float22bfloat162_rn(r1);
        const float2 y2 = __bfloat1622float2(x2);
        const __nv_bfloat162 x3 = __float22bfloat162_rn(make_float2(r1.x - y2.x, r1.y - y2.y));
        p1[q] = *reinterpret_cast<const uint32_t *>(&x1);
        p2[q] = *reinterpret_cast<const uint32_t *>(&x2);
        p3[q] = *reinterpret_cast<const uint32_t *>(&x3);
    }
    const uint32_t off = tc::sw128(key, 8 * j);
    *reinterpret_cast<uint4 *>(tiles + 0 * 16384 + off) = make_uint4(p1[0], p1[1], p1[2], p1[3]);
    *reinterpret_cast<uint4 *>(tiles + 1 * 16384 + off) = make_uint4(p2[0], p2[1], p2[2], p2[3]);
    *reinterpret_cast<uint4 *>(tiles + 2 * 16384 + off) = make_uint4(p3[0], p3[1], p3[2], p3[3]);
}

template <typename Tg, int V>
__global__ void __launch_bounds__(NTS, 1) bwd_chunk_sums_tc(BwdArgs a)
{
    using L = SumsSmem<Tg, V>;
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char *sm = smraw + ((1024u - (tc::smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + L::TSLOT);
    const __nv_bfloat16 *Rq = reinterpret_cast<const __nv_bfloat16 *>(sm + L::RQ);
    const __nv_bfloat16 *Rk = reinterpret_cast<const __nv_bfloat16 *>(sm + L::RK);
    const Tg *Rg = reinterpret_cast<const Tg *>(sm + L::RG);
    const int j = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int n, bos, eos;
    if (a.table) {
        const int4 e = a.table[j];
        if (e.x < 0)
            return;
        n = e.x;
        bos = e.z;
        eos = e.w;
    } else {
        n = j / a.NC;
        const int c = j - n * a.NC;
        bos = n * a.T + c * CT;
        eos = min(bos + CT, n * a.T + a.T);
    }
    const int len = eos - bos, H = a.H;
    const size_t rb = row_head(bos, h, H, a.T, a.hf);   // row t of the chunk: row-head index rb + t * rs
    const int rs = a.hf ? 1 : H;
    // ---- every valid row of q, k, v, do, g by 16-byte asynchronous copies (one latency for all of them)
    {
        const char *srcs[5] = {static_cast<const char *>(a.q), static_cast<const char *>(a.k),
                               static_cast<const char *>(a.v), static_cast<const char *>(a.dout),
                               static_cast<const char *>(a.g)};
        const int rowb[5] = {KT * 2, KT * 2, V * 2, V * 2, KT * (int)sizeof(Tg)};   // bytes per row
        const int dsto[5] = {L::RQ, L::RK, L::RV, L::RD, L::RG};
#pragma unroll
        for (int x = 0; x < 5; ++x) {
            const int per = rowb[x] / 16;
            for (int e = tid; e < CT * per; e += NTS) {
                const int t = e / per, c = e - t * per;
                if (t < len)
                    cp_async16(sm + dsto[x] + t * rowb[x] + 16 * c, srcs[x] + (rb + (size_t)t * rs) * rowb[x] + 16 * c);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    if (tid == 0) {
        tc::bar_init(bar, 1);
        tc::bar_fence_init();
    }
    if (warp == 0)
        tc::tmem_alloc(tslot, 2 * V);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;
    // ---- thread: key = tid % 128, row groups jj = tid / 128 + 2 i (i < 4).  Cumsum of its key from the raw
    //      gates (twice: the total first), then k e^{G_l - G} (three terms, to the A tiles) and q e^{G} (kept)
    const int key = tid & 127, j0 = tid >> 7;
    float gl = 0.f;
    for (int t = 0; t < len; ++t)
        gl += wide<Tg>(Rg[t * KT + key]);
    float xq[4][8];
    {
        float run = 0.f;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            float xk[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = 8 * jj + u;
                const bool in = t < len;
                run += in ? wide<Tg>(Rg[t * KT + key]) : 0.f;
                if ((jj & 1) == j0) {
                    xk[u] = in ? __bfloat162float(Rk[t * KT + key]) * expf(gl - run) : 0.f;
                    xq[jj >> 1][u] = in ? __bfloat162float(Rq[t * KT + key]) * expf(run) : 0.f;
                }
            }
            if ((jj & 1) == j0)
                split3_store(sm + L::AT, key, jj, xk);
        }
    }
    // v^T: task (value column c, row group jj), from the raw rows
    auto write_bt = [&](int roff) {
        const unsigned short *R = reinterpret_cast<const unsigned short *>(sm + roff);
        for (int e = tid; e < V * 8; e += NTS) {
            const int jj = e / V, c = e - jj * V;
            uint32_t p[4];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                const int t0 = 8 * jj + 2 * qq;
                const uint32_t lo = t0 < len ? R[t0 * V + c] : 0u;
                const uint32_t hi = t0 + 1 < len ? R[(t0 + 1) * V + c] : 0u;
                p[qq] = lo | (hi << 16);
            }
            *reinterpret_cast<uint4 *>(sm + L::BT + tc::sw128(c, 8 * jj)) = make_uint4(p[0], p[1], p[2], p[3]);
        }
    };
    write_bt(L::RV);
    tc::fence_proxy_async();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    constexpr uint32_t idesc = idesc_bf16(128, V);
    const uint32_t at = tc::smem_u32(sm + L::AT), bt = tc::smem_u32(sm + L::BT);
    auto issue = [&](uint32_t d) {
#pragma unroll
        for (int term = 0; term < 3; ++term)
#pragma unroll
            for (int ks = 0; ks < CT / 16; ++ks)
                tc::mma_ss(d, tc::sdesc_sw128(at + term * 16384 + 32 * ks), tc::sdesc_sw128(bt + 32 * ks), idesc,
                           (term | ks) ? 1u : 0u);
        tc::mma_commit(bar);
    };
    if (tid == 0)
        issue(tmem);   // dS -> columns [0, V)
    bool ok = tc::bar_wait(bar, 0);
    tc::fence_after();
    // ---- the tiles are free again: (q e^{G})^T in three terms and do^T
#pragma unroll
    for (int i = 0; i < 4; ++i)
        split3_store(sm + L::AT, key, j0 + 2 * i, xq[i]);
    write_bt(L::RD);
    tc::fence_proxy_async();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (tid == 0)
        issue(tmem + V);   // dR (unscaled) -> columns [V, 2V)
    ok = tc::bar_wait(bar, 1) && ok;
    tc::fence_after();
    if (!ok) {
        if (tid == 0)
            report(a.status, GLA_ERR_TIMEOUT);
    } else {
        // ---- epilogue: warps 0-3 dS, warps 4-7 dR; lane = key, a row of V values per thread
        const int rkey = 32 * (warp & 3) + lane;
        const bool isR = warp >= 4;
        float *dst = (isR ? a.dR : a.dS) + (((size_t)j * H + h) * KT + rkey) * a.V;
        const float mul = isR ? a.scale : 1.f;
        const uint32_t base = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (isR ? V : 0);
#pragma unroll
        for (int cc = 0; cc < V / 32; ++cc) {
            uint32_t r[32];
            tc::tmem_ld32(base + 32 * cc, r);
            tc::tmem_wait_ld(r);
#pragma unroll
            for (int w4 = 0; w4 < 8; ++w4)
                *reinterpret_cast<float4 *>(dst + 32 * cc + 4 * w4) =
                    make_float4(mul * __uint_as_float(r[4 * w4]), mul * __uint_as_float(r[4 * w4 + 1]),
                                mul * __uint_as_float(r[4 * w4 + 2]), mul * __uint_as_float(r[4 * w4 + 3]));
        }
        if (tid < KT)
            a.gl[((size_t)j * H + h) * KT + tid] = gl;
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0)
        tc::tmem_dealloc(tmem, 2 * V);
}

template <typename Tg, int V>
cudaError_t launch_sums_tc(const BwdArgs &a, int J, cudaStream_t s)
{
    auto f = bwd_chunk_sums_tc<Tg, V>;
    const size_t bytes = SumsSmem<Tg, V>::BYTES + 1024;
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
    f<<<dim3(J, a.H), NTS, bytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool bwd_sums_tc_supported(int dtype, int K, int V)
{
    return (dtype == GLA_BF16 || dtype == GLA_BF16_GF32) && K == 128 && (V == 64 || V == 128);
}

cudaError_t launch_bwd_sums_tc(const BwdArgs &a, int J, int dtype, cudaStream_t s)
{
    if (dtype == GLA_BF16_GF32)
        return a.V == 64 ? launch_sums_tc<float, 64>(a, J, s) : launch_sums_tc<float, 128>(a, J, s);
    return a.V == 64 ? launch_sums_tc<__nv_bfloat16, 64>(a, J, s) : launch_sums_tc<__nv_bfloat16, 128>(a, J, s);
}

}  // namespace gla
