// Backward chunk sums on the tensor cores (bf16 inputs, K = 128; page "fla/ops/gla/fused_chunk.py":
// fused_chunk_gla_bwd_kernel, whose state and adjoint carries these sums feed):
//     dS = sum_t (k_t e^{G_l - G_t})^T v_t,    dR = scale sum_t (q_t e^{G_t})^T do_t,    G_l
// per chunk of C = 64 rows and head, with G the chunk-local inclusive cumsum of the gates (natural log).
//
// One CTA per (chunk, head).  Both products are D[k][v] = sum_t A[k][t] B[v][t] with tcgen05 kind::f16 MMAs
// (bf16 operands, fp32 accumulation in TMEM): M = 128 keys, N = V, K = the chunk's 64 rows in steps of 16.
// The A operands (k e^{G_l - G} and q e^{G}, fp32 on chip) are split into three bf16 terms x = x1 + x2 + x3
// (exact to fp32 rounding) and written transposed into 128-byte-swizzled K-major tiles; the B operands
// (v and do, bf16 already) are written transposed into one tile each.  The rows of g, k and v arrive first by
// 16-byte asynchronous copies (g inside the A-tile region until its cumsum is taken); a thread owns one key
// and keeps its cumsum in registers for both gated operands.  dS is formed first; q and do are fetched into
// the places of k and v while its MMAs run, and the tiles are reused for dR.  Rows past the end of a chunk are
// zero in every tile.  The epilogue stages each result from TMEM (lane = key) in shared memory and writes
// whole rows of dS and dR (fp32, [slot][H][K][V]) with lanes on consecutive columns.  About 97 KB per CTA:
// two CTAs share an SM.
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
    static constexpr int AT = 0;                   // [3 terms] A^T tiles, 128 rows x 128 bytes each; the raw
                                                   // gates [64][128] (Tg) live here until the cumsum is taken
    static constexpr int BT = AT + 3 * 16384;      // B^T tile, V rows x 128 bytes
    static constexpr int RK = BT + V * 128;        // raw rows [64][128] bf16: k, then q
    static constexpr int RV = RK + CT * KT * 2;    // raw rows [64][V] bf16: v, then do
    static constexpr int BAR = RV + CT * V * 2;
    static constexpr int TSLOT = BAR + 8;
    static constexpr int BYTES = TSLOT + 8;
    static constexpr int SROW = V + 1;             // epilogue staging [128][V + 1] fp32 over AT .. RK
    static_assert(KT * SROW * 4 <= RV, "staging fits below the raw v rows");
    static_assert(CT * KT * (int)sizeof(Tg) <= BT, "raw gates fit in the A tiles");
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
__global__ void __launch_bounds__(NTS, 2) bwd_chunk_sums_tc(BwdArgs a)
{
    using L = SumsSmem<Tg, V>;
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char *sm = smraw + ((1024u - (tc::smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + L::TSLOT);
    const __nv_bfloat16 *Rk = reinterpret_cast<const __nv_bfloat16 *>(sm + L::RK);
    const Tg *Rg = reinterpret_cast<const Tg *>(sm + L::AT);
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
    // 16-byte asynchronous copies of the valid rows of a [rows, H, width] tensor (global rows of strideb bytes)
    // into shared rows of rowb bytes
    auto stage = [&](const void *src, int rowb, int strideb, int dst) {
        const int per = rowb / 16;
        const char *s8 = static_cast<const char *>(src);
        for (int e = tid; e < CT * per; e += NTS) {
            const int t = e / per, c = e - t * per;
            if (t < len)
                cp_async16(sm + dst + t * rowb + 16 * c, s8 + (rb + (size_t)t * rs) * strideb + 16 * c);
        }
    };
    stage(a.g, KT * (int)sizeof(Tg), KT * (int)sizeof(Tg), L::AT);
    stage(a.k, KT * 2, KT * 2, L::RK);
    stage(a.v, V * 2, a.ldv * 2, L::RV);
    asm volatile("cp.async.commit_group;" ::: "memory");
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
    // ---- thread: key = tid % 128, row groups jj = tid / 128 + 2 i (i < 4); its cumsum from the staged gates
    //      (the total first), kept in registers for both gated operands
    const int key = tid & 127, j0 = tid >> 7;
    float gl = 0.f;
    for (int t = 0; t < len; ++t)
        gl += wide<Tg>(Rg[t * KT + key]);
    float gv[4][8];
    {
        float run = 0.f;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = 8 * jj + u;
                run += t < len ? wide<Tg>(Rg[t * KT + key]) : 0.f;
                if ((jj & 1) == j0)
                    gv[jj >> 1][u] = run;
            }
    }
    __syncthreads();   // the raw gates are read: the A tiles may be written
    // ---- (k e^{G_l - G})^T in three terms, v^T in one
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int jj = j0 + 2 * i;
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int t = 8 * jj + u;
            x[u] = t < len ? __bfloat162float(Rk[t * KT + key]) * expf(gl - gv[i][u]) : 0.f;
        }
        split3_store(sm + L::AT, key, jj, x);
    }
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
    // the raw k and v rows are consumed: fetch q and do into their places while the MMAs run
    stage(a.q, KT * 2, KT * 2, L::RK);
    stage(a.dout, V * 2, a.ldv * 2, L::RV);
    asm volatile("cp.async.commit_group;" ::: "memory");
    bool ok = tc::bar_wait(bar, 0);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    tc::fence_before();
    __syncthreads();   // q, do visible; the first MMA group no longer reads the tiles
    tc::fence_after();
    // ---- (q e^{G})^T in three terms, do^T in one
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int jj = j0 + 2 * i;
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int t = 8 * jj + u;
            x[u] = t < len ? __bfloat162float(Rk[t * KT + key]) * expf(gv[i][u]) : 0.f;
        }
        split3_store(sm + L::AT, key, jj, x);
    }
    write_bt(L::RV);
    tc::fence_proxy_async();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (tid == 0)
        issue(tmem + V);   // dR (unscaled) -> columns [V, 2V)
    ok = tc::bar_wait(bar, 1) && ok;
    tc::fence_after();
    __syncthreads();   // every warp past the wait before the tiles become staging
    if (!ok) {
        if (tid == 0)
            report(a.status, GLA_ERR_TIMEOUT);
    } else {
        // ---- epilogue, dS then dR: TMEM (lane = key) -> staging [key][V + 1] (warps 0-3 the first half of
        //      the columns, warps 4-7 the second) -> whole rows of the workspace tile, lanes on columns
        float *stg = reinterpret_cast<float *>(sm + L::AT);
        const int rkey = 32 * (warp & 3) + lane;
        float *const dsts[2] = {a.dS, a.dR};
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const float mul = which ? a.scale : 1.f;
#pragma unroll
            for (int cc = 0; cc < V / 64; ++cc) {
                const int c0 = (warp >> 2) * (V / 2) + 32 * cc;
                uint32_t r[32];
                tc::tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(which * V + c0), r);
                tc::tmem_wait_ld(r);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    stg[rkey * L::SROW + c0 + i] = mul * __uint_as_float(r[i]);
            }
            __syncthreads();
            float *dst = dsts[which] + ((size_t)j * H + h) * KT * V;
            for (int e = tid; e < KT * V; e += NTS) {
                const int kr = e / V, c = e - kr * V;
                dst[e] = stg[kr * L::SROW + c];
            }
            __syncthreads();
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
