// TTT-linear forward on the tensor cores (bf16 q, k, v, D = 128; page "fla/ops/ttt/fused_chunk.py":
// fused_chunk_ttt_linear_fwd_kernel, then the norm_residual step of fused_chunk_ttt_linear).  Per mini-batch
// of BT rows, with the inner model h [D][D] (row = input feature, column = output feature) and hb [D]:
//   kh_i = k_i h + hb, xhat_i = LN(kh_i), g_i = (xhat_i w + b + k_i - v_i) w,
//   v2_i = rstd_i / D (D g_i - sum g_i - xhat_i sum(g_i xhat_i))
//   o_i  = scale q_i h + hb - eta_i sum_{j<=i} (scale q_i . k_j + 1) v2_j;   o_i += LN(o_i) w + b
//   h   -= eta_last sum_j k_j^T v2_j,   hb -= eta_last sum_j v2_j
//
// One CTA per (sequence, head).  The state lives in TMEM, transposed and in fp32: lane m holds column m of
// h (h^T[m][.]).  Per mini-batch:
//   * h^T is split into two bf16 terms (h = h1 + h2 + e, |e| <= 2^-17 |h|, each term cut by integer
//     rounding), written back to TMEM as the 16-bit A operand of the products [k h, q h]^T = h^T [k; q]^T
//     (tcgen05 kind::f16, M = 128, N = 2 BT, K = D; k and q are exact in bf16); q k^T comes from one more
//     product with the same shared-memory tile of [k; q] rows;
//   * the rows' LayerNorm statistics and the two gradient sums are taken over the 128 lanes (four warps
//     of 32, merged through shared memory);
//   * the update h^T += (-eta_last v2)^T k is one more product accumulating into the fp32 state: -eta_last v2
//     split exactly into three bf16 terms (MN-major A) times the k rows of the same tile (MN-major B),
//     M = N = D, K = BT, so the state itself is never rewritten by the CUDA cores and carries no split error;
//   * the outputs of a mini-batch (which the state chain does not need) are formed by a second group of warps
//     one mini-batch behind: its q h columns, scores, v2 and learning rates are kept in buffers by parity,
//     handed over and released through mbarriers, so the output LayerNorm runs beside the next mini-batch's
//     state chain.
// The next mini-batch's k, q, v rows and learning rates arrive by asynchronous copies while the current one
// runs.  Rows past the end of a sequence are zero in k and q and take no part in the update (as the CUDA-core
// path).
#include <cuda_bf16.h>

#include "gla_internal.h"
#include "tc_ptx.cuh"

namespace gla {

namespace {

constexpr int D = 128;
constexpr int NTH = 512;   // warps 0-7: the state chain; warps 8-15: the outputs (lane quadrant x row half)

template <int BT>
struct TtcLayout {
    static constexpr int XH = 2 * BT * 128;          // one 64-feature half of the [k; q] tile (2 BT rows)
    static constexpr int XB = 2 * XH;                // one [k; q] tile
    static constexpr int X0 = 0;                     // [2] [k; q] tiles (K-major, 128-byte swizzle), by parity
    static constexpr int VR = X0 + 2 * XB;           // [2][BT][D] raw v rows (bf16)
    static constexpr int V2T = VR + 2 * BT * D * 2;  // [3] terms of -eta_last v2, MN-major: [BT rows][2 halves]
    static constexpr int V2H = BT * 128;             // one 64-column half of a term
    static constexpr int V2F = V2T + 3 * 2 * V2H;    // [2][BT][D] v2 fp32, by parity
    static constexpr int AS = V2F + 2 * BT * D * 4;  // [2][BT][BT] q k^T (unscaled), by parity
    static constexpr int RED = AS + 2 * BT * BT * 4; // [4 quadrants][BT][2] per-row partial statistics
    static constexpr int ET = RED + 4 * BT * 2 * 4;  // [2][BT] learning rates (0 past the end), by parity
    static constexpr int E2 = ET + 2 * BT * 4;       // [2][BT + 1] the outputs' learning rates and eta_last
    static constexpr int RED2 = E2 + 2 * (BT + 4) * 4;   // [4][BT][2] the output warps' partial statistics
    static constexpr int BAR = RED2 + 4 * BT * 2 * 4;    // mma, v2_full[2], out_free[2], TMEM address, abort
    // the q k^T product reads rows 0..127 of the tile with K-halves XH apart: keep that span allocated
    static constexpr int END = BAR + 64 > X0 + XB + XH + 128 * 128 ? BAR + 64 : X0 + XB + XH + 128 * 128;
    static constexpr int BYTES = END + 1024;
    // TMEM columns: the state, its two bf16 terms (64 columns each), [k h, q h]^T and q k^T by parity
    static constexpr uint32_t HT = 0, HS = 128, DA = 256, DC = 384, COLS = 512;
};

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(tc::smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(tc::smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}

// Exact split of two fp32 values into three bf16x2 words (x = x1 + x2 + x3 for each; every term rounded to
// 8 significant bits by an integer carry, the remainders exact by Sterbenz's lemma).  Low halves: a.
__device__ __forceinline__ uint32_t bf16_cut(uint32_t u) { return (u + 0x8000u) & 0xFFFF0000u; }
__device__ __forceinline__ void split3(float a, float b, uint32_t &w1, uint32_t &w2, uint32_t &w3)
{
    const uint32_t a1 = bf16_cut(__float_as_uint(a)), b1 = bf16_cut(__float_as_uint(b));
    const float ra = a - __uint_as_float(a1), rb = b - __uint_as_float(b1);
    const uint32_t a2 = bf16_cut(__float_as_uint(ra)), b2 = bf16_cut(__float_as_uint(rb));
    const float sa = ra - __uint_as_float(a2), sb = rb - __uint_as_float(b2);
    w1 = __byte_perm(a1, b1, 0x7632);
    w2 = __byte_perm(a2, b2, 0x7632);
    w3 = __byte_perm(__float_as_uint(sa), __float_as_uint(sb), 0x7632);
}
// Two fp32 values -> two bf16x2 words, x = x1 + x2 + e with |e| <= 2^-17 |x| (x1 rounded to 8 significant bits,
// x2 the exact remainder rounded the same way).
__device__ __forceinline__ void split2(float a, float b, uint32_t &w1, uint32_t &w2)
{
    const uint32_t a1 = bf16_cut(__float_as_uint(a)), b1 = bf16_cut(__float_as_uint(b));
    const float ra = a - __uint_as_float(a1), rb = b - __uint_as_float(b1);
    w1 = __byte_perm(a1, b1, 0x7632);
    w2 = __byte_perm(bf16_cut(__float_as_uint(ra)), bf16_cut(__float_as_uint(rb)), 0x7632);
}
__device__ __forceinline__ float bf(uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); }

// (mean, M2) of one value per lane over the warp (pairwise merges of equal counts)
__device__ __forceinline__ void warp_stats(float x, float &mean, float &m2)
{
    mean = x;
    m2 = 0.f;
#pragma unroll
    for (int o = 1, n = 1; o < 32; o <<= 1, n <<= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, mean, o), o2 = __shfl_xor_sync(0xffffffffu, m2, o);
        const float d = om - mean;
        m2 = m2 + o2 + d * d * (0.5f * n);   // two groups of n: n * n / (2 n)
        mean = 0.5f * (mean + om);
    }
}
__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
// merge the four quadrants' (mean, M2) of 32 values each: mean and 1 / sqrt(var + eps)
__device__ __forceinline__ void merge4(const float *red, int BT, int i, float eps, float &mean, float &rstd)
{
    float m = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        m += red[(q * BT + i) * 2];
    m *= 0.25f;
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float d = red[(q * BT + i) * 2] - m;
        s += red[(q * BT + i) * 2 + 1] + 32.f * d * d;
    }
    mean = m;
    rstd = rsqrtf(fmaf(s, 1.f / D, eps));
}

// x[0..N) = N consecutive 32-bit TMEM columns of this thread's lane (N = 4, 8, 16 or 32)
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, uint32_t (&x)[N])
{
    if constexpr (N == 4) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
                     : "r"(taddr));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    } else if constexpr (N == 8) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7])
                     : "r"(taddr));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    } else if constexpr (N == 16) {
        tc::tmem_ld16(taddr, x);
        tc::tmem_wait_ld(x);
    } else {
        tc::tmem_ld32(taddr, x);
        tc::tmem_wait_ld(x);
    }
}

__device__ __forceinline__ void chain_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ void out_sync() { asm volatile("bar.sync 2, 256;" ::: "memory"); }

template <int BT>
__global__ void __launch_bounds__(NTH, 1) ttt_linear_tc(TttArgs a)
{
    using L = TtcLayout<BT>;
    constexpr int HB = BT / 2;   // rows per thread (row half)
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char *sm = smraw + ((1024u - (tc::smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);
    uint64_t *v2_full = bar + 1, *out_free = bar + 3;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + L::BAR + 40);
    volatile int *abort_w = reinterpret_cast<volatile int *>(sm + L::BAR + 44);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, qd = warp & 3, rh = (warp >> 2) & 1;
    const int ctid = tid & 255;                          // index within the role
    const int m = 32 * qd + lane;                        // this thread's TMEM lane: output feature m
    const uint32_t lrow = (uint32_t)(32 * qd) << 16;
    const int n = blockIdx.x / a.H, h = blockIdx.x - n * a.H, H = a.H;
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
    const __nv_bfloat16 *gq = static_cast<const __nv_bfloat16 *>(a.q), *gk = static_cast<const __nv_bfloat16 *>(a.k);
    const __nv_bfloat16 *gv = static_cast<const __nv_bfloat16 *>(a.v);

    if (tid == 0) {
        tc::bar_init(bar, 1);
        for (int b = 0; b < 2; ++b) {
            tc::bar_init(&v2_full[b], 256);
            tc::bar_init(&out_free[b], 256);
        }
        *abort_w = 0;
        tc::bar_fence_init();
    }
    if (warp == 0)
        tc::tmem_alloc(tslot, L::COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot, sb = tc::smem_u32(sm), tl = tmem + lrow;
    const size_t st = (size_t)n * H + h;
    const float scale = a.scale, eps = a.eps;
    const float wm = a.w[(size_t)h * D + m], bm = a.b[(size_t)h * D + m];
    float hb = a.hb0 ? a.hb0[st * D + m] : 0.f;   // each role keeps its own copy, updated identically
    bool ok = true;

    if (warp < 8) {
        // ================================ the state chain ================================
        // initial state: h^T[m][c] = h0[c][m] for this thread's 64 columns c (row half rh)
#pragma unroll 1
        for (int c32 = 0; c32 < 2; ++c32) {
            uint32_t r[32];
            const int c0 = 64 * rh + 32 * c32;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                r[u] = __float_as_uint(a.h0 ? a.h0[(st * D + c0 + u) * D + m] : 0.f);
            tc::tmem_st32(tl + L::HT + c0, r);
        }
        tc::tmem_wait_st();

        // rows [r0, r0 + BT) of k, q (into the [k; q] tile of parity p, zero past the end), v, learning rates
        auto copy_rows = [&](int r0, int p) {
            const int len = min(BT, eos - r0);
            unsigned char *xt = sm + L::X0 + p * L::XB;
            for (int e = ctid; e < 3 * BT * 16; e += 256) {
                const int which = e / (BT * 16), rem = e - which * (BT * 16), i = rem >> 4, c = rem & 15;
                const bool in = i < len;
                const size_t row = (size_t)(r0 + (in ? i : 0)) * H + h;
                if (which < 2) {
                    const __nv_bfloat16 *src = (which == 0 ? gk : gq) + row * D + 8 * c;
                    const int rr = which * BT + i;   // tile row: k rows, then q rows
                    cp_async16(xt + (c >> 3) * L::XH + tc::sw128(rr, 8 * (c & 7)), src, in ? 16u : 0u);
                } else {
                    cp_async16(sm + L::VR + p * BT * D * 2 + i * D * 2 + 16 * c, gv + row * D + 8 * c,
                               in ? 16u : 0u);
                }
            }
            if (ctid < BT)
                cp_async4(sm + L::ET + (p * BT + ctid) * 4, a.eta + (size_t)(r0 + (ctid < len ? ctid : 0)) * H + h,
                          ctid < len ? 4u : 0u);
            asm volatile("cp.async.commit_group;" ::: "memory");
        };

        float *RED = reinterpret_cast<float *>(sm + L::RED);
        constexpr uint32_t ID_A = idesc_bf16(128, 2 * BT), ID_C = idesc_bf16(128, BT);
        constexpr uint32_t ID_B = idesc_bf16(128, D) | tc::kIdescAMajorMN | tc::kIdescBMajorMN;
        uint32_t phase = 0;
        if (bos < eos)
            copy_rows(bos, 0);
        int p = 0, t = 0;
        for (int r0 = bos; r0 < eos; r0 += BT, p ^= 1, ++t) {
            const int len = min(BT, eos - r0);
            // the previous update is complete (it read the k rows of the other tile): the next mini-batch's
            // rows may come into that tile
            if (t > 0) {
                ok = tc::bar_wait(bar, phase & 1, abort_w) && ok;
                ++phase;
            }
            tc::fence_after();
            if (r0 + BT < eos)
                copy_rows(r0 + BT, p ^ 1);
            else
                asm volatile("cp.async.commit_group;" ::: "memory");
            asm volatile("cp.async.wait_group 1;" ::: "memory");   // this mini-batch's rows
            const unsigned char *xt = sm + L::X0 + p * L::XB;
            const uint32_t xs = sb + L::X0 + p * L::XB;

            // ---- split h^T into its two bf16 terms (TMEM -> TMEM): this thread's 64 columns
#pragma unroll 1
            for (int c32 = 0; c32 < 2; ++c32) {
                uint32_t r[32], w1[16], w2[16];
                const int c0 = 64 * rh + 32 * c32;
                tc::tmem_ld32(tl + L::HT + c0, r);
                tc::tmem_wait_ld(r);
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    split2(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]), w1[u], w2[u]);
                tc::tmem_st16(tl + L::HS + 0 * 64 + c0 / 2, w1);
                tc::tmem_st16(tl + L::HS + 1 * 64 + c0 / 2, w2);
            }
            tc::tmem_wait_st();
            tc::fence_proxy_async();   // the copied rows of this mini-batch -> visible to the MMAs
            tc::fence_before();
            chain_sync();
            tc::fence_after();
            // the outputs of two mini-batches ago are done with this parity's TMEM columns and buffers
            if (t >= 2)
                ok = tc::bar_wait(&out_free[p], ((t >> 1) - 1) & 1, abort_w) && ok;
            tc::fence_after();

            // ---- [k h, q h]^T = h^T [k; q]^T (two terms of h) and q k^T, into this parity's columns
            if (ctid == 0) {
#pragma unroll 1
                for (int tt = 0; tt < 2; ++tt)
                    for (int ks = 0; ks < D / 16; ++ks)
                        tc::mma_ts(tmem + L::DA + 64 * p, tmem + L::HS + 64 * tt + 8 * ks,
                                   tc::sdesc_sw128(xs + (ks >> 2) * L::XH + (ks & 3) * 32), ID_A, (tt | ks) ? 1u : 0u);
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t dx = tc::sdesc_sw128(xs + (ks >> 2) * L::XH + (ks & 3) * 32);
                    tc::mma_ss(tmem + L::DC + 32 * p, dx, dx, ID_C, ks ? 1u : 0u);
                }
                tc::mma_commit(bar);
            }
            ok = tc::bar_wait(bar, phase & 1, abort_w) && ok;
            ++phase;
            tc::fence_after();

            // ---- this half's rows of k h + hb; q k^T to shared memory; LayerNorm statistics
            float kh[HB];
            {
                uint32_t r[HB];
                tmem_ldn<HB>(tl + L::DA + 64 * p + HB * rh, r);
#pragma unroll
                for (int u = 0; u < HB; ++u)
                    kh[u] = __uint_as_float(r[u]) + hb;
            }
            // q k^T: TMEM lanes BT .. 2 BT - 1 (the q rows of the tile), columns j < BT; the whole warp of row half 0
            // that holds those lanes loads (a warp-wide instruction), its lanes in range keep the values
            if (warp == (BT == 16 ? 0 : 1)) {
                uint32_t r[BT];
                tmem_ldn<BT>(tl + L::DC + 32 * p, r);
                float *AS = reinterpret_cast<float *>(sm + L::AS + p * BT * BT * 4);
                if (m >= BT && m < 2 * BT)
#pragma unroll
                    for (int j = 0; j < BT; j += 4)
                        *reinterpret_cast<float4 *>(AS + (m - BT) * BT + j) =
                            make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]), __uint_as_float(r[j + 2]),
                                        __uint_as_float(r[j + 3]));
            }
#pragma unroll
            for (int u = 0; u < HB; ++u) {
                float mean, m2;
                warp_stats(kh[u], mean, m2);
                if (lane == 0) {
                    RED[(qd * BT + HB * rh + u) * 2] = mean;
                    RED[(qd * BT + HB * rh + u) * 2 + 1] = m2;
                }
            }
            chain_sync();
            // ---- gradient of the inner loss; its two row sums over the features
            float xh[HB], gg[HB], rs[HB];
            const uint16_t *vr = reinterpret_cast<const uint16_t *>(sm + L::VR + p * BT * D * 2);
#pragma unroll
            for (int u = 0; u < HB; ++u) {
                const int i = HB * rh + u;
                float mean;
                merge4(RED, BT, i, eps, mean, rs[u]);
                xh[u] = (kh[u] - mean) * rs[u];
                const float ki = bf(*reinterpret_cast<const uint16_t *>(xt + (m >> 6) * L::XH + tc::sw128(i, m & 63)));
                gg[u] = i < len ? (fmaf(xh[u], wm, bm) + ki - bf(vr[i * D + m])) * wm : 0.f;
            }
            chain_sync();   // every thread has read the statistics: the buffer takes the gradient sums
#pragma unroll
            for (int u = 0; u < HB; ++u) {
                const float sg = warp_sum(gg[u]), sgx = warp_sum(gg[u] * xh[u]);
                if (lane == 0) {
                    RED[(qd * BT + HB * rh + u) * 2] = sg;
                    RED[(qd * BT + HB * rh + u) * 2 + 1] = sgx;
                }
            }
            chain_sync();
            const float *ET = reinterpret_cast<const float *>(sm + L::ET + p * BT * 4);
            const float el = ET[len - 1];
            float *V2F = reinterpret_cast<float *>(sm + L::V2F + p * BT * D * 4);
            float v2[HB];
#pragma unroll
            for (int u = 0; u < HB; ++u) {
                const int i = HB * rh + u;
                float sg = 0.f, sgx = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    sg += RED[(q * BT + i) * 2];
                    sgx += RED[(q * BT + i) * 2 + 1];
                }
                v2[u] = rs[u] * (1.f / D) * (D * gg[u] - sg - xh[u] * sgx);
                V2F[i * D + m] = v2[u];
            }
            if (ctid <= BT) {   // the learning rates and eta_last for the output warps
                float *E2 = reinterpret_cast<float *>(sm + L::E2 + p * (BT + 4) * 4);
                E2[ctid] = ctid < BT ? ET[ctid] : el;
            }
            // -eta_last v2 in three bf16 terms (exact), MN-major: row i, feature m (two rows per split)
#pragma unroll
            for (int u = 0; u < HB; u += 2) {
                const int i = HB * rh + u;
                uint32_t wv[3];
                split3(-el * v2[u], -el * v2[u + 1], wv[0], wv[1], wv[2]);
                const uint32_t off0 = (m >> 6) * L::V2H + tc::sw128(i, m & 63);
                const uint32_t off1 = (m >> 6) * L::V2H + tc::sw128(i + 1, m & 63);
#pragma unroll
                for (int tt = 0; tt < 3; ++tt) {
                    *reinterpret_cast<uint16_t *>(sm + L::V2T + tt * 2 * L::V2H + off0) = (uint16_t)(wv[tt] & 0xFFFFu);
                    *reinterpret_cast<uint16_t *>(sm + L::V2T + tt * 2 * L::V2H + off1) = (uint16_t)(wv[tt] >> 16);
                }
            }
            tc::fence_proxy_async();
            tc::fence_before();
            chain_sync();
            tc::fence_after();
            // ---- the update h^T += (-eta_last v2)^T k, accumulating into the fp32 state
            if (ctid == 0) {
                for (int tt = 0; tt < 3; ++tt)
                    for (int ks = 0; ks < BT / 16; ++ks)
                        tc::mma_ss(tmem + L::HT,
                                   tc::sdesc_mn_sw128(sb + L::V2T + tt * 2 * L::V2H + ks * 2048, L::V2H),
                                   tc::sdesc_mn_sw128(xs + ks * 2048, L::XH), ID_B, 1u);
                tc::mma_commit(bar);
            }
            tc::bar_arrive(&v2_full[p]);   // this mini-batch's q h columns, scores, v2 and rates: to the outputs
            float sv = 0.f;
#pragma unroll
            for (int j = 0; j < BT; ++j)
                sv += V2F[j * D + m];
            hb = fmaf(-el, sv, hb);
        }
        if (bos < eos) {
            ok = tc::bar_wait(bar, phase & 1, abort_w) && ok;   // the last update
            ++phase;
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        tc::fence_after();
        if (a.ht) {
#pragma unroll 1
            for (int c32 = 0; c32 < 2; ++c32) {
                uint32_t r[32];
                const int c0 = 64 * rh + 32 * c32;
                tc::tmem_ld32(tl + L::HT + c0, r);
                tc::tmem_wait_ld(r);
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    a.ht[(st * D + c0 + u) * D + m] = __uint_as_float(r[u]);
            }
        }
        if (a.hbt && rh == 0)
            a.hbt[st * D + m] = hb;
    } else {
        // ================================ the outputs, one mini-batch behind ================================
        // q h + hb - eta_i sum_{j<=i} (scale q_i.k_j + 1) v2_j from the mini-batch's q h columns, scores and
        // v2, then o + LN(o) w + b
        float *RED2 = reinterpret_cast<float *>(sm + L::RED2);
        int p = 0, t = 0;
        for (int r0 = bos; r0 < eos; r0 += BT, p ^= 1, ++t) {
            const int len = min(BT, eos - r0);
            ok = tc::bar_wait(&v2_full[p], (t >> 1) & 1, abort_w) && ok;
            tc::fence_after();
            uint32_t r[HB];
            tmem_ldn<HB>(tl + L::DA + 64 * p + BT + HB * rh, r);
            const float *V2F = reinterpret_cast<const float *>(sm + L::V2F + p * BT * D * 4);
            const float *AS = reinterpret_cast<const float *>(sm + L::AS + p * BT * BT * 4);
            const float *E2 = reinterpret_cast<const float *>(sm + L::E2 + p * (BT + 4) * 4);
            float v2c[BT];
#pragma unroll
            for (int j = 0; j < BT; ++j)
                v2c[j] = V2F[j * D + m];
            float ov[HB];
#pragma unroll
            for (int u = 0; u < HB; ++u) {
                const int i = HB * rh + u;
                float acc = 0.f;
#pragma unroll
                for (int j4 = 0; j4 < BT; j4 += 4) {
                    const float4 s4 = *reinterpret_cast<const float4 *>(AS + i * BT + j4);
                    acc = fmaf(j4 <= i ? fmaf(scale, s4.x, 1.f) : 0.f, v2c[j4], acc);
                    acc = fmaf(j4 + 1 <= i ? fmaf(scale, s4.y, 1.f) : 0.f, v2c[j4 + 1], acc);
                    acc = fmaf(j4 + 2 <= i ? fmaf(scale, s4.z, 1.f) : 0.f, v2c[j4 + 2], acc);
                    acc = fmaf(j4 + 3 <= i ? fmaf(scale, s4.w, 1.f) : 0.f, v2c[j4 + 3], acc);
                }
                ov[u] = fmaf(-E2[i], acc, fmaf(scale, __uint_as_float(r[u]), hb));
                float mean, m2;
                warp_stats(ov[u], mean, m2);
                if (lane == 0) {
                    RED2[(qd * BT + i) * 2] = mean;
                    RED2[(qd * BT + i) * 2 + 1] = m2;
                }
            }
            const float el = E2[BT];
            float sv = 0.f;
#pragma unroll
            for (int j = 0; j < BT; ++j)
                sv += v2c[j];
            out_sync();
#pragma unroll
            for (int u = 0; u < HB; ++u) {
                const int i = HB * rh + u;
                float mean, rstd;
                merge4(RED2, BT, i, eps, mean, rstd);
                if (i < len)
                    a.o[((size_t)(r0 + i) * H + h) * D + m] = ov[u] + fmaf((ov[u] - mean) * rstd, wm, bm);
            }
            hb = fmaf(-el, sv, hb);
            tc::fence_before();
            out_sync();   // RED2 is free again
            tc::bar_arrive(&out_free[p]);
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (!ok && (tid & 31) == 0)
        report(a.status, GLA_ERR_TIMEOUT);
    if (warp == 0)
        tc::tmem_dealloc(tmem, L::COLS);
}

template <int BT>
cudaError_t launch_bt(const TttArgs &a, cudaStream_t s)
{
    using L = TtcLayout<BT>;
    auto f = ttt_linear_tc<BT>;
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
    if (e != cudaSuccess)
        return e;
    f<<<a.N * a.H, NTH, L::BYTES, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool ttt_tc_supported(int dtype, int Dh, int BT)
{
    return dtype == GLA_BF16 && Dh == D && (BT == 16 || BT == 32);
}

cudaError_t launch_ttt_linear_tc(const TttArgs &a, cudaStream_t s)
{
    return a.BT == 16 ? launch_bt<16>(a, s) : launch_bt<32>(a, s);
}

}  // namespace gla
