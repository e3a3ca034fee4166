// TTT-linear forward on the tensor cores (bf16 q, k, v, D = 128; page "fla/ops/ttt/fused_chunk.py":
// fused_chunk_ttt_linear_fwd_kernel, then the norm_residual step of fused_chunk_ttt_linear).  Per mini-batch
// of BT rows, with the inner model h [D][D] (row = input feature, column = output feature) and hb [D]:
//   kh_i = k_i h + hb, xhat_i = LN(kh_i), g_i = (xhat_i w + b + k_i - v_i) w,
//   v2_i = rstd_i / D (D g_i - sum g_i - xhat_i sum(g_i xhat_i))
//   o_i  = scale q_i h + hb - eta_i sum_{j<=i} (scale q_i . k_j + 1) v2_j;   o_i += LN(o_i) w + b
//   h   -= eta_last sum_j k_j^T v2_j,   hb -= eta_last sum_j v2_j
//
// One CTA per (sequence, head).  The state lives in TMEM, transposed and in fp32: lane m holds column m of
// h (h^T[m][.]).  The serial chain of mini-batches never waits for a product of the state: with W_t =
// -eta_last v2_t (the update h_{t+1} = h_t + k_t^T W_t),
//   k_t h_t = k_t h_{t-1} + (k_t k_{t-1}^T) W_{t-1},
// so k_t h_{t-1} is taken one mini-batch ahead and the correction, a product of k_t k_{t-1}^T (staged in
// two bf16 terms one mini-batch ahead) with W_{t-1}, is the first product issued once W_{t-1} is known.
// Per mini-batch t:
//   * the split warps (which also form the outputs) cut h_t into two bf16 terms as soon as the update that
//     made it is complete (h = h1 + h2 + e, |e| <= 2^-18 |h|, each term rounded to nearest by conversion);
//   * one issuing thread then takes h_t^T [q_t; k_{t+1}]^T (tcgen05 kind::f16, A the two terms from TMEM,
//     M = 128, N = 2 BT, K = D: the outputs' q h and the next mini-batch's k h_t), the correction and the
//     update; the row products of the tile [k_t; q_t; k_{t+1}] with k_t (q k^T for the outputs, k_{t+1} k_t^T
//     for the next correction) need no state and are issued a mini-batch ahead by a second issuing thread
//     (which also issues the outputs' small products), and two staging warps turn them into the B operands of
//     the small products with W_t (two bf16 terms each);
//   * the chain warps move k h (transposed in TMEM) to shared memory once and run the rest of the step on rows,
//     so the LayerNorm statistics and the two gradient sums are reductions within a warp; W_t = -eta_last v2_t
//     is split exactly into three bf16 terms (MN-major A): the update h^T += W^T k is one more product
//     accumulating into the fp32 state on all three (B: the k rows of the tile, MN-major), so the state itself
//     is never rewritten by the CUDA cores, and the small products (the correction, the outputs'
//     score-weighted sums) take the first two, which leave at most 2^-18 |W_t|;
//   * the outputs of a mini-batch are formed one mini-batch behind from its q h columns, hb and the product
//     of its masked scores with W_t, through shared memory to rows for their LayerNorm, with the buffers kept
//     by parity and released through mbarriers.
// Rows arrive by asynchronous copies two mini-batches ahead (three tiles in turn); rows past the end of a
// sequence are zero in k and q and take no part in the update (as the CUDA-core path).
#include <cuda_bf16.h>

#include "gla_internal.h"
#include "tc_ptx.cuh"

namespace gla {

namespace {

constexpr int D = 128;
constexpr int NTH = 640;   // warps 0-7: the chain; 8-15: the state split and the outputs; 16-19: MMA issue, row
                           // copies and the two warps that stage the small products' B operands

template <int BT>
struct TtcLayout {
    static constexpr int XH = 3 * BT * 128;          // one 64-feature half of a tile [k_t; q_t; k_{t+1}]
    static constexpr int XB = 2 * XH;                // one tile
    static constexpr int X0 = 0;                     // [3] tiles (K-major, 128-byte swizzle), by mini-batch mod 3
    static constexpr int VR = X0 + 3 * XB;           // [3][BT][D] raw v rows (bf16), likewise
    static constexpr int V2T = VR + 3 * BT * D * 2;  // [2][3] terms of -eta_last v2 by parity, MN-major: [BT rows][2 halves]
    static constexpr int V2H = BT * 128;             // one 64-column half of a term
    static constexpr int V2P = 3 * 2 * V2H;          // one parity's three terms
    static constexpr int V2F = V2T + 2 * V2P;        // [BT][D] v2 fp32 (the chain's sums over rows for hb)
    // the B operands of the small products with W = -eta_last v2 (K-major, 128-byte swizzle, BT rows of BT
    // K values): two bf16 terms of k_{t+1} k_t^T (the next correction), two of the outputs' scaled scores
    static constexpr int TB = BT * 128;
    static constexpr int MT = (V2F + BT * D * 4 + 1023) / 1024 * 1024;
    static constexpr int KKT = MT, MST = MT + 2 * TB;
    static constexpr int KH = MT + 4 * TB;           // [BT][D] k_t h_t + hb (fp32): the chain's rows
    static constexpr int ET = KH + BT * D * 4;       // [3][BT] learning rates (0 past the end)
    static constexpr int HBP = ET + 3 * BT * 4;      // [2][D] hb at the start of a mini-batch, by parity
    static constexpr int OV = HBP + 2 * D * 4;       // [BT][D] the outputs before their LayerNorm (fp32)
    // prod, upd, hs_half[0], v2t(0), v2_full[2], out_free[2], xfull[3], slot_free[3], kk(0), tail[2], corr, rows,
    // hs_half[1], v2t(1), kk(1); TMEM address; abort word
    static constexpr int BAR = (OV + BT * D * 4 + 7) / 8 * 8;
    // the row products read rows 0..127 of a tile with K-halves XH apart: keep that span allocated
    static constexpr int END = BAR + 192 > X0 + 2 * XB + XH + 128 * 128 ? BAR + 192 : X0 + 2 * XB + XH + 128 * 128;
    static constexpr int BYTES = END + 1024;
    // TMEM columns: the state, its two bf16 terms (64 columns each), [q h_t, k_{t+1} h_t]^T by parity, the row
    // products by parity, the outputs' score-weighted sums of v2 by parity
    static constexpr uint32_t HT = 0, HS = 128, DA = 256, DC = 384, DO = 448, COLS = 512;
    static_assert(VR % 1024 == 0 && V2T % 1024 == 0 && V2P % 1024 == 0, "swizzled tiles are 1024-byte aligned");
    static_assert(BYTES <= 227 * 1024, "shared memory of one CTA");
};

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// A shared-memory descriptor advanced by `bytes` (the start-address field holds address >> 4 and shared
// addresses stay below 2^18, so the add cannot carry out of it).  The MMA loops below are fully unrolled over
// descriptors formed once: an issuing thread then spends about half the cycles per tcgen05.mma that a loop
// forming each descriptor from its address does (44 against 88 cycles at N = 32, measured).
__device__ __forceinline__ uint64_t sd_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// Half `HALF` of the state products [q_t h_t, k_{t+1} h_t]^T: the K steps c / 16 = HALF*2 + {0, 1} and
// 4 + HALF*2 + {0, 1} of both terms of h_t (A from TMEM), B the tile's rows BT .. 3 BT - 1 (dq: descriptor of
// those rows' first K-half)
template <int BT, int HALF>
__device__ __forceinline__ void state_products(uint32_t d, uint32_t hs, uint64_t dq, uint32_t idesc, int xh)
{
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int ks = (kk & 1) + 2 * HALF + 4 * (kk >> 1);
            tc::mma_ts(d, hs + 64 * tt + 8 * ks, sd_add(dq, (uint32_t)((ks >> 2) * xh + (ks & 3) * 32)), idesc,
                       (HALF | tt | kk) ? 1u : 0u);
        }
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
// Two fp32 values -> two bf16x2 words by the conversion instruction (round to nearest): x = x1 + x2 + e with
// |e| <= 2^-18 |x| (x1 = bf16(x), x2 = bf16(x - x1), the remainder exact by Sterbenz's lemma).  Six
// instructions a pair against the integer cut's twelve.
__device__ __forceinline__ void split2_rn(float a, float b, uint32_t &w1, uint32_t &w2)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);   // .x = a (low half), .y = b
    w1 = *reinterpret_cast<const uint32_t *>(&h);
    const float ra = a - __uint_as_float(w1 << 16), rb = b - __uint_as_float(w1 & 0xFFFF0000u);
    const __nv_bfloat162 l = __floats2bfloat162_rn(ra, rb);
    w2 = *reinterpret_cast<const uint32_t *>(&l);
}

// x[n] <- its sum over the warp's 32 lanes, the N sums interleaved
template <int N>
__device__ __forceinline__ void warp_sums(float (&x)[N])
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int n = 0; n < N; ++n)
            x[n] += __shfl_xor_sync(0xffffffffu, x[n], o);
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
// barrier of the 256 threads of a role (named barrier id) that also returns the AND of x over them, so that
// a wait taken by one thread gives every thread the same outcome
__device__ __forceinline__ bool role_all(bool x, int id)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, 256, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}\n"
                 : "=r"(r)
                 : "r"((uint32_t)x), "r"(id)
                 : "memory");
    return r != 0;
}

template <int BT>
__global__ void __launch_bounds__(NTH, 1) ttt_linear_tc(TttArgs a)
{
    using L = TtcLayout<BT>;
    constexpr int HB = BT / 2;   // rows per thread (row half)
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char *sm = smraw + ((1024u - (tc::smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);
    uint64_t *prod = bar, *upd = bar + 1;
    auto v2t = [bar](int q) { return bar + (q ? 20 : 3); };   // W_t's terms written, by parity
    // the state's two terms of columns c (K of the state products) in two chunks: c in [0, 32) + [64, 96), then
    // the rest (each split thread takes 32 columns of its row half at a time)
    uint64_t *const hs_half[2] = {bar + 2, bar + 19};
    uint64_t *v2_full = bar + 4, *out_free = bar + 6;
    uint64_t *xfull = bar + 8, *slot_free = bar + 11;   // [3] by mini-batch mod 3: the tile's rows landed / free
    auto kk = [bar](int q) { return bar + (q ? 21 : 14); };   // the small products' B operands staged, by parity
    uint64_t *tail = bar + 15;                           // [2] the small products with W_t done, by parity
    uint64_t *corr = bar + 17;                           // the correction onto the next k h is done
    uint64_t *rows = bar + 18;                           // the row products of a tile are done
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + L::BAR + 176);
    volatile int *abort_w = reinterpret_cast<volatile int *>(sm + L::BAR + 180);
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
    const int nmb = (eos - bos + BT - 1) / BT;   // mini-batches
    const __nv_bfloat16 *gq = static_cast<const __nv_bfloat16 *>(a.q), *gk = static_cast<const __nv_bfloat16 *>(a.k);
    const __nv_bfloat16 *gv = static_cast<const __nv_bfloat16 *>(a.v);

    if (tid == 0) {
        tc::bar_init(prod, 1);
        tc::bar_init(upd, 1);
        tc::bar_init(hs_half[0], 256);
        tc::bar_init(hs_half[1], 256);
        tc::bar_init(v2t(0), 1);
        tc::bar_init(v2t(1), 1);
        for (int b = 0; b < 2; ++b) {
            tc::bar_init(&v2_full[b], 256);
            tc::bar_init(&out_free[b], 256);
        }
        for (int b = 0; b < 3; ++b) {
            tc::bar_init(&xfull[b], 32);   // one completion-tracked arrival per lane of the copy warp
            tc::bar_init(&slot_free[b], 2);   // the row products, and the update
        }
        tc::bar_init(kk(0), 2);   // one arrival per staging warp
        tc::bar_init(kk(1), 2);
        tc::bar_init(&tail[0], 1);
        tc::bar_init(&tail[1], 1);
        tc::bar_init(corr, 1);
        tc::bar_init(rows, 1);
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
    const int r0h = HB * rh;   // first row of this thread's half
    bool ok = true;

    // warps 16-19: the two staging warps are the ones whose TMEM lane quarter holds the row products' score rows
    // (lanes BT..2 BT-1) and k_{t+1} k_t^T rows (lanes 2 BT..3 BT-1); the issue and copy warps take the others
    constexpr int W_SC = 16 + BT / 32, W_KK = 16 + BT / 16, W_ISSUE = BT == 16 ? 18 : 16, W_COPY = 19;
    if (warp == W_ISSUE) {
        // ================================ MMA issue ================================
        if (lane == 0) {
            constexpr uint32_t ID_Q = idesc_bf16(128, 2 * BT), ID_C = idesc_bf16(128, BT);
            constexpr uint32_t ID_B = idesc_bf16(128, D) | tc::kIdescAMajorMN | tc::kIdescBMajorMN;
            constexpr uint32_t ID_W = idesc_bf16(128, BT) | tc::kIdescAMajorMN;
            const uint64_t dkk = tc::sdesc_sw128(sb + L::KKT);   // k_{t+1} k_t^T's two terms
            for (int t = 0; t < nmb && ok; ++t) {
                const int p = t & 1;
                const uint32_t xs = sb + L::X0 + (t % 3) * L::XB;
                // the first chunk of h_t's two terms and the tile's rows are in place; the outputs of t - 2 are
                // done with this parity's columns
                ok = tc::bar_wait(hs_half[0], t & 1, abort_w) && tc::bar_wait(&xfull[t % 3], (t / 3) & 1, abort_w);
                if (ok && t >= 2)
                    ok = tc::bar_wait(&out_free[p], ((t >> 1) - 1) & 1, abort_w);
                if (!ok)
                    break;
                tc::fence_after();
                tc::fence_proxy_async();   // the copied rows -> the tensor cores
                // [q_t h_t, k_{t+1} h_t]^T: tile rows BT .. 3 BT - 1, K steps of the first chunk (c / 16 = 0, 1, 4,
                // 5), then of the second while it is being split
                const uint64_t dq = tc::sdesc_sw128(xs + BT * 128);
                state_products<BT, 0>(tmem + L::DA + 64 * p, tmem + L::HS, dq, ID_Q, L::XH);
                if (!(ok = tc::bar_wait(hs_half[1], t & 1, abort_w)))
                    break;
                tc::fence_after();
                if (t == 0) {   // k_0 h_0, the first mini-batch's rows (columns BT.. of the other parity)
                    const uint64_t dk = tc::sdesc_sw128(xs);
#pragma unroll
                    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks)
                            tc::mma_ts(tmem + L::DA + 64 + BT, tmem + L::HS + 64 * tt + 8 * ks,
                                       sd_add(dk, (uint32_t)((ks >> 2) * L::XH + (ks & 3) * 32)), ID_C,
                                       (tt | ks) ? 1u : 0u);
                }
                state_products<BT, 1>(tmem + L::DA + 64 * p, tmem + L::HS, dq, ID_Q, L::XH);
                tc::mma_commit(prod);
                // W_t's terms (the chain) and the small products' B operands (the staging warps) are in place
                if (!(ok = tc::bar_wait(v2t(p), (t >> 1) & 1, abort_w) && tc::bar_wait(kk(p), (t >> 1) & 1, abort_w)))
                    break;
                tc::fence_after();
                // first the correction (k_{t+1} k_t^T) W_t onto k_{t+1} h_t, which the chain waits for: W_t's
                // first two terms (MN-major A; they leave at most 2^-18 |W_t|) by k_{t+1} k_t^T's two, without
                // the product of the two second terms (at most 2^-18 of the whole)
                const uint64_t dw = tc::sdesc_mn_sw128(sb + L::V2T + p * L::V2P, L::V2H);   // W_t's terms
                if (t + 1 < nmb) {
#pragma unroll
                    for (int tw = 0; tw < 2; ++tw)
#pragma unroll
                        for (int tb = 0; tb < 2 - tw; ++tb)
#pragma unroll
                            for (int ks = 0; ks < BT / 16; ++ks)
                                tc::mma_ss(tmem + L::DA + 64 * p + BT, sd_add(dw, tw * 2 * L::V2H + ks * 2048),
                                           sd_add(dkk, tb * L::TB + ks * 32), ID_W, 1u);
                }
                tc::mma_commit(corr);
                // the update h^T += W_t^T k_t into the fp32 state, on all three (exact) terms
                {
                    const uint64_t dkr = tc::sdesc_mn_sw128(xs, L::XH);   // the tile's k_t rows, MN-major
#pragma unroll
                    for (int tt = 0; tt < 3; ++tt)
#pragma unroll
                        for (int ks = 0; ks < BT / 16; ++ks)
                            tc::mma_ss(tmem + L::HT, sd_add(dw, tt * 2 * L::V2H + ks * 2048), sd_add(dkr, ks * 2048),
                                       ID_B, 1u);
                }
                tc::mma_commit(upd);
                tc::mma_commit(&slot_free[t % 3]);
            }
        }
    } else if (warp == W_SC || warp == W_KK) {
        // ============ the B operands of the small products with W_t ============
        // to shared memory in two bf16 terms: the outputs' scores (eta_i / eta_last)(scale q_i.k_j + 1) for
        // j <= i (0 above the diagonal), and k_{t+1} k_t^T, once the mini-batch's row products are complete
        // and the last mini-batch's small products (which read these buffers) are done
        // Lane 0 of the k_{t+1} k_t^T warp is the second MMA issuer: per mini-batch the outputs' sums
        // -eta_i sum_j (scale q_i.k_j + 1) v2_j (W_t's first two terms) and the next tile's row products, so
        // that the main issuer keeps only the state products, the correction and the update (each issuing
        // thread waits about 120 cycles per tcgen05.mma, whatever its size; issuers in different warps overlap)
        const bool sc = warp == W_SC;
        constexpr uint32_t ID_C = idesc_bf16(128, BT), ID_W = idesc_bf16(128, BT) | tc::kIdescAMajorMN;
        // the row products of tile tt (they need no state): its rows times k_tt, lanes BT.. q_tt k_tt^T, lanes
        // 2 BT.. k_{tt+1} k_tt^T.  Issued a mini-batch ahead; with the update they release the tile.
        auto row_products = [&](int tt) {
            const uint32_t xr = sb + L::X0 + (tt % 3) * L::XB;
            if (!tc::bar_wait(&xfull[tt % 3], (tt / 3) & 1, abort_w))
                return false;
            tc::fence_after();
            tc::fence_proxy_async();   // the copied rows -> the tensor cores
            const uint64_t d0 = tc::sdesc_sw128(xr);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint64_t dx = sd_add(d0, (uint32_t)((ks >> 2) * L::XH + (ks & 3) * 32));
                tc::mma_ss(tmem + L::DC + 32 * (tt & 1), dx, dx, ID_C, ks ? 1u : 0u);
            }
            tc::mma_commit(rows);
            tc::mma_commit(&slot_free[tt % 3]);
            return true;
        };
        if (!sc && lane == 0 && nmb > 0)
            ok = row_products(0);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        for (int t = 0; t < nmb && ok; ++t) {
            const int p = t & 1, len = min(BT, eos - (bos + t * BT));
            // (the last mini-batch's small products: the outputs' sums from the second issuer, the correction
            // from the first)
            ok = tc::bar_wait(&xfull[t % 3], (t / 3) & 1, abort_w) && tc::bar_wait(rows, t & 1, abort_w) &&
                 (t == 0 || (tc::bar_wait(&tail[p ^ 1], ((t - 1) >> 1) & 1, abort_w) &&
                             tc::bar_wait(corr, (t - 1) & 1, abort_w)));
            if (!ok)
                break;
            tc::fence_after();
            uint32_t r[BT];
            tmem_ldn<BT>(tl + L::DC + 32 * p, r);
            const int row = m - (sc ? BT : 2 * BT);
            if (row >= 0 && row < BT) {
                const float *ET = reinterpret_cast<const float *>(sm + L::ET + (t % 3) * BT * 4);
                const float f = sc ? ET[row] / ET[len - 1] : 1.f;
                unsigned char *t0 = sm + (sc ? L::MST : L::KKT), *t1 = t0 + L::TB;
#pragma unroll
                for (int j = 0; j < BT; j += 8) {
                    uint32_t w1[4], w2[4];
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        float x0 = __uint_as_float(r[j + e]), x1 = __uint_as_float(r[j + e + 1]);
                        if (sc) {
                            x0 = j + e <= row ? f * fmaf(scale, x0, 1.f) : 0.f;
                            x1 = j + e + 1 <= row ? f * fmaf(scale, x1, 1.f) : 0.f;
                        }
                        split2_rn(x0, x1, w1[e / 2], w2[e / 2]);
                    }
                    const uint32_t off = tc::sw128(row, j);
                    *reinterpret_cast<uint4 *>(t0 + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
                    *reinterpret_cast<uint4 *>(t1 + off) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
                }
                tc::fence_proxy_async();
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0)
                tc::bar_arrive(kk(p));
            if (!sc) {
                // W_t's terms are in place, both B operands staged, and the outputs of t - 2 are done with this
                // parity's columns
                if (lane == 0) {
                    ok = tc::bar_wait(v2t(p), (t >> 1) & 1, abort_w) && tc::bar_wait(kk(p), (t >> 1) & 1, abort_w) &&
                         (t < 2 || tc::bar_wait(&out_free[p], ((t >> 1) - 1) & 1, abort_w));
                    if (ok) {
                        tc::fence_after();
                        const uint64_t dw = tc::sdesc_mn_sw128(sb + L::V2T + p * L::V2P, L::V2H);
                        const uint64_t dm = tc::sdesc_sw128(sb + L::MST);
#pragma unroll
                        for (int tw = 0; tw < 2; ++tw)   // (without the product of the two second terms)
#pragma unroll
                            for (int tb = 0; tb < 2 - tw; ++tb)
#pragma unroll
                                for (int ks = 0; ks < BT / 16; ++ks)
                                    tc::mma_ss(tmem + L::DO + 32 * p, sd_add(dw, tw * 2 * L::V2H + ks * 2048),
                                               sd_add(dm, tb * L::TB + ks * 32), ID_W, (tw | tb | ks) ? 1u : 0u);
                        tc::mma_commit(&tail[p]);
                        if (t + 1 < nmb)
                            ok = row_products(t + 1);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            }
        }
    } else if (warp == W_COPY) {
        // ================================ row copies ================================
        // mini-batch t's rows into tile t mod 3: k_t (rows 0..BT-1), q_t (BT..), k_{t+1} (2 BT..), zero past the
        // end; its v rows and learning rates.  Each lane's copies arrive on the tile's barrier as they land.
        // Lane l copies the 16-byte chunk l mod 16 (eight features) of every other row, starting at row l / 16.
        const int c = lane & 15, ib = lane >> 4;
        const size_t rs = (size_t)H * D;   // elements from one row to the next
        const size_t col = (size_t)h * D + 8 * c;
        for (int t = 0; t < nmb && ok; ++t) {
            const int r0 = bos + t * BT, slot = t % 3;
            if (t >= 3 && !(ok = tc::bar_wait(&slot_free[slot], ((t / 3) - 1) & 1, abort_w)))
                break;
            unsigned char *xt = sm + L::X0 + slot * L::XB + (c >> 3) * L::XH;
            unsigned char *vt = sm + L::VR + slot * BT * D * 2 + 16 * c;
            const size_t g0 = (size_t)r0 * rs + col;   // this lane's chunk of row r0 (in every tensor)
#pragma unroll 1
            for (int which = 0; which < 4; ++which) {   // k_t, q_t, k_{t+1}, v_t
                const __nv_bfloat16 *src = which == 1 ? gq : which == 3 ? gv : gk;
                const int roff = which == 2 ? BT : 0;
#pragma unroll
                for (int u = 0; u < BT / 2; ++u) {
                    const int i = ib + 2 * u;
                    const bool in = r0 + roff + i < eos;
                    const __nv_bfloat16 *g = src + g0 + (in ? (size_t)(roff + i) * rs : 0);
                    unsigned char *dst = which < 3 ? xt + tc::sw128(which * BT + i, 8 * (c & 7)) : vt + i * D * 2;
                    cp_async16(dst, g, in ? 16u : 0u);
                }
            }
            if (lane < BT) {
                const bool in = r0 + lane < eos;
                cp_async4(sm + L::ET + (slot * BT + lane) * 4, a.eta + (size_t)(in ? r0 + lane : r0) * H + h,
                          in ? 4u : 0u);
            }
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(&xfull[slot]))
                         : "memory");
        }
        asm volatile("cp.async.wait_all;" ::: "memory");   // nothing lands after the CTA is gone
    } else if (warp < 8) {
        // ================================ the chain ================================
        // k h arrives transposed (thread (qd, rh): feature m of rows r0h ..); it goes to shared memory once,
        // and the rest of the step runs on rows: warp w takes rows RW w .. RW w + RW - 1 and lane l the
        // features 4 l .. 4 l + 3, so every row statistic and gradient sum is a reduction within one warp
        constexpr int RW = BT / 8;
        const int i0 = RW * warp, f0 = 4 * lane;
        float hb = a.hb0 ? a.hb0[st * D + m] : 0.f;   // (feature m)
        float wf[4], bv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            wf[e] = a.w[(size_t)h * D + f0 + e];
            bv[e] = a.b[(size_t)h * D + f0 + e];
        }
        float *KH = reinterpret_cast<float *>(sm + L::KH);
        for (int t = 0; t < nmb && ok; ++t) {
            const int p = t & 1, r0 = bos + t * BT, len = min(BT, eos - r0);
            const unsigned char *xt = sm + L::X0 + (t % 3) * L::XB;
            // ---- k_t h_t + hb = (k_t h_{t-1} + (k_t k_{t-1}^T) W_{t-1}) + hb for this half's rows
            if (t == 0) {
                ok = tc::bar_wait(prod, 0, abort_w) && ok;   // k_0 h_0
                tc::fence_after();
            } else {
                // k_t h_{t-1} and its correction (k_t k_{t-1}^T) W_{t-1} are summed in TMEM
                if (ctid == 0)
                    ok = tc::bar_wait(corr, (t - 1) & 1, abort_w) && ok;
                ok = role_all(ok, 1);
                tc::fence_after();
            }
            {
                uint32_t r[HB];
                tmem_ldn<HB>(tl + L::DA + 64 * (p ^ 1) + BT + r0h, r);
#pragma unroll
                for (int u = 0; u < HB; ++u)
                    KH[(r0h + u) * D + m] = __uint_as_float(r[u]) + hb;
            }
            // this mini-batch's rows have landed, and the outputs of two mini-batches ago are done with this
            // parity's buffers (and so are the products that read this parity's W terms): one thread waits,
            // the barrier passes it on
            if (ctid == 0) {
                ok = tc::bar_wait(&xfull[t % 3], (t / 3) & 1, abort_w) && ok;
                if (t >= 2)
                    ok = tc::bar_wait(&out_free[p], ((t >> 1) - 1) & 1, abort_w) && ok;
            }
            ok = role_all(ok, 1);
            // ---- LayerNorm of the rows (two passes over registers)
            const float *ET = reinterpret_cast<const float *>(sm + L::ET + (t % 3) * BT * 4);
            const float el = ET[len - 1];
            float x[RW][4], s1[RW], s2[RW], rs[RW];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const float4 q4 = *reinterpret_cast<const float4 *>(KH + (i0 + r) * D + f0);
                x[r][0] = q4.x;
                x[r][1] = q4.y;
                x[r][2] = q4.z;
                x[r][3] = q4.w;
                s1[r] = (q4.x + q4.y) + (q4.z + q4.w);
            }
            warp_sums<RW>(s1);
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const float mean = s1[r] * (1.f / D);
                s2[r] = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    x[r][e] -= mean;
                    s2[r] = fmaf(x[r][e], x[r][e], s2[r]);
                }
            }
            warp_sums<RW>(s2);
            // ---- gradient of the inner loss; its two row sums over the features
            float gg[RW][4], gs[2 * RW];
            const unsigned char *vt = sm + L::VR + (t % 3) * BT * D * 2;
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int i = i0 + r;
                rs[r] = rsqrtf(fmaf(s2[r], 1.f / D, eps));
                const uint2 kw = *reinterpret_cast<const uint2 *>(xt + (f0 >> 6) * L::XH + tc::sw128(i, f0 & 63));
                const uint2 vw = *reinterpret_cast<const uint2 *>(vt + (i * D + f0) * 2);
                const float kv[4] = {__uint_as_float(kw.x << 16), __uint_as_float(kw.x & 0xFFFF0000u),
                                     __uint_as_float(kw.y << 16), __uint_as_float(kw.y & 0xFFFF0000u)};
                const float vv[4] = {__uint_as_float(vw.x << 16), __uint_as_float(vw.x & 0xFFFF0000u),
                                     __uint_as_float(vw.y << 16), __uint_as_float(vw.y & 0xFFFF0000u)};
                float sg = 0.f, sgx = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float xh = x[r][e] * rs[r];
                    x[r][e] = xh;
                    const float g = i < len ? (fmaf(xh, wf[e], bv[e]) + kv[e] - vv[e]) * wf[e] : 0.f;
                    gg[r][e] = g;
                    sg += g;
                    sgx = fmaf(g, xh, sgx);
                }
                gs[2 * r] = sg;
                gs[2 * r + 1] = sgx;
            }
            warp_sums<2 * RW>(gs);
            // ---- v2 (fp32, for the outputs and hb) and W = -eta_last v2 in three bf16 terms (exact), MN-major
            float *V2F = reinterpret_cast<float *>(sm + L::V2F);
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int i = i0 + r;
                float v2[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    v2[e] = rs[r] * (1.f / D) * (D * gg[r][e] - gs[2 * r] - x[r][e] * gs[2 * r + 1]);
                *reinterpret_cast<float4 *>(V2F + i * D + f0) = make_float4(v2[0], v2[1], v2[2], v2[3]);
                uint32_t wa[3], wb[3];
                split3(-el * v2[0], -el * v2[1], wa[0], wa[1], wa[2]);
                split3(-el * v2[2], -el * v2[3], wb[0], wb[1], wb[2]);
                const uint32_t off = (f0 >> 6) * L::V2H + tc::sw128(i, f0 & 63);
#pragma unroll
                for (int tt = 0; tt < 3; ++tt)
                    *reinterpret_cast<uint2 *>(sm + L::V2T + p * L::V2P + tt * 2 * L::V2H + off) =
                        make_uint2(wa[tt], wb[tt]);
            }
            if (rh == 0)   // hb of this mini-batch (feature m) for the outputs
                reinterpret_cast<float *>(sm + L::HBP)[p * D + m] = hb;
            tc::fence_proxy_async();
            tc::fence_before();
            chain_sync();
            if (ctid == 0)
                tc::bar_arrive(v2t(p));
            float sv = 0.f;
#pragma unroll
            for (int j = 0; j < BT; ++j)
                sv += V2F[j * D + m];
            hb = fmaf(-el, sv, hb);
            tc::bar_arrive(&v2_full[p]);   // this mini-batch's hb: to the outputs
        }
        if (nmb > 0) {
            ok = tc::bar_wait(upd, (nmb - 1) & 1, abort_w) && ok;   // the last update
            tc::fence_after();
        }
        if (a.ht && nmb > 0) {
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
        } else if (a.ht) {   // an empty sequence: the initial state (the split warps fill the TMEM state unordered)
            for (int u = 0; u < 64; ++u) {
                const size_t e = (st * D + 64 * rh + u) * D + m;
                a.ht[e] = a.h0 ? a.h0[e] : 0.f;
            }
        }
        if (a.hbt && rh == 0)
            a.hbt[st * D + m] = hb;
    } else if (warp < 16) {
        // ============ warps 8-15: the state split, and the outputs one mini-batch behind ============
        // h^T (fp32, this thread's 64 columns) -> its two bf16 terms
        auto split_state = [&]() {
#pragma unroll 1
            for (int c32 = 0; c32 < 2; ++c32) {
                uint32_t r[32], w1[16], w2[16];
                const int c0 = 64 * rh + 32 * c32;
                tc::tmem_ld32(tl + L::HT + c0, r);
                tc::tmem_wait_ld(r);
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    split2_rn(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]), w1[u], w2[u]);
                tc::tmem_st16(tl + L::HS + 0 * 64 + c0 / 2, w1);
                tc::tmem_st16(tl + L::HS + 1 * 64 + c0 / 2, w2);
                tc::tmem_wait_st();
                tc::fence_before();
                tc::bar_arrive(c32 ? hs_half[1] : hs_half[0]);   // this chunk of the terms: to the state products
            }
        };
        // initial state: h^T[m][c] = h0[c][m] for this thread's 64 columns c (row half rh), and its two terms
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
        if (nmb > 0)
            split_state();
        // q h + hb - eta_i sum_{j<=i} (scale q_i.k_j + 1) v2_j from the mini-batch's q h columns and the
        // score-weighted sums of v2 (both in TMEM, transposed: feature m of rows r0h ..), then through shared
        // memory to rows (warp w - 8 takes rows RW (w - 8) .., lane l the features 4 l .. 4 l + 3):
        // o + LN(o) w + b with the row statistics reduced within the warp
        constexpr int RW = BT / 8;
        const int i0 = RW * (warp - 8), f0 = 4 * lane;
        float wf[4], bv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            wf[e] = a.w[(size_t)h * D + f0 + e];
            bv[e] = a.b[(size_t)h * D + f0 + e];
        }
        float *OV = reinterpret_cast<float *>(sm + L::OV);
        for (int t = 0; t < nmb && ok; ++t) {
            const int p = t & 1, r0 = bos + t * BT, len = min(BT, eos - r0);
            // h_{t+1} = h_t + k_t^T W_t is complete (and with it the products that read h_t's terms, among them
            // this mini-batch's q h columns): its terms
            if (ctid == 0)
                ok = tc::bar_wait(upd, t & 1, abort_w) && ok;
            ok = role_all(ok, 2);
            tc::fence_after();
            if (t + 1 < nmb)
                split_state();
            ok = tc::bar_wait(&v2_full[p], (t >> 1) & 1, abort_w) && ok;
            if (ctid == 0)
                ok = tc::bar_wait(&tail[p], (t >> 1) & 1, abort_w) && ok;   // the score-weighted sums of v2
            ok = role_all(ok, 2);   // (also: the last mini-batch's rows of OV have been read)
            tc::fence_after();
            {
                uint32_t r[HB], dz[HB];
                tmem_ldn<HB>(tl + L::DA + 64 * p + r0h, r);
                tmem_ldn<HB>(tl + L::DO + 32 * p + r0h, dz);
                const float hbm = reinterpret_cast<const float *>(sm + L::HBP)[p * D + m];
#pragma unroll
                for (int u = 0; u < HB; ++u)
                    OV[(r0h + u) * D + m] = fmaf(scale, __uint_as_float(r[u]), hbm) + __uint_as_float(dz[u]);
            }
            tc::fence_before();
            tc::bar_arrive(&out_free[p]);   // this parity's TMEM columns and hb are read
            out_sync();
            float x[RW][4], s1[RW], s2[RW];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const float4 q4 = *reinterpret_cast<const float4 *>(OV + (i0 + r) * D + f0);
                x[r][0] = q4.x;
                x[r][1] = q4.y;
                x[r][2] = q4.z;
                x[r][3] = q4.w;
                s1[r] = (q4.x + q4.y) + (q4.z + q4.w);
            }
            warp_sums<RW>(s1);
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const float mean = s1[r] * (1.f / D);
                s2[r] = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float d = x[r][e] - mean;
                    s2[r] = fmaf(d, d, s2[r]);
                }
                s1[r] = mean;
            }
            warp_sums<RW>(s2);
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                const int i = i0 + r;
                const float rstd = rsqrtf(fmaf(s2[r], 1.f / D, eps));
                float y[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    y[e] = x[r][e] + fmaf((x[r][e] - s1[r]) * rstd, wf[e], bv[e]);
                if (i < len)
                    *reinterpret_cast<float4 *>(a.o + ((size_t)(r0 + i) * H + h) * D + f0) =
                        make_float4(y[0], y[1], y[2], y[3]);
            }
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
