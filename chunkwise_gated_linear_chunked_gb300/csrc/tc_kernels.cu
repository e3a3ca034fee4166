// Tensor-core (tcgen05) kernels of the chunkwise GLA forward for bf16 inputs, K = 128, V a multiple of 128.
//
// Method (page "fla/ops/gla/fused_chunk.py"): per chunk of C = 64 rows with chunk-local cumsum G of the
// gates (FusedChunkGLAFunction.forward, kernel a), the state contribution (k*exp(G_last-G))^T V
// (prepare_qg_kg, fused_chunk_gla_fwd_kernel: kernel b), and the output = inter-chunk term (q*exp(G)) S plus
// the causally masked intra-chunk term with the inclusive diagonal (fwd_inner_chunk, the A @ v product of
// FusedChunkGLAFunction.forward: kernel d), with scale applied to the sum.  Segments of a long sequence are
// combined by the decayed scan S_in(p+1) = diag(exp(Gtot(p))) S_in(p) + dS(p) (kernel c), which the output
// kernel evaluates in its prologue from the state pass's per-segment dS and Gtot.  Gates are summed in log2
// units (g * log2(e)) so every decay factor is one hardware exp2.
//
// One CTA owns one (segment, head, 128-wide value tile).  The K x V state lives in TMEM transposed
// (lane = value column v, column = key dimension), so every MMA has M = 128:
//   (c) S^T += V^T   k^^T     A = V^T [v][t]  (K-major, smem), B = k^^T [key][t] (K-major, smem)
//   (a) O^T  = S'^T  q~^T      A = S' from TMEM (fp16),        B = q~  [t][key]   (K-major, smem)
//   (b) P    = q~    k~^T      A = q~ (rows 64..127 unused),   B = k~  [s][key]   (K-major, smem)
//   (d) O^T += V^T   P^T      A = V^T [v][s],                  B = P   [t][s]     (K-major, smem)
// with q~ = q*exp(G-G_a), k~ = k*exp(G_a-G), k^ = k*exp(G_last-G), S' = diag(exp(G_a)) S, and the anchor a
// the middle row of the chunk.  Operands are fp16 (bf16 inputs widen exactly; 11-bit significands keep the
// result within the parity bounds where single-rounded bf16 operands do not); accumulation is fp32 in TMEM.
// The state pass walks its segment's chunks last to first and folds the decay of the later chunks into k^
// (k * exp(G_last - G + later decay) <= |k|), so its state accumulates with no rescaling at all.
//
// Pipeline (one CTA per SM): three 64 KB stages hold a chunk's raw tiles and, converted in place, its
// operands — TMA loads q and k already in the 128-byte-swizzled K-major layout the MMA reads, so q~ and k~
// overwrite q and k element by element; k^^T and V^T are written over the g and v tiles once those have been
// read into registers.  S' and O^T are double-buffered in TMEM so consecutive chunks overlap.  Warp roles:
//   warps 0-7    gating group: cumsum and gating, running ahead of the tensor cores;
//   warps 8-11   state group: state conversion (S', decay) of the output pass;
//   warps 12-15  output group: masked scores -> P, then O^T -> shared memory -> TMA tensor store (scalar
//                stores for a ragged chunk);
//   warp 16      lane 0 issues the TMA loads and the MMAs.
// (Warps w of the state and output groups own TMEM lanes 32*(w%4)..+31.)  An operand that leaves the fp16
// range makes the outputs non-finite; the kernels check o, ht and dS and report GLA_ERR_RANGE.  Every mbarrier
// wait is bounded; on timeout the kernel records GLA_ERR_TIMEOUT, drains its own copies, stores and MMAs,
// frees TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <type_traits>

#include "gla_internal.h"
#include "tc_ptx.cuh"

namespace gla {
namespace {

using namespace tc;

constexpr int C = 64;            // chunk rows
constexpr int KD = 128;          // key dimension handled by this path
constexpr int VT = 128;          // value tile = TMEM lanes
constexpr int NA = 256;          // gating group: 8 warps
constexpr int NB = 128;          // state group
constexpr int NC = 128;          // output group
constexpr int WB = NA / 32, WC = (NA + NB) / 32, WCTL = (NA + NB + NC) / 32;   // first warp of each group
constexpr int NTHREADS = NA + NB + NC + 32;
constexpr float L2E = 1.4426950408889634f;

// one stage (64 KB): [q kb0 | k kb0 | q kb1 | k kb1] (8 KB each, SW128 K-major, 64 rows), g (16 KB),
// v (16 KB).  g and v are loaded unswizzled as [t][128] and later hold k^^T and V^T ([128][t], SW128).
constexpr int NSTAGE = 3;
constexpr int STAGE = 65536;
constexpr int ST_Q0 = 0, ST_K0 = 8192, ST_G = 32768, ST_V = 49152;
constexpr int OFF_P = NSTAGE * STAGE;          // P [t][s] fp16, 8 KB
constexpr int OFF_EG = OFF_P + 8192;           // per stage: exp(G_a)[128], exp(G_last)[128]
constexpr int OFF_PS = OFF_EG + NSTAGE * 1024; // gating-group partial sums: [2 parity][4 quarters][128]
constexpr int OFF_OST = OFF_PS + 4096;         // output staging: 32 rows x 128 fp32 (16 KB)
constexpr int OFF_BAR = OFF_OST + 16384;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;

// TMEM columns (fp32 unless noted)
constexpr uint32_t TM_S = 0;      // S^T accumulator: 128 columns (key)
constexpr uint32_t TM_SOP = 128;  // S'^T fp16 operand, two buffers of 64 columns (key pairs)
constexpr uint32_t TM_O = 256;    // O^T, two buffers of 64 columns (t)
constexpr uint32_t TM_P = 384;    // P: 64 columns (s), lanes t
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t ID_N64 = idesc_f16_f32(128, 64);
constexpr uint32_t ID_N128 = idesc_f16_f32(128, 128);

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ bool finite(float x) { return fabsf(x) <= 3.402823466e38f; }
// running max of |x| that keeps NaN (a single max.NaN per element)
__device__ __forceinline__ float amax_nan(float m, float x)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(fabsf(x)));
    return r;
}

template <typename T>
__device__ __forceinline__ T to_out(float x);
template <>
__device__ __forceinline__ float to_out<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ void sync_gating() { asm volatile("bar.sync 1, %0;" ::"n"(NA) : "memory"); }
__device__ __forceinline__ void sync_output() { asm volatile("bar.sync 2, %0;" ::"n"(NC) : "memory"); }

template <bool OUT, typename Tout>
__global__ void __launch_bounds__(NTHREADS, 1)
    gla_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_v,
           const __grid_constant__ CUtensorMap tm_o, Args a, int multi)
{
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *full = bars + 0, *prep = bars + 3, *ops_ready = bars + 6, *p_ready = bars + 7;
    uint64_t *mma_st = bars + 8, *mma1 = bars + 9, *mma2 = bars + 10, *o_free = bars + 11;   // o_free[2]
    uint64_t *fin = bars + 13;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 14);

    // the varlen slot table comes from the preceding plan kernel
    if (a.table || !OUT)
        grid_dep_wait();
    const int vt = blockIdx.x, h = blockIdx.y, j = blockIdx.z;
    int n, p, bos, eos, send;
    if (!resolve_slot(a, j, n, p, bos, eos, send))
        return;
    if (!OUT && eos == send)
        return;   // state contributions are needed for non-final segments only
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, V = a.V, v0 = vt * VT;
    const int nchunks = (eos - bos + C - 1) / C;
    // chunk handled at step i: in order for the output pass, last to first for the state pass
    auto chunk_of = [&](int i) { return OUT ? i : nchunks - 1 - i; };

    if (warp == 0)
        tmem_alloc(tmem_slot, TM_COLS);
    if (tid == NA + NB + NC) {
        for (int s = 0; s < NSTAGE; ++s) {
            bar_init(&full[s], 1);
            bar_init(&prep[s], NA);
        }
        bar_init(ops_ready, NB);
        bar_init(p_ready, NC);
        bar_init(mma_st, 1);
        bar_init(mma1, 1);
        bar_init(mma2, 1);
        bar_init(&o_free[0], NC);
        bar_init(&o_free[1], NC);
        bar_init(fin, 1);
        bar_fence_init();
        if (OUT) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_o);
        }
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_g);
        tma_prefetch_desc(&tm_v);
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (!OUT)
        grid_dep_launch();   // every CTA of this grid is running: the output pass may start launching
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == WCTL) {
        // ---------------------------------------------------------------------- control: TMA + MMA
        if (lane == 0) {
            constexpr uint32_t tx = (OUT ? 4 : 3) * 16384;
            int last_issued[NSTAGE] = {-1, -1, -1};
            auto issue = [&](int i) {
                const int s = i % NSTAGE;
                uint8_t *st = sm + s * STAGE;
                const int row0 = bos + chunk_of(i) * C;
                bar_expect_tx(&full[s], tx);
                if (OUT) {
                    tma_load_3d(st + ST_Q0, &tm_q, 0, h, row0, &full[s]);
                    tma_load_3d(st + 16384 + ST_Q0, &tm_q, 64, h, row0, &full[s]);
                }
                tma_load_3d(st + ST_K0, &tm_k, 0, h, row0, &full[s]);
                tma_load_3d(st + 16384 + ST_K0, &tm_k, 64, h, row0, &full[s]);
                tma_load_3d(st + ST_G, &tm_g, 0, h, row0, &full[s]);
                tma_load_3d(st + ST_V, &tm_v, v0, h, row0, &full[s]);
                last_issued[s] = i;
            };
            for (int i = 0; i < NSTAGE && i < nchunks; ++i)
                issue(i);
            const uint32_t pt = smem_u32(sm + OFF_P);
            for (int i = 0; i < nchunks; ++i) {
                const uint32_t ph = i & 1;
                const int s = i % NSTAGE;
                const uint32_t st = smem_u32(sm + s * STAGE);
                // refill the stage of step i-1 (once its MMAs are complete) with step i+2
                if (i >= 1 && i + 2 < nchunks) {
                    if (!(ok = bar_wait(mma2, (i - 1) & 1)))
                        break;
                    issue(i + 2);
                }
                // output pass: the state group's conversion (which follows the gating); state pass: gating
                if (!(ok = OUT ? bar_wait(ops_ready, ph) : bar_wait(&prep[s], (i / NSTAGE) & 1)))
                    break;
                fence_after();
                // (c) S^T += V^T k^^T : K = t (first, so the next chunk's state conversion can start early)
                for (int k = 0; k < C / 16; ++k)
                    mma_ss(tmem + TM_S, sdesc_sw128(st + ST_V + k * 32), sdesc_sw128(st + ST_G + k * 32),
                           ID_N128, (OUT || i > 0 || k > 0) ? 1u : 0u);
                mma_commit(mma_st);
                if (OUT) {
                    const uint32_t ob = tmem + TM_O + (i & 1) * 64;
                    if (i >= 2 && !(ok = bar_wait(&o_free[i & 1], ((i - 2) >> 1) & 1)))
                        break;
                    fence_after();
                    // (a) O^T = S'^T q~^T : A = S' (TMEM), B = q~ rows t, K = key
                    for (int k = 0; k < KD / 16; ++k)
                        mma_ts(ob, tmem + TM_SOP + (i & 1) * 64 + k * 8,
                               sdesc_sw128(st + (k >> 2) * 16384 + ST_Q0 + (k & 3) * 32), ID_N64, k > 0);
                    // (b) P = q~ k~^T : A = q~ (128-row view), B = k~ rows s
                    for (int k = 0; k < KD / 16; ++k)
                        mma_ss(tmem + TM_P, sdesc_sw128(st + (k >> 2) * 16384 + ST_Q0 + (k & 3) * 32),
                               sdesc_sw128(st + (k >> 2) * 16384 + ST_K0 + (k & 3) * 32), ID_N64, k > 0);
                    mma_commit(mma1);
                    if (!(ok = bar_wait(p_ready, ph)))
                        break;
                    fence_after();
                    // (d) O^T += V^T P^T : K = s
                    for (int k = 0; k < C / 16; ++k)
                        mma_ss(ob, sdesc_sw128(st + ST_V + k * 32), sdesc_sw128(pt + k * 32), ID_N64, 1);
                }
                mma_commit(mma2);
            }
            mma_commit(fin);
            bool drained = bar_wait(fin, 0);
            for (int s = 0; s < NSTAGE; ++s)
                if (last_issued[s] >= 0)
                    drained &= bar_wait(&full[s], (last_issued[s] / NSTAGE) & 1);
            if (!ok || !drained)
                report(a.status, GLA_ERR_TIMEOUT);
        }
    } else if (warp < WB) {
        // ---------------------------------------------------------------------- gating group (8 warps)
        // thread: key pair kp (keys 2kp, 2kp+1; value columns likewise), row quarter rq (rows 16rq..+15)
        const int kp = tid & 63, rq = tid >> 6;
        const int key = 2 * kp;
        const int kb = key >> 6, kc = key & 63;   // K-block and column inside the 128-byte row
        float *psum = reinterpret_cast<float *>(sm + OFF_PS);
        float D0 = 0.f, D1 = 0.f;                  // state pass: decay (log2) of the chunks already done
        for (int i = 0; i < nchunks; ++i) {
            const int s = i % NSTAGE;
            uint8_t *st = sm + s * STAGE;
            const int len = min(C, eos - (bos + chunk_of(i) * C));
            if (!(ok = bar_wait(&full[s], (i / NSTAGE) & 1)))
                break;
            // pass 1: this thread's g and v rows into registers (rows >= len are zero); log2 partial sums
            uint32_t gr[16], vr[16];
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int t = 16 * rq + u;
                const bool in = t < len;
                gr[u] = in ? *reinterpret_cast<const uint32_t *>(st + ST_G + t * 256 + kp * 4) : 0u;
                vr[u] = in ? *reinterpret_cast<const uint32_t *>(st + ST_V + t * 256 + kp * 4) : 0u;
                s0 = fmaf(bf_lo(gr[u]), L2E, s0);
                s1 = fmaf(bf_hi(gr[u]), L2E, s1);
            }
            float *ps = psum + (i & 1) * 512;
            ps[rq * 128 + key] = s0;
            ps[rq * 128 + key + 1] = s1;
            sync_gating();   // partial sums visible; every g / v tile read is done
            float p0[4], p1[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                p0[r] = ps[r * 128 + key];
                p1[r] = ps[r * 128 + key + 1];
            }
            const float ga0 = p0[0] + p0[1], ga1 = p1[0] + p1[1];                 // G(anchor = row 31)
            const float gl0 = ga0 + (p0[2] + p0[3]), gl1 = ga1 + (p1[2] + p1[3]);   // G(last row)
            float X0 = rq == 0 ? 0.f : rq == 1 ? p0[0] : rq == 2 ? ga0 : ga0 + p0[2];
            float X1 = rq == 0 ? 0.f : rq == 1 ? p1[0] : rq == 2 ? ga1 : ga1 + p1[2];
            uint32_t kh[16];
            uint8_t *qk = st + kb * 16384;
            if (OUT) {
                if (rq == 0) {
                    float *eg = reinterpret_cast<float *>(sm + OFF_EG + s * 1024);
                    eg[key] = ex2(ga0);
                    eg[key + 1] = ex2(ga1);
                    eg[128 + key] = ex2(gl0);
                    eg[128 + key + 1] = ex2(gl1);
                }
                const float cl0 = ex2(gl0 - ga0), cl1 = ex2(gl1 - ga1);
                // X relative to the anchor; swizzled offsets of this thread's column in rows 16rq + u
                X0 -= ga0;
                X1 -= ga1;
                uint32_t xo[8];
#pragma unroll
                for (int w = 0; w < 8; ++w)
                    xo[w] = sw128(16 * rq + w, kc);
                auto gate = [&](auto full_tag) {
                    constexpr bool FULL = decltype(full_tag)::value;
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int t = 16 * rq + u;
                        X0 = fmaf(bf_lo(gr[u]), L2E, X0);
                        X1 = fmaf(bf_hi(gr[u]), L2E, X1);
                        const uint32_t off = xo[u & 7] + (u >> 3) * 1024;
                        const uint32_t qw = *reinterpret_cast<const uint32_t *>(qk + ST_Q0 + off);
                        const uint32_t kw = *reinterpret_cast<const uint32_t *>(qk + ST_K0 + off);
                        float q0 = bf_lo(qw) * ex2(X0), q1 = bf_hi(qw) * ex2(X1);
                        float k0 = bf_lo(kw) * ex2(-X0), k1 = bf_hi(kw) * ex2(-X1);
                        if (!FULL && t >= len)
                            q0 = q1 = k0 = k1 = 0.f;
                        *reinterpret_cast<uint32_t *>(qk + ST_Q0 + off) = pack_h2(q0, q1);
                        *reinterpret_cast<uint32_t *>(qk + ST_K0 + off) = pack_h2(k0, k1);
                        kh[u] = pack_h2(k0 * cl0, k1 * cl1);
                        vr[u] = pack_h2(bf_lo(vr[u]), bf_hi(vr[u]));   // bf16 -> fp16
                    }
                };
                if (len == C)
                    gate(std::true_type{});
                else
                    gate(std::false_type{});
            } else {
                // k^ = k * 2^(G_last - G + D): this chunk's decay to its end, then the later chunks' decay
                const float e0 = gl0 + D0, e1 = gl1 + D1;
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int t = 16 * rq + u;
                    X0 = fmaf(bf_lo(gr[u]), L2E, X0);
                    X1 = fmaf(bf_hi(gr[u]), L2E, X1);
                    const uint32_t kw = *reinterpret_cast<const uint32_t *>(qk + ST_K0 + sw128(t, kc));
                    const bool in = t < len;
                    const float k0 = in ? bf_lo(kw) * ex2(e0 - X0) : 0.f;
                    const float k1 = in ? bf_hi(kw) * ex2(e1 - X1) : 0.f;
                    kh[u] = pack_h2(k0, k1);
                    vr[u] = pack_h2(bf_lo(vr[u]), bf_hi(vr[u]));
                }
                D0 = e0;
                D1 = e1;
            }
            // k^^T and V^T rows (key / value column 2kp and 2kp+1), columns t = 16rq.., over the g / v tiles
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int t0 = 16 * rq + 8 * jj;
                uint32_t k_lo[4], k_hi[4], v_lo[4], v_hi[4];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint32_t a0 = kh[8 * jj + 2 * w], a1 = kh[8 * jj + 2 * w + 1];
                    const uint32_t b0 = vr[8 * jj + 2 * w], b1 = vr[8 * jj + 2 * w + 1];
                    k_lo[w] = __byte_perm(a0, a1, 0x5410);
                    k_hi[w] = __byte_perm(a0, a1, 0x7632);
                    v_lo[w] = __byte_perm(b0, b1, 0x5410);
                    v_hi[w] = __byte_perm(b0, b1, 0x7632);
                }
                *reinterpret_cast<uint4 *>(st + ST_G + sw128(key, t0)) = make_uint4(k_lo[0], k_lo[1], k_lo[2], k_lo[3]);
                *reinterpret_cast<uint4 *>(st + ST_G + sw128(key + 1, t0)) = make_uint4(k_hi[0], k_hi[1], k_hi[2], k_hi[3]);
                *reinterpret_cast<uint4 *>(st + ST_V + sw128(key, t0)) = make_uint4(v_lo[0], v_lo[1], v_lo[2], v_lo[3]);
                *reinterpret_cast<uint4 *>(st + ST_V + sw128(key + 1, t0)) = make_uint4(v_hi[0], v_hi[1], v_hi[2], v_hi[3]);
            }
            fence_proxy_async();
            bar_arrive(&prep[s]);
        }
        if (ok && !OUT && vt == 0 && rq == 0) {
            float *gt = a.gtot + ((size_t)j * H + h) * KD;   // total decay of the segment, log2 units
            gt[key] = D0;
            gt[key + 1] = D1;
        }
        if (!ok)
            report(a.status, GLA_ERR_TIMEOUT);
    } else if (warp < WC) {
        // ---------------------------------------------------------------------- state group
        const int b = tid - NA;                                   // TMEM lane = value column
        const uint32_t lrow = static_cast<uint32_t>((warp & 3) * 32) << 16;
        // initial state of the segment -> TMEM (S^T[v][key] = S[key][v])
        {
            const size_t hoff = ((size_t)n * H + h) * KD * V;
            if (!OUT && p == 0 && a.h0 && a.h0c) {
                // keep a copy of this sequence's h0: the output pass reads it after ht (which may be the
                // same buffer) has been written by the sequence's last segment
                for (int k = 0; k < KD; ++k)
                    a.h0c[hoff + (size_t)k * V + v0 + b] = __ldg(a.h0 + hoff + (size_t)k * V + v0 + b);
            }
            const bool several = OUT && multi && !(p == 0 && eos == send);   // sequence has > 1 segment
            const float *h0p = nullptr;
            if (OUT && a.h0)
                h0p = several ? a.h0c + hoff : a.h0 + hoff;
            const bool scan = several && p > 0;
            if (several)
                grid_dep_wait();   // h0 copy and per-segment contributions come from the state pass
            const int j0 = j - p;
            // (the state pass starts its accumulator with the first MMA instead)
            for (int kc = 0; OUT && kc < KD / 32; ++kc) {
                uint32_t r[32];
                float acc[32];
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    acc[u] = h0p ? __ldg(h0p + (size_t)(kc * 32 + u) * V + v0 + b) : 0.f;
                if (scan) {
                    for (int m = 0; m < p; ++m) {
                        const size_t jm = (size_t)(j0 + m) * H + h;
                        const float *dS = a.ss + jm * KD * V + (size_t)(kc * 32) * V + v0 + b;
                        const float *gt = a.gtot + jm * KD + kc * 32;
#pragma unroll
                        for (int u = 0; u < 32; ++u)
                            acc[u] = fmaf(ex2(__ldg(gt + u)), acc[u], __ldg(dS + (size_t)u * V));
                    }
                }
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    r[u] = __float_as_uint(acc[u]);
                tmem_st32(tmem + lrow + TM_S + kc * 32, r);
            }
            if (OUT)
                tmem_wait_st();
        }
        if (OUT) {
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % NSTAGE;
                if (c > 0 && !(ok = bar_wait(mma_st, (c - 1) & 1)))   // the previous chunk's state update
                    break;
                if (!(ok = bar_wait(&prep[s], (c / NSTAGE) & 1)))
                    break;
                fence_after();
                const float *eg = reinterpret_cast<const float *>(sm + OFF_EG + s * 1024);
                // S' = diag(exp(G_a)) S (fp16 operand); S <- diag(exp(G_last)) S; 16 columns at a time with
                // the next load in flight
                uint32_t ra[16], rb[16];
                auto convert = [&](uint32_t(&r)[16], int q) {
                    uint32_t op[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float2 e = *reinterpret_cast<const float2 *>(eg + q * 16 + 2 * u);
                        op[u] = pack_h2(__uint_as_float(r[2 * u]) * e.x, __uint_as_float(r[2 * u + 1]) * e.y);
                    }
#pragma unroll
                    for (int u = 0; u < 16; u += 4) {
                        const float4 e = *reinterpret_cast<const float4 *>(eg + 128 + q * 16 + u);
                        r[u] = __float_as_uint(__uint_as_float(r[u]) * e.x);
                        r[u + 1] = __float_as_uint(__uint_as_float(r[u + 1]) * e.y);
                        r[u + 2] = __float_as_uint(__uint_as_float(r[u + 2]) * e.z);
                        r[u + 3] = __float_as_uint(__uint_as_float(r[u + 3]) * e.w);
                    }
                    tmem_st8(tmem + lrow + TM_SOP + (c & 1) * 64 + q * 8, op);
                    tmem_st16(tmem + lrow + TM_S + q * 16, r);
                };
                // two 16-column blocks per step, the next block's load in flight while one is converted
                tmem_ld16(tmem + lrow + TM_S, ra);
                tmem_wait_ld(ra);
#pragma unroll 1
                for (int q = 0; q < KD / 16; q += 2) {
                    tmem_ld16(tmem + lrow + TM_S + (q + 1) * 16, rb);
                    convert(ra, q);
                    tmem_wait_ld(rb);
                    if (q + 2 < KD / 16)
                        tmem_ld16(tmem + lrow + TM_S + (q + 2) * 16, ra);
                    convert(rb, q + 1);
                    if (q + 2 < KD / 16)
                        tmem_wait_ld(ra);
                }
                tmem_wait_st();
                fence_before();
                bar_arrive(ops_ready);
            }
        }

        // final state of the segment: ht (output pass, last segment) or dS (state pass), once every MMA
        // is complete.  (`fin` completes a single phase; the per-chunk barriers cannot be used here because
        // a parity wait only tells the current phase from the one before it, and the state pass's MMAs may
        // run any number of phases ahead of this group.)
        if (ok)
            ok = bar_wait(fin, 0);
        if (ok) {
            fence_after();
            float *dst = nullptr;
            if (OUT)
                dst = (eos == send && a.ht) ? a.ht + ((size_t)n * H + h) * KD * V : nullptr;
            else
                dst = a.ss + ((size_t)j * H + h) * KD * V;
            if (dst) {
                bool fin_ok = true;
                for (int kc = 0; kc < KD / 32; ++kc) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lrow + TM_S + kc * 32, r);
                    tmem_wait_ld(r);
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        const float x = __uint_as_float(r[u]);
                        fin_ok &= finite(x);
                        dst[(size_t)(kc * 32 + u) * V + v0 + b] = x;
                    }
                }
                if (!fin_ok)
                    report(a.status, GLA_ERR_RANGE);
            }
        }
        if (!ok)
            report(a.status, GLA_ERR_TIMEOUT);
    } else if (OUT) {
        // ---------------------------------------------------------------------- output group
        const int b = tid - NA - NB;   // TMEM lane: row t of P, value column of O^T
        const uint32_t lrow = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const bool leader = b == 0;
        float *ost = reinterpret_cast<float *>(sm + OFF_OST);
        Tout *go = static_cast<Tout *>(a.o);
        const size_t rstride = (size_t)H * V;
        float omax = 0.f;
        for (int c = 0; c < nchunks; ++c) {
            const int row0 = bos + c * C;
            const int len = min(C, eos - row0);
            // masked scores -> fp16 P[t][s] (lanes t < 64: the first two warps of the group)
            if (!(ok = bar_wait(mma1, c & 1)))
                break;
            fence_after();
            if ((warp & 3) < 2) {
                const int t = b;
                for (int sc = 0; sc < 2; ++sc) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lrow + TM_P + sc * 32, r);
                    tmem_wait_ld(r);
#pragma unroll
                    for (int u0 = 0; u0 < 32; u0 += 8) {
                        uint32_t pk[4];
#pragma unroll
                        for (int u = 0; u < 8; u += 2) {
                            const int sa = sc * 32 + u0 + u;
                            const float p0 = sa <= t ? __uint_as_float(r[u0 + u]) : 0.f;
                            const float p1 = sa + 1 <= t ? __uint_as_float(r[u0 + u + 1]) : 0.f;
                            pk[u / 2] = pack_h2(p0, p1);
                        }
                        *reinterpret_cast<uint4 *>(sm + OFF_P + sw128(t, sc * 32 + u0)) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
            }
            fence_proxy_async();
            fence_before();
            bar_arrive(p_ready);

            // output: o[t, v] = scale * O^T[v][t]
            if (!(ok = bar_wait(mma2, c & 1)))
                break;
            fence_after();
            const uint32_t ob = tmem + lrow + TM_O + (c & 1) * 64;
            const bool tma = sizeof(Tout) == 4 && len == C;
            for (int half = 0; half < 2; ++half) {
                uint32_t r[32];
                tmem_ld32(ob + half * 32, r);
                tmem_wait_ld(r);
                if (tma) {
                    if (leader)
                        bulk_wait_read();   // the previous store has read the staging buffer
                    sync_output();
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        const float x = a.scale * __uint_as_float(r[u]);
                        omax = amax_nan(omax, x);
                        ost[u * 128 + b] = x;
                    }
                    fence_proxy_async();
                    sync_output();
                    if (leader) {
                        tma_store_3d(&tm_o, ost, v0, h, row0 + half * 32);
                        bulk_commit();
                    }
                } else {
                    Tout *orow = go + ((size_t)row0 * H + h) * V + v0 + b;
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        const int t = half * 32 + u;
                        const float x = a.scale * __uint_as_float(r[u]);
                        if (t < len) {
                            omax = amax_nan(omax, x);
                            orow[(size_t)t * rstride] = to_out<Tout>(x);
                        }
                    }
                }
            }
            fence_before();
            bar_arrive(&o_free[c & 1]);
        }
        if (leader)
            bulk_wait_all();
        if (!finite(omax))
            report(a.status, GLA_ERR_RANGE);
        if (!ok)
            report(a.status, GLA_ERR_TIMEOUT);
    }

    fence_before();
    __syncthreads();
    if (warp == 0) {
        fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// [rows][H][D] tensor of bf16 or fp32; box = `inner` elements x 1 head x `brows` rows.
bool encode_rows(CUtensorMap *m, const void *ptr, int D, int H, long long rows, int inner, int brows, bool swizzle,
                 bool f32 = false)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t es = f32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)H * D * es};
    cuuint32_t box[3] = {(cuuint32_t)inner, 1, (cuuint32_t)brows};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr),
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool OUT, typename Tout>
cudaError_t launch_one(const Plan &pl, const Args &a, cudaStream_t s, bool pdl)
{
    const long long rows = pl.varlen ? (long long)pl.T : (long long)pl.B * pl.T;
    CUtensorMap mq, mk, mg, mv, mo;
    if (!encode_rows(&mq, a.q, pl.K, pl.H, rows, 64, C, true) || !encode_rows(&mk, a.k, pl.K, pl.H, rows, 64, C, true) ||
        !encode_rows(&mg, a.g, pl.K, pl.H, rows, 128, C, false) ||
        !encode_rows(&mv, a.v, pl.V, pl.H, rows, 128, C, false))
        return cudaErrorInvalidValue;
    // o: fp32 rows, box 128 x 1 x 32 (the output group's 16 KB staging buffer); unused for bf16 o
    if (!encode_rows(&mo, OUT && sizeof(Tout) == 4 ? a.o : a.v, pl.V, pl.H, rows, 128, 32, false,
                     OUT && sizeof(Tout) == 4))
        return cudaErrorInvalidValue;
    auto f = gla_tc<OUT, Tout>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.V / VT, pl.H, pl.J);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = pdl ? 1 : 0;
    int multi = pl.multi ? 1 : 0;
    void *args[] = {&mq, &mk, &mg, &mv, &mo, const_cast<Args *>(&a), &multi};
    cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(f), args);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(int dtype, int K, int V)
{
    return dtype != GLA_F32 && K == KD && V % VT == 0 && V <= 256;
}

cudaError_t launch_state_tc(const Plan &pl, const Args &a, cudaStream_t s)
{
    return launch_one<false, float>(pl, a, s, pl.varlen);
}

cudaError_t launch_out_tc(const Plan &pl, const Args &a, cudaStream_t s)
{
    const bool pdl = pl.multi || pl.varlen;   // a kernel of this call precedes it in the stream
    if (pl.dtype == GLA_BF16_OBF16)
        return launch_one<true, __nv_bfloat16>(pl, a, s, pdl);
    return launch_one<true, float>(pl, a, s, pdl);
}

}  // namespace gla
