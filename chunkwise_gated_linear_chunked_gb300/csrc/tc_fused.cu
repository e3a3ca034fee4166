// Persistent fused tensor-core kernel of the chunkwise GLA forward (bf16 or fp16 inputs, K = 128, V in
// {128, 256}).
//
// Method (page "fla/ops/gla/fused_chunk.py"): per chunk of C = 64 rows with chunk-local cumsum G of the gates
// (FusedChunkGLAFunction.forward, kernel a), the state contribution (k*exp(G_last-G))^T V (prepare_qg_kg,
// fused_chunk_gla_fwd_kernel: kernel b), and the output = inter-chunk term (q*exp(G)) S plus the causally
// masked intra-chunk term with the inclusive diagonal (fwd_inner_chunk and the A @ v product of
// FusedChunkGLAFunction.forward: kernel d), scale applied to the sum.  A long sequence is cut into segments
// whose states are chained by the decayed scan S_out(p) = diag(exp(Gtot(p))) S_in(p) + dS(p),
// S_in(p+1) = S_out(p), S_in(0) = h0 (kernel c).
//
// Work item = (segment slot, head, 128-wide value tile), claimed from a global counter in order, so the
// item of a segment's predecessor was always claimed earlier by a running CTA.  For an item whose segment is
// not the last of its sequence the CTA
//   1. walks the segment's chunks last to first and accumulates dS = sum_t k_t^T v_t exp(G_end - G_t) in
//      TMEM with no rescaling (the later chunks' decay is folded into k^ <= |k|),
//   2. finds its start state S_in from the predecessors' published contributions and end states by a
//      fixed two-level scan (blocks of lb segments; workspace flags, cleared before each call; segment 0
//      reads h0) and publishes its own contribution or end state, and
//   3. runs the output pass over the same chunks, first to last, while they are still in L2.
// The last segment of a sequence skips 1. and 2.'s publication and writes ht at the end.  One segment per
// sequence is the plain single pass.
//
// MMAs (M = 128; the state lives in TMEM transposed, lane = value column v, column = key dimension):
//   (c) S^T += V^T   k^^T     A = V^T [v][t]  (K-major, smem), B = k^^T [key][t] (K-major, smem)
//   (a) O^T  = S'^T  q~^T      A = S' from TMEM (fp16),        B = q~  [t][key]   (K-major, smem)
//   (b) P    = q~    k~^T      A = q~ (rows 64..127 unused),   B = k~  [s][key]   (K-major, smem)
//   (d) O^T += V^T   P^T      A = V^T [v][s],                  B = P   [t][s]     (K-major, smem)
// q~ = q*exp(G-G_a), k~ = k*exp(G_a-G), k^ = k*exp(G_last-G), S' = diag(exp(G_a)) S, anchor a = row 31.
// Operands are fp16 (bf16 inputs widen exactly; 11-bit significands keep the result within the parity bounds
// where single-rounded bf16 operands do not); accumulation is fp32 in TMEM; gates are summed in log2 units.
//
// Roles: warps 0-7 gating (cumsum, gating, operand conversion in place in the TMA stage); warps 8-11 state
// (S' and decay per chunk, final state); warps 12-15 output (P, O^T -> smem -> TMA store); warps 8-15
// together run the start-state scan of an item; warp 16 lane 0 issues the MMAs, warp 17 lane 0 the TMA
// loads (three 64 KB stages, freed by MMA commits).  Every wait is bounded and a CTA-wide abort word ends
// all roles quickly after the first failure (GLA_ERR_TIMEOUT); non-finite outputs report GLA_ERR_RANGE.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <type_traits>

#include "gla_internal.h"
#include "tc_ptx.cuh"

namespace gla {
namespace {

using namespace tc;

constexpr int C = 64;
constexpr int KD = 128;
constexpr int VT = 128;
constexpr int NA = 256;          // gating group
constexpr int NB = 128;          // state group
constexpr int NC = 128;          // output group
constexpr int WB = NA / 32, WC = (NA + NB) / 32, WCTL = (NA + NB + NC) / 32, WPRD = WCTL + 1;
constexpr int CTL = NA + NB + NC;   // MMA issue thread
constexpr int NTHREADS = NA + NB + NC + 64;
constexpr float L2E = 1.4426950408889634f;
constexpr uint32_t kEpochMask = 0x3FFFFFFFu;   // a flag holds (epoch << 2) | kind

constexpr int NSTAGE = 3;
constexpr int STAGE = 65536;
constexpr int ST_Q0 = 0, ST_K0 = 8192, ST_G = 32768, ST_V = 49152;
constexpr int OFF_P = NSTAGE * STAGE;             // P [t][s] fp16, 8 KB
constexpr int OFF_EG = OFF_P + 8192;              // per stage: exp(G_a)[128], exp(G_last)[128]
constexpr int OFF_PS = OFF_EG + NSTAGE * 1024;    // gating partial sums [2][4][128]
constexpr int OFF_OST = OFF_PS + 4096;            // output staging, 32 rows x 128 fp32
constexpr int OFF_GT = OFF_OST + 16384;           // segment decay (log2) per key, [128]
constexpr int OFF_WL = OFF_GT + 512;             // look-back: running log2 weight per key, [128]
constexpr int OFF_MISC = OFF_WL + 512;            // item slot, abort word, look-back flag value
constexpr int OFF_BAR = OFF_MISC + 64;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;

constexpr uint32_t TM_S = 0, TM_SOP = 128, TM_O = 256, TM_P = 384, TM_COLS = 512;
constexpr uint32_t ID_N64 = idesc_f16_f32(128, 64);
constexpr uint32_t ID_N128 = idesc_f16_f32(128, 128);

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}
// A 32-bit word of two 16-bit inputs: widened halves, and the pair as an fp16 operand word (bf16 rounds
// once to fp16; fp16 inputs are already in operand form).
template <typename Tin>
struct In;
template <>
struct In<__nv_bfloat16> {
    static __device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
    static __device__ __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
    static __device__ __forceinline__ uint32_t op(uint32_t w);
};
template <>
struct In<__half> {
    static __device__ __forceinline__ float lo(uint32_t w)
    {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
    }
    static __device__ __forceinline__ float hi(uint32_t w)
    {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
    }
    static __device__ __forceinline__ uint32_t op(uint32_t w) { return w; }
};
__device__ __forceinline__ uint32_t In<__nv_bfloat16>::op(uint32_t w) { return pack_h2(lo(w), hi(w)); }
__device__ __forceinline__ bool finite(float x) { return fabsf(x) <= 3.402823466e38f; }
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
// the chain team: state and output groups together
__device__ __forceinline__ void sync_team() { asm volatile("bar.sync 4, %0;" ::"n"(NB + NC) : "memory"); }
__device__ __forceinline__ bool team_all(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 4, %2, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v), "n"(NB + NC)
                 : "memory");
    return r != 0;
}
__device__ __forceinline__ float4 f4(const uint32_t *r)
{
    return make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]), __uint_as_float(r[2]), __uint_as_float(r[3]));
}

template <typename Tin, typename Tout, bool HF>
__global__ void __launch_bounds__(NTHREADS, 1)
    gla_fused(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_o, Args a, int nitems)
{
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *full = bars + 0, *prep = bars + 3;
    uint64_t *ops_ready = bars + 6, *p_ready = bars + 7, *mma_st = bars + 8, *mma1 = bars + 9, *mma2 = bars + 10;
    uint64_t *o_free = bars + 11;                                   // [2]
    uint64_t *mma_a = bars + 13, *a_done = bars + 14, *g_done = bars + 15, *tmem_free = bars + 16;
    uint64_t *item_done = bars + 17;
    uint64_t *empty = bars + 18;                                    // [3]: stage free again
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 21);
    volatile int *misc = reinterpret_cast<volatile int *>(sm + OFF_MISC);   // [0] item, [1] abort, [2] flag
    volatile int *abort_w = misc + 1;
    float *gts = reinterpret_cast<float *>(sm + OFF_GT);
    float *wl = reinterpret_cast<float *>(sm + OFF_WL);

    if (a.table)
        grid_dep_wait();   // the varlen slot table comes from the preceding plan kernel
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // launch epoch: publication flags of this launch carry it, so flags left by earlier launches need no
    // clearing; the last CTA out advances it (no CTA can still be starting by then)
    const uint32_t tag = static_cast<uint32_t>(*reinterpret_cast<volatile int *>(a.ctr + 2)) & kEpochMask;
    const int H = a.H, V = a.V, NV = V / VT;

    if (warp == 0)
        tmem_alloc(tmem_slot, TM_COLS);
    if (tid == CTL) {
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
        bar_init(mma_a, 1);
        bar_init(a_done, 1);
        bar_init(g_done, NA);
        bar_init(tmem_free, NB);
        bar_init(item_done, 1);
        for (int s = 0; s < NSTAGE; ++s)
            bar_init(&empty[s], 1);
        bar_fence_init();
        misc[1] = 0;
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_g);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_o);
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;

    // CTA-wide running counts (identical in every role): chunks through the stage ring, output-pass chunks,
    // state-pass chunks, items with a state pass, items completed
    int qbase = 0, nbbase = 0, nabase = 0, naitems = 0, items = 0;
    // per-role persistent state
    float omax = 0.f;

    for (;;) {
        if (tid == CTL)
            misc[0] = atomicAdd(a.ctr + 0, 1);
        __syncthreads();
        const int u = misc[0];
        const bool stop = u < 0 || u >= nitems || *abort_w;
        __syncthreads();   // every thread has read the slot before the next claim
        if (stop)
            break;
        const int j = u / (H * NV), rem = u - j * (H * NV), h = rem / NV, vt = rem - h * NV;
        int n, p, bos, eos, send;
        if (!resolve_slot(a, j, n, p, bos, eos, send))
            continue;   // unused varlen slot (uniform across the CTA)
        const int v0 = vt * VT;
        const int nchunks = (eos - bos + C - 1) / C;
        const bool last = eos == send;
        const int nA = last ? 0 : nchunks;   // state-pass chunks (reverse order)
        const int nQ = nA + nchunks;         // chunks through the ring: state pass, then output pass
        auto chunk_of = [&](int q) { return q < nA ? nA - 1 - q : q - nA; };

        // ---------------------------------------------------------------------- chain team
        // Start state of the item's segment into TMEM S.  Segments are grouped in blocks of lb; the first
        // segment of a block (a boundary, p % lb == 0) publishes its end state S_out = 2^Gtot S_in + dS
        // (flag 2), every other segment with a state pass publishes its contribution dS and decay Gtot
        // (flag 1) as soon as the pass is done.  With p0 the last boundary before p,
        //   S_in(p) = sum_{i = p-1 .. p0+1} 2^(Gtot(p-1) + ... + Gtot(i+1)) dS(i) + 2^(Gtot(p-1) + ... + Gtot(p0+1)) S_out(p0),
        // summed newest first, and S_in(0) = h0.  The grouping is fixed, so the result does not depend on
        // timing; lb = 1 is the plain serial chain (one tile read and one written per segment), a larger lb
        // shortens the chain of dependent publications when all items run at once.
        // 256 threads, lane = value column; the state group takes keys 0..63, the output group 64..127.
        // TMEM S' (free until the output pass) accumulates the sum.  Published tiles are key-interleaved
        // (float4 of 4 keys per value column) so a warp reads 512 contiguous bytes per load.
        auto chain = [&]() -> bool {
            const int half = warp >= WC ? 1 : 0;
            const int b = tid - NA - half * NB;
            const int kb0 = 64 * half;
            const uint32_t lrow = static_cast<uint32_t>((warp & 3) * 32) << 16;
            const bool leader = tid == NA;
            const size_t tile = (size_t)KD * VT;
            const size_t mine = ((size_t)j * H + h) * NV + vt;
            const int HN = H * NV;
            const bool boundary = p % a.lb == 0;
            const size_t soff = ((size_t)n * H + h) * KD * V + v0 + b;
            // the first segment of a sequence with a state pass stages h0 in TMEM S' while the pass runs
            const bool h0pre = p == 0 && nA > 0 && a.h0 != nullptr;
            if (h0pre) {
                for (int sub = 0; sub < 4; ++sub) {
                    const int k1 = kb0 + 16 * sub;
                    uint32_t x[16];
#pragma unroll
                    for (int uu = 0; uu < 16; ++uu)
                        x[uu] = __float_as_uint(__ldcg(a.h0 + soff + (size_t)(k1 + uu) * V));
                    tmem_st16(tmem + lrow + TM_SOP + k1, x);
                }
                tmem_wait_st();
            }
            bool ok = true;
            if (nA > 0)
                ok = bar_wait(g_done, naitems & 1, abort_w) && bar_wait(a_done, naitems & 1, abort_w);
            if (!team_all(ok))
                return false;
            fence_after();
            if (nA > 0 && !boundary) {
                float4 *dst = reinterpret_cast<float4 *>(a.agg + mine * tile);
                for (int sub = 0; sub < 4; ++sub) {
                    const int k0 = kb0 + 16 * sub;
                    uint32_t r[16];
                    tmem_ld16(tmem + lrow + TM_S + k0, r);
                    tmem_wait_ld(r);
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        __stcg(dst + (size_t)(k0 / 4 + w) * VT + b, f4(r + 4 * w));
                }
                if (b < 64)
                    __stcg(a.gtot + mine * KD + kb0 + b, gts[kb0 + b]);
                __threadfence();
                sync_team();
                if (leader)
                    flag_set(a.flags + u, static_cast<int>(tag << 2 | 1u));
            }
            const int p0 = p > 0 ? (p - 1) / a.lb * a.lb : 0;
            if (p > 0) {
                if (b < 64)
                    wl[kb0 + b] = 0.f;
                for (int i = p - 1; i > p0; --i) {
                    const int back = p - i;
                    if (leader)
                        misc[2] = flag_wait_tag(a.flags + (u - back * HN), tag, 1, abort_w);
                    sync_team();
                    if (misc[2] == 0)
                        return false;   // uniform: every thread read the same value
                    const size_t ti = mine - (size_t)back * HN;
                    const float4 *src = reinterpret_cast<const float4 *>(a.agg + ti * tile);
                    const float gi = b < 64 ? __ldcg(a.gtot + ti * KD + kb0 + b) : 0.f;
                    for (int sub = 0; sub < 2; ++sub) {
                        // 32 keys of loads in flight, consumed 16 TMEM columns at a time
                        const int k0 = kb0 + 32 * sub;
                        float4 x[8];
#pragma unroll
                        for (int w = 0; w < 8; ++w)
                            x[w] = __ldcg(src + (size_t)(k0 / 4 + w) * VT + b);
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int k1 = k0 + 16 * hh;
                            uint32_t r[16];
                            if (back > 1) {
                                tmem_ld16(tmem + lrow + TM_SOP + k1, r);
                                tmem_wait_ld(r);
                            } else {
#pragma unroll
                                for (int uu = 0; uu < 16; ++uu)
                                    r[uu] = 0u;
                            }
#pragma unroll
                            for (int w = 0; w < 4; ++w) {
                                const float4 e = *reinterpret_cast<const float4 *>(wl + k1 + 4 * w);
                                const float4 xv = x[4 * hh + w];
                                r[4 * w] = __float_as_uint(fmaf(ex2(e.x), xv.x, __uint_as_float(r[4 * w])));
                                r[4 * w + 1] = __float_as_uint(fmaf(ex2(e.y), xv.y, __uint_as_float(r[4 * w + 1])));
                                r[4 * w + 2] = __float_as_uint(fmaf(ex2(e.z), xv.z, __uint_as_float(r[4 * w + 2])));
                                r[4 * w + 3] = __float_as_uint(fmaf(ex2(e.w), xv.w, __uint_as_float(r[4 * w + 3])));
                            }
                            tmem_st16(tmem + lrow + TM_SOP + k1, r);
                        }
                    }
                    tmem_wait_st();
                    sync_team();   // every thread has used this step's weights
                    if (b < 64)
                        wl[kb0 + b] += gi;
                }
                // the end state of the block's boundary segment
                if (leader)
                    misc[2] = flag_wait_tag(a.flags + (u - (p - p0) * HN), tag, 2, abort_w);
                sync_team();
                if (misc[2] == 0)
                    return false;
            }
            // S_in -> TMEM S; a boundary segment with a state pass publishes S_out = 2^Gtot * S_in + dS
            const bool acc = p - 1 > p0;   // contributions were summed into TMEM S'
            const bool pub = nA > 0 && boundary;
            const float4 *bsrc = reinterpret_cast<const float4 *>(a.ss + (mine - (size_t)(p - p0) * HN) * tile);
            float4 *bdst = reinterpret_cast<float4 *>(a.ss + mine * tile);
#pragma unroll 1
            for (int sub = 0; sub < 4; ++sub) {
                const int k1 = kb0 + 16 * sub;
                uint32_t sn[16];
                if (p > 0) {
                    float4 x[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        x[w] = __ldcg(bsrc + (size_t)(k1 / 4 + w) * VT + b);
                    if (acc) {
                        tmem_ld16(tmem + lrow + TM_SOP + k1, sn);
                        tmem_wait_ld(sn);
                    } else {
#pragma unroll
                        for (int uu = 0; uu < 16; ++uu)
                            sn[uu] = 0u;
                    }
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float4 e = *reinterpret_cast<const float4 *>(wl + k1 + 4 * w);
                        sn[4 * w] = __float_as_uint(fmaf(ex2(e.x), x[w].x, __uint_as_float(sn[4 * w])));
                        sn[4 * w + 1] = __float_as_uint(fmaf(ex2(e.y), x[w].y, __uint_as_float(sn[4 * w + 1])));
                        sn[4 * w + 2] = __float_as_uint(fmaf(ex2(e.z), x[w].z, __uint_as_float(sn[4 * w + 2])));
                        sn[4 * w + 3] = __float_as_uint(fmaf(ex2(e.w), x[w].w, __uint_as_float(sn[4 * w + 3])));
                    }
                } else if (h0pre) {
                    tmem_ld16(tmem + lrow + TM_SOP + k1, sn);
                    tmem_wait_ld(sn);
                } else if (a.h0) {
#pragma unroll
                    for (int uu = 0; uu < 16; ++uu)
                        sn[uu] = __float_as_uint(__ldcg(a.h0 + soff + (size_t)(k1 + uu) * V));
                } else {
#pragma unroll
                    for (int uu = 0; uu < 16; ++uu)
                        sn[uu] = 0u;
                }
                if (pub) {
                    uint32_t r[16];
                    tmem_ld16(tmem + lrow + TM_S + k1, r);
                    tmem_wait_ld(r);
#pragma unroll
                    for (int uu = 0; uu < 16; ++uu)
                        r[uu] = __float_as_uint(fmaf(ex2(gts[k1 + uu]), __uint_as_float(sn[uu]), __uint_as_float(r[uu])));
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        __stcg(bdst + (size_t)(k1 / 4 + w) * VT + b, f4(r + 4 * w));
                }
                tmem_st16(tmem + lrow + TM_S + k1, sn);
            }
            tmem_wait_st();
            if (pub)
                __threadfence();
            fence_before();
            sync_team();
            fence_after();
            if (pub && leader)
                flag_set(a.flags + u, static_cast<int>(tag << 2 | 2u));
            return true;
        };

        if (warp == WPRD) {
            // ------------------------------------------------------------------ TMA producer
            if (lane == 0) {
                bool ok = true;
                for (int q = 0; q < nQ; ++q) {
                    const int gq = qbase + q, s = gq % NSTAGE;
                    // the stage is free once the MMAs of the chunk three places earlier are complete
                    if (gq >= NSTAGE && !(ok = bar_wait(&empty[s], (gq / NSTAGE - 1) & 1, abort_w)))
                        break;
                    uint8_t *st = sm + s * STAGE;
                    const int row0 = bos + chunk_of(q) * C;
                    // tensor-map coordinates of the chunk: (head, row) time-major, (row in sequence,
                    // sequence * H + head) head-first
                    const int tc1 = HF ? row0 - n * a.T : h, tc2 = HF ? n * H + h : row0;
                    const bool out = q >= nA;
                    bar_expect_tx(&full[s], (out ? 4 : 3) * 16384);
                    if (out) {
                        tma_load_3d(st + ST_Q0, &tm_q, 0, tc1, tc2, &full[s]);
                        tma_load_3d(st + 16384 + ST_Q0, &tm_q, 64, tc1, tc2, &full[s]);
                    }
                    tma_load_3d(st + ST_K0, &tm_k, 0, tc1, tc2, &full[s]);
                    tma_load_3d(st + 16384 + ST_K0, &tm_k, 64, tc1, tc2, &full[s]);
                    tma_load_3d(st + ST_G, &tm_g, 0, tc1, tc2, &full[s]);
                    tma_load_3d(st + ST_V, &tm_v, v0, tc1, tc2, &full[s]);
                }
                if (!ok) {
                    *abort_w = 1;
                    report(a.status, GLA_ERR_TIMEOUT);
                }
            }
        } else if (warp == WCTL) {
            // ------------------------------------------------------------------ MMA issue
            if (lane == 0) {
                bool ok = true;
                // the previous item's MMAs are complete and its final state has been read once the state
                // group releases TMEM S
                if (items > 0)
                    ok = bar_wait(tmem_free, (items - 1) & 1, abort_w);
                const uint32_t pt = smem_u32(sm + OFF_P);
                for (int q = 0; ok && q < nQ; ++q) {
                    const int s = (qbase + q) % NSTAGE;
                    const uint32_t st = smem_u32(sm + s * STAGE);
                    if (q < nA) {
                        if (!(ok = bar_wait(&prep[s], ((qbase + q) / NSTAGE) & 1, abort_w)))
                            break;
                        fence_after();
                        for (int k = 0; k < C / 16; ++k)
                            mma_ss(tmem + TM_S, sdesc_sw128(st + ST_V + k * 32), sdesc_sw128(st + ST_G + k * 32),
                                   ID_N128, (q > 0 || k > 0) ? 1u : 0u);
                        mma_commit(mma_a);
                        mma_commit(&empty[s]);
                        if (q == nA - 1)
                            mma_commit(a_done);
                    } else {
                        const int gb = nbbase + q - nA;   // CTA-wide output-pass chunk index
                        if (!(ok = bar_wait(ops_ready, gb & 1, abort_w)))
                            break;
                        fence_after();
                        for (int k = 0; k < C / 16; ++k)
                            mma_ss(tmem + TM_S, sdesc_sw128(st + ST_V + k * 32), sdesc_sw128(st + ST_G + k * 32),
                                   ID_N128, 1);
                        mma_commit(mma_st);
                        const uint32_t ob = tmem + TM_O + (gb & 1) * 64;
                        if (gb >= 2 && !(ok = bar_wait(&o_free[gb & 1], ((gb - 2) >> 1) & 1, abort_w)))
                            break;
                        fence_after();
                        for (int k = 0; k < KD / 16; ++k)
                            mma_ts(ob, tmem + TM_SOP + (gb & 1) * 64 + k * 8,
                                   sdesc_sw128(st + (k >> 2) * 16384 + ST_Q0 + (k & 3) * 32), ID_N64, k > 0);
                        for (int k = 0; k < KD / 16; ++k)
                            mma_ss(tmem + TM_P, sdesc_sw128(st + (k >> 2) * 16384 + ST_Q0 + (k & 3) * 32),
                                   sdesc_sw128(st + (k >> 2) * 16384 + ST_K0 + (k & 3) * 32), ID_N64, k > 0);
                        mma_commit(mma1);
                        if (!(ok = bar_wait(p_ready, gb & 1, abort_w)))
                            break;
                        fence_after();
                        for (int k = 0; k < C / 16; ++k)
                            mma_ss(ob, sdesc_sw128(st + ST_V + k * 32), sdesc_sw128(pt + k * 32), ID_N64, 1);
                        mma_commit(mma2);
                        mma_commit(&empty[s]);
                    }
                }
                mma_commit(item_done);
                if (!ok) {
                    *abort_w = 1;
                    report(a.status, GLA_ERR_TIMEOUT);
                }
            }
        } else if (warp < WB) {
            // ------------------------------------------------------------------ gating group (8 warps)
            const int kp = tid & 63, rq = tid >> 6;
            const int key = 2 * kp;
            const int kb = key >> 6, kc = key & 63;
            float *psum = reinterpret_cast<float *>(sm + OFF_PS);
            uint32_t xo[8];
#pragma unroll
            for (int w = 0; w < 8; ++w)
                xo[w] = sw128(16 * rq + w, kc);
            float D0 = 0.f, D1 = 0.f;   // state pass: decay (log2) of the chunks already walked
            for (int q = 0; q < nQ; ++q) {
                const int gq = qbase + q;
                const int s = gq % NSTAGE;
                uint8_t *st = sm + s * STAGE;
                const int len = min(C, eos - (bos + chunk_of(q) * C));
                if (!bar_wait(&full[s], (gq / NSTAGE) & 1, abort_w))
                    break;
                uint32_t gr[16], vr[16];
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int uu = 0; uu < 16; ++uu) {
                    const int t = 16 * rq + uu;
                    const bool in = t < len;
                    gr[uu] = in ? *reinterpret_cast<const uint32_t *>(st + ST_G + t * 256 + kp * 4) : 0u;
                    vr[uu] = in ? *reinterpret_cast<const uint32_t *>(st + ST_V + t * 256 + kp * 4) : 0u;
                    s0 = fmaf(In<Tin>::lo(gr[uu]), L2E, s0);
                    s1 = fmaf(In<Tin>::hi(gr[uu]), L2E, s1);
                }
                float *ps = psum + (gq & 1) * 512;
                ps[rq * 128 + key] = s0;
                ps[rq * 128 + key + 1] = s1;
                sync_gating();
                float p0[4], p1[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    p0[r] = ps[r * 128 + key];
                    p1[r] = ps[r * 128 + key + 1];
                }
                const float ga0 = p0[0] + p0[1], ga1 = p1[0] + p1[1];
                const float gl0 = ga0 + (p0[2] + p0[3]), gl1 = ga1 + (p1[2] + p1[3]);
                float X0 = rq == 0 ? 0.f : rq == 1 ? p0[0] : rq == 2 ? ga0 : ga0 + p0[2];
                float X1 = rq == 0 ? 0.f : rq == 1 ? p1[0] : rq == 2 ? ga1 : ga1 + p1[2];
                uint32_t kh[16];
                uint8_t *qk = st + kb * 16384;
                if (q >= nA) {
                    // output pass: q~, k~ in place; k^ = k~ * exp(G_last - G_a)
                    if (rq == 0) {
                        float *eg = reinterpret_cast<float *>(sm + OFF_EG + s * 1024);
                        eg[key] = ex2(ga0);
                        eg[key + 1] = ex2(ga1);
                        eg[128 + key] = ex2(gl0);
                        eg[128 + key + 1] = ex2(gl1);
                    }
                    const float cl0 = ex2(gl0 - ga0), cl1 = ex2(gl1 - ga1);
                    X0 -= ga0;
                    X1 -= ga1;
                    auto gate = [&](auto full_tag) {
                        constexpr bool FULL = decltype(full_tag)::value;
#pragma unroll
                        for (int uu = 0; uu < 16; ++uu) {
                            const int t = 16 * rq + uu;
                            X0 = fmaf(In<Tin>::lo(gr[uu]), L2E, X0);
                            X1 = fmaf(In<Tin>::hi(gr[uu]), L2E, X1);
                            const uint32_t off = xo[uu & 7] + (uu >> 3) * 1024;
                            const uint32_t qw = *reinterpret_cast<const uint32_t *>(qk + ST_Q0 + off);
                            const uint32_t kw = *reinterpret_cast<const uint32_t *>(qk + ST_K0 + off);
                            float q0 = In<Tin>::lo(qw) * ex2(X0), q1 = In<Tin>::hi(qw) * ex2(X1);
                            float k0 = In<Tin>::lo(kw) * ex2(-X0), k1 = In<Tin>::hi(kw) * ex2(-X1);
                            if (!FULL && t >= len)
                                q0 = q1 = k0 = k1 = 0.f;
                            *reinterpret_cast<uint32_t *>(qk + ST_Q0 + off) = pack_h2(q0, q1);
                            *reinterpret_cast<uint32_t *>(qk + ST_K0 + off) = pack_h2(k0, k1);
                            kh[uu] = pack_h2(k0 * cl0, k1 * cl1);
                            vr[uu] = In<Tin>::op(vr[uu]);
                        }
                    };
                    if (len == C)
                        gate(std::true_type{});
                    else
                        gate(std::false_type{});
                } else {
                    // state pass: k^ = k * 2^(G_last - G + D)
                    const float e0 = gl0 + D0, e1 = gl1 + D1;
#pragma unroll
                    for (int uu = 0; uu < 16; ++uu) {
                        const int t = 16 * rq + uu;
                        X0 = fmaf(In<Tin>::lo(gr[uu]), L2E, X0);
                        X1 = fmaf(In<Tin>::hi(gr[uu]), L2E, X1);
                        const uint32_t kw =
                            *reinterpret_cast<const uint32_t *>(qk + ST_K0 + xo[uu & 7] + (uu >> 3) * 1024);
                        const bool in = t < len;
                        const float k0 = in ? In<Tin>::lo(kw) * ex2(e0 - X0) : 0.f;
                        const float k1 = in ? In<Tin>::hi(kw) * ex2(e1 - X1) : 0.f;
                        kh[uu] = pack_h2(k0, k1);
                        vr[uu] = In<Tin>::op(vr[uu]);
                    }
                    D0 = e0;
                    D1 = e1;
                }
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
                if (q == nA - 1 && rq == 0) {
                    gts[key] = D0;   // the segment's total decay, for the chain step
                    gts[key + 1] = D1;
                }
                fence_proxy_async();
                bar_arrive(&prep[s]);
                if (q == nA - 1)
                    bar_arrive(g_done);
            }
        } else if (warp < WC) {
            // ------------------------------------------------------------------ state group
            const int b = tid - NA;
            const uint32_t lrow = static_cast<uint32_t>((warp & 3) * 32) << 16;
            const size_t soff = ((size_t)n * H + h) * KD * V + v0 + b;   // ht column of this lane
            bool ok = chain();
            // output pass: per chunk S' = diag(exp(G_a)) S (fp16), S <- diag(exp(G_last)) S
            for (int c = 0; ok && c < nchunks; ++c) {
                const int gq = qbase + nA + c, gb = nbbase + c;
                const int s = gq % NSTAGE;
                if (c > 0 && !(ok = bar_wait(mma_st, (gb - 1) & 1, abort_w)))
                    break;
                if (!(ok = bar_wait(&prep[s], (gq / NSTAGE) & 1, abort_w)))
                    break;
                fence_after();
                const float *eg = reinterpret_cast<const float *>(sm + OFF_EG + s * 1024);
                uint32_t ra[16], rb[16];
                auto convert = [&](uint32_t(&r)[16], int qq) {
                    uint32_t op[8];
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const float2 e = *reinterpret_cast<const float2 *>(eg + qq * 16 + 2 * w);
                        op[w] = pack_h2(__uint_as_float(r[2 * w]) * e.x, __uint_as_float(r[2 * w + 1]) * e.y);
                    }
#pragma unroll
                    for (int w = 0; w < 16; w += 4) {
                        const float4 e = *reinterpret_cast<const float4 *>(eg + 128 + qq * 16 + w);
                        r[w] = __float_as_uint(__uint_as_float(r[w]) * e.x);
                        r[w + 1] = __float_as_uint(__uint_as_float(r[w + 1]) * e.y);
                        r[w + 2] = __float_as_uint(__uint_as_float(r[w + 2]) * e.z);
                        r[w + 3] = __float_as_uint(__uint_as_float(r[w + 3]) * e.w);
                    }
                    tmem_st8(tmem + lrow + TM_SOP + (gb & 1) * 64 + qq * 8, op);
                    tmem_st16(tmem + lrow + TM_S + qq * 16, r);
                };
                tmem_ld16(tmem + lrow + TM_S, ra);
                tmem_wait_ld(ra);
#pragma unroll 1
                for (int qq = 0; qq < KD / 16; qq += 2) {
                    tmem_ld16(tmem + lrow + TM_S + (qq + 1) * 16, rb);
                    convert(ra, qq);
                    tmem_wait_ld(rb);
                    if (qq + 2 < KD / 16)
                        tmem_ld16(tmem + lrow + TM_S + (qq + 2) * 16, ra);
                    convert(rb, qq + 1);
                    if (qq + 2 < KD / 16)
                        tmem_wait_ld(ra);
                }
                tmem_wait_st();
                fence_before();
                bar_arrive(ops_ready);
            }
            // end of the item: final state (ht for a sequence's last segment), then release TMEM S
            if (ok)
                ok = bar_wait(item_done, items & 1, abort_w);
            if (ok && last && a.ht) {
                fence_after();
                float *dst = a.ht + soff;
                float fmax = 0.f;
                for (int kc = 0; kc < KD / 32; ++kc) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lrow + TM_S + kc * 32, r);
                    tmem_wait_ld(r);
#pragma unroll
                    for (int uu = 0; uu < 32; ++uu) {
                        const float x = __uint_as_float(r[uu]);
                        fmax = amax_nan(fmax, x);
                        dst[(size_t)(kc * 32 + uu) * V] = x;
                    }
                }
                if (!finite(fmax))
                    report(a.status, GLA_ERR_RANGE);
            }
            fence_before();
            bar_arrive(tmem_free);
            if (!ok)
                report(a.status, GLA_ERR_TIMEOUT);
        } else {
            // ------------------------------------------------------------------ output group
            const int b = tid - NA - NB;
            const uint32_t lrow = static_cast<uint32_t>((warp & 3) * 32) << 16;
            const bool leader = b == 0;
            float *ost = reinterpret_cast<float *>(sm + OFF_OST);
            Tout *go = static_cast<Tout *>(a.o);
            const size_t rstride = HF ? (size_t)V : (size_t)H * V;   // between consecutive rows of o
            bool ok = chain();
            for (int c = 0; ok && c < nchunks; ++c) {
                const int gb = nbbase + c;
                const int row0 = bos + c * C;
                const int len = min(C, eos - row0);
                if (!(ok = bar_wait(mma1, gb & 1, abort_w)))
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
                            for (int w = 0; w < 8; w += 2) {
                                const int sa = sc * 32 + u0 + w;
                                const float p0 = sa <= t ? __uint_as_float(r[u0 + w]) : 0.f;
                                const float p1 = sa + 1 <= t ? __uint_as_float(r[u0 + w + 1]) : 0.f;
                                pk[w / 2] = pack_h2(p0, p1);
                            }
                            *reinterpret_cast<uint4 *>(sm + OFF_P + sw128(t, sc * 32 + u0)) =
                                make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        }
                    }
                }
                fence_proxy_async();
                fence_before();
                bar_arrive(p_ready);
                if (!(ok = bar_wait(mma2, gb & 1, abort_w)))
                    break;
                fence_after();
                const uint32_t ob = tmem + lrow + TM_O + (gb & 1) * 64;
                const bool tma = sizeof(Tout) == 4 && len == C;
                for (int half = 0; half < 2; ++half) {
                    uint32_t r[32];
                    tmem_ld32(ob + half * 32, r);
                    tmem_wait_ld(r);
                    if (tma) {
                        if (leader)
                            bulk_wait_read();
                        sync_output();
#pragma unroll
                        for (int uu = 0; uu < 32; ++uu) {
                            const float x = a.scale * __uint_as_float(r[uu]);
                            omax = amax_nan(omax, x);
                            ost[uu * 128 + b] = x;
                        }
                        fence_proxy_async();
                        sync_output();
                        if (leader) {
                            if (HF)
                                tma_store_3d(&tm_o, ost, v0, row0 - n * a.T + half * 32, n * H + h);
                            else
                                tma_store_3d(&tm_o, ost, v0, h, row0 + half * 32);
                            bulk_commit();
                        }
                    } else {
                        Tout *orow = go + row_head(row0, h, H, a.T, HF ? 1 : 0) * V + v0 + b;
#pragma unroll
                        for (int uu = 0; uu < 32; ++uu) {
                            const int t = half * 32 + uu;
                            const float x = a.scale * __uint_as_float(r[uu]);
                            if (t < len) {
                                omax = amax_nan(omax, x);
                                orow[(size_t)t * rstride] = to_out<Tout>(x);
                            }
                        }
                    }
                }
                fence_before();
                bar_arrive(&o_free[gb & 1]);
            }
            if (!ok)
                report(a.status, GLA_ERR_TIMEOUT);
        }
        qbase += nQ;
        nbbase += nchunks;
        nabase += nA;
        naitems += nA > 0 ? 1 : 0;
        items += 1;
    }

    // drain, then let the last CTA out reset the work counters for the next call
    if (warp == WCTL && lane == 0 && items > 0)
        bar_wait(tmem_free, (items - 1) & 1, abort_w);   // the last item's MMAs and final-state read are done
    if (tid == NA + NB) {
        bulk_wait_all();
        if (!finite(omax))
            report(a.status, GLA_ERR_RANGE);
    }
    if (tid >= NA + NB && tid < NA + NB + NC && !finite(omax))
        report(a.status, GLA_ERR_RANGE);
    fence_before();
    __syncthreads();
    if (tid == CTL) {
        __threadfence();
        if (atomicAdd(a.ctr + 1, 1) == (int)gridDim.x - 1) {
            a.ctr[0] = 0;   // the last CTA out leaves the counters zeroed for the next call
            a.ctr[1] = 0;
            a.ctr[2] = static_cast<int>((tag + 1) & kEpochMask);
            __threadfence();
        }
    }
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

// 3-D map of a [rows, H, D] tensor (time-major), or of a [B, H, T, D] one as {D, T, B*H} (head-first, T > 0);
// boxes of `inner` x `brows` rows of one head.
bool encode_rows(CUtensorMap *m, const void *ptr, int D, int H, long long rows, int inner, int brows, bool swizzle,
                 CUtensorMapDataType type, bool hf, int T)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t es = type == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? 4 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)H * D * es};
    cuuint32_t box[3] = {(cuuint32_t)inner, 1, (cuuint32_t)brows};
    if (hf && T > 0) {
        dims[1] = (cuuint64_t)T;
        dims[2] = (cuuint64_t)(rows / T) * H;
        strides[0] = (cuuint64_t)D * es;
        strides[1] = (cuuint64_t)T * D * es;
        box[1] = (cuuint32_t)brows;
        box[2] = 1;
    }
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, type, 3, const_cast<void *>(ptr),
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Tin, typename Tout, bool HF>
cudaError_t launch_fused_t(const Plan &pl, const Args &a, cudaStream_t s, int sms)
{
    const long long rows = pl.varlen ? (long long)pl.T : (long long)pl.B * pl.T;
    const CUtensorMapDataType tin =
        std::is_same<Tin, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap mq, mk, mg, mv, mo;
    const bool hf = HF;
    if (!encode_rows(&mq, a.q, pl.K, pl.H, rows, 64, C, true, tin, hf, pl.T) ||
        !encode_rows(&mk, a.k, pl.K, pl.H, rows, 64, C, true, tin, hf, pl.T) ||
        !encode_rows(&mg, a.g, pl.K, pl.H, rows, 128, C, false, tin, hf, pl.T) ||
        !encode_rows(&mv, a.v, pl.V, pl.H, rows, 128, C, false, tin, hf, pl.T))
        return cudaErrorInvalidValue;
    const bool f32o = sizeof(Tout) == 4;
    if (!encode_rows(&mo, f32o ? a.o : a.v, pl.V, pl.H, rows, 128, 32, false,
                     f32o ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, hf, pl.T))
        return cudaErrorInvalidValue;
    auto f = gla_fused<Tin, Tout, HF>;
    // the shared-memory opt-in is per device: remember it per device ordinal (set every time beyond 64)
    static std::atomic<unsigned long long> attr_set{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (!bit || !(attr_set.load(std::memory_order_acquire) & bit)) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        attr_set.fetch_or(bit, std::memory_order_release);
    }
    int nitems = pl.J * pl.H * (pl.V / VT);
    // scan block length: when every item runs at once the chain of end-state publications is the critical
    // path, so only every 8th segment publishes one; with several waves the predecessors finished earlier
    // and the plain chain (one tile read per item) costs least
    Args ka = a;
    ka.lb = nitems <= sms ? 8 : 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min(nitems, sms));
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = pl.varlen ? 1 : 0;
    void *args[] = {&mq, &mk, &mg, &mv, &mo, &ka, &nitems};
    cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(f), args);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(int dtype, int K, int V)
{
    // 16-bit q, k, v and g (an fp32 g tile does not fit the stage ring: those shapes run on CUDA cores)
    return (dtype == GLA_BF16 || dtype == GLA_BF16_OBF16 || dtype == GLA_F16) && K == KD && V % VT == 0 &&
           V <= 256;
}

cudaError_t launch_fused_tc(const Plan &pl, const Args &a, cudaStream_t s, int sms)
{
    // the layout is a template parameter, so the time-major kernel carries no layout branches
    if (pl.dtype == GLA_BF16_OBF16)
        return a.hf ? launch_fused_t<__nv_bfloat16, __nv_bfloat16, true>(pl, a, s, sms)
                    : launch_fused_t<__nv_bfloat16, __nv_bfloat16, false>(pl, a, s, sms);
    if (pl.dtype == GLA_F16)
        return a.hf ? launch_fused_t<__half, float, true>(pl, a, s, sms)
                    : launch_fused_t<__half, float, false>(pl, a, s, sms);
    return a.hf ? launch_fused_t<__nv_bfloat16, float, true>(pl, a, s, sms)
                : launch_fused_t<__nv_bfloat16, float, false>(pl, a, s, sms);
}

}  // namespace gla
