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
//      fixed two-level scan (blocks of lb segments; publication flags in the workspace carry the launch
//      epoch, so nothing is cleared between calls; segment 0 reads h0) and publishes its own contribution
//      or end state, and
//   3. runs the output pass over the same chunks, first to last, while they are still in L2.
// The last segment of a sequence skips 1. and 2.'s publication and writes ht at the end.  One segment per
// sequence is the plain single pass.
//
// Items are pipelined inside a CTA: the TMA producer claims the next item as soon as it has issued the
// loads of the current one and passes it to the other roles through a small queue in shared memory, so the
// next item's loads, gating and state pass overlap the current item's last output chunks, and the gating of
// an item's first output chunks overlaps its start-state scan.  The state accumulator is double-buffered
// in TMEM by item parity.
//
// MMAs (M = 128; the state lives in TMEM transposed, lane = value column v, column = key dimension):
//   (c) S^T += V^T   k^^T     A = V  [t][v]   (MN-major, smem), B = k^ [t][key] (MN-major, smem)
//       (output pass: B = k~ [t][key], the per-key factor 2^(G_last - G_a) is applied to the state instead)
//   (a) O^T  = S'^T  q~^T      A = S' from TMEM (fp16),          B = q~ [t][key] (K-major, smem)
//   (b) P    = q~    k~^T      A = q~ (rows 64..127 unused),     B = k~ [s][key] (K-major, smem)
//   (d) O^T += V^T   P^T      A = V  [s][v]   (MN-major, smem), B = P  [t][s]   (K-major, smem)
// q~ = q*exp(G-G_a), k~ = k*exp(G_a-G), k^ = k*exp(G_last-G), S' = diag(exp(G_a)) S, anchor a = row 31.
// Every smem operand is in the row layout its TMA box lands in (128-byte swizzle), so nothing is
// transposed on chip: V is converted to fp16 in place and k^ is written over the consumed gate rows.
// Operands are fp16 (bf16 inputs widen exactly; 11-bit significands keep the result within the parity bounds
// where single-rounded bf16 operands do not); accumulation is fp32 in TMEM; gates are summed in log2 units.
//
// Roles: warps 0-7 gating (cumsum, gating, operand conversion in place in the TMA stage); warps 8-11 state
// (S' and decay per chunk, final state); warps 12-15 output (P, O^T -> coalesced global stores); warps 8-15
// together run the start-state scan of an item; warp 16 lane 0 issues the MMAs, warp 17 lane 0 claims items
// and issues the TMA loads (three 64 KB stages, freed by MMA commits).  Every wait is bounded and a CTA-wide
// abort word ends all roles quickly after the first failure (GLA_ERR_TIMEOUT); a role whose threads must act
// together agrees on every wait's outcome by a barrier vote first; non-finite outputs report GLA_ERR_RANGE.
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
constexpr int NC = 128;          // output group (epilogue)
constexpr int NP = 64;           // P group: warps 16 and 17 reach TMEM lanes 0..63, the rows of P
constexpr int WB = NA / 32, WC = (NA + NB) / 32, WP = (NA + NB + NC) / 32, WCTL = WP + 2, WPRD = WCTL + 1;
constexpr int CTL = NA + NB + NC + NP;   // MMA issue thread
constexpr int NTHREADS = NA + NB + NC + NP + 64;
constexpr float L2E = 1.4426950408889634f;
constexpr uint32_t kEpochMask = 0x3FFFFFFFu;   // a flag holds (epoch << 2) | kind
constexpr int IQ = 4;                          // item queue depth
constexpr uint32_t kHalf = 8192;               // one 64-column half of a 64-row 16-bit tile

// Stage: q and k as two 64-key halves each (128-byte swizzle, K-major for (a) and (b)), the raw gate rows
// (unswizzled, 16 or 32 KB by the gate's element size; overwritten by k^ in two swizzled 64-key halves), V as
// two swizzled 64-column halves.  64 KB stages with a 16-bit gate (three in the ring), 80 KB with an fp32 gate
// (two).
constexpr int ST_Q0 = 0, ST_K0 = 8192, ST_G = 32768;
constexpr int NBARS = 42;
template <int GB>   // bytes per gate element
struct Ring {
    static constexpr int NSTAGE = GB == 2 ? 3 : 2;
    static constexpr int ST_V = ST_G + C * KD * GB;
    static constexpr int STAGE = ST_V + 16384;
    static constexpr int OFF_P = NSTAGE * STAGE;          // P [t][s] fp16, 8 KB
    static constexpr int OFF_EG = OFF_P + 8192;           // per output chunk (index mod 4): e[128], cl[128]
    static constexpr int OFF_PS = OFF_EG + 4 * 1024;      // gating partial sums [2][4][128]
    static constexpr int OFF_GT = OFF_PS + 4096;          // segment decay (log2) per key, [4][128] by state-pass item
    static constexpr int OFF_WL = OFF_GT + 2048;          // look-back: running log2 weight per key, [128], its
                                                          // power of two [128], the segment decay factor [128]
    static constexpr int OFF_CL = OFF_WL + 1536;          // state group: exp(G_last - G_a) of an item's last chunk
    static constexpr int OFF_MISC = OFF_CL + 1024;        // [0..3] item queue, [4] abort word, [5] look-back flag
    static constexpr int OFF_BAR = OFF_MISC + 64;
    static constexpr int SMEM_BYTES = OFF_BAR + NBARS * 8 + 16 + 1024;
};
static_assert(Ring<2>::SMEM_BYTES <= 232448 && Ring<4>::SMEM_BYTES <= 232448, "shared memory per CTA");

// TMEM columns: two state buffers (by item parity), two S' buffers (fp16, 64 columns each, by output chunk
// parity; together also the start-state scan's accumulator), O^T, P.
constexpr uint32_t TM_S = 0, TM_SOP = 256, TM_O = 384, TM_P = 448, TM_COLS = 512;
constexpr uint32_t ID_C = idesc_f16_f32(128, 128) | kIdescAMajorMN | kIdescBMajorMN;
constexpr uint32_t kQK = 16384;                // between the two 64-key halves of q (and of k) in a stage
constexpr uint32_t ID_D = idesc_f16_f32(128, 64) | kIdescAMajorMN;
constexpr uint32_t ID_N64 = idesc_f16_f32(128, 64);

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
// One row's gate values of keys 2 kp and 2 kp + 1 as the stage holds them (a 32-bit pair of 16-bit values,
// or two floats), widened.
template <typename Tg>
struct GateW {
    using W = uint32_t;
    static __device__ __forceinline__ W load(const uint8_t *g, int t, int kp)
    {
        return *reinterpret_cast<const uint32_t *>(g + t * 256 + kp * 4);
    }
    static __device__ __forceinline__ W zero() { return 0u; }
    static __device__ __forceinline__ float lo(W w) { return In<Tg>::lo(w); }
    static __device__ __forceinline__ float hi(W w) { return In<Tg>::hi(w); }
};
template <>
struct GateW<float> {
    using W = float2;
    static __device__ __forceinline__ W load(const uint8_t *g, int t, int kp)
    {
        return *reinterpret_cast<const float2 *>(g + t * 512 + kp * 8);
    }
    static __device__ __forceinline__ W zero() { return make_float2(0.f, 0.f); }
    static __device__ __forceinline__ float lo(W w) { return w.x; }
    static __device__ __forceinline__ float hi(W w) { return w.y; }
};
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

// Named barriers: 1 gating group, 2 output group, 3 state group, 4 the chain team (state and output groups
// together), 5 P group.
// The *_all forms are barriers that also return whether every participating thread passed `v`, so that a
// group whose threads must act together (named barriers, warp-collective TMEM access) agrees on the outcome
// of a bounded wait before acting on it.
template <int ID, int N>
__device__ __forceinline__ bool group_all(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v), "n"(ID), "n"(N)
                 : "memory");
    return r != 0;
}
__device__ __forceinline__ void sync_team() { asm volatile("bar.sync 4, %0;" ::"n"(NB + NC) : "memory"); }
__device__ __forceinline__ bool gating_all(bool v) { return group_all<1, NA>(v); }
__device__ __forceinline__ bool output_all(bool v) { return group_all<2, NC>(v); }
__device__ __forceinline__ bool team_all(bool v) { return group_all<4, NB + NC>(v); }
__device__ __forceinline__ bool p_all(bool v) { return group_all<5, NP>(v); }
__device__ __forceinline__ void sync_state() { asm volatile("bar.sync 3, %0;" ::"n"(NB) : "memory"); }
__device__ __forceinline__ float4 f4(const uint32_t *r)
{
    return make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]), __uint_as_float(r[2]), __uint_as_float(r[3]));
}

// V tile of one stage (two swizzled 64-column halves of 64 rows) into fp16 operand form in place; rows at or
// past `len` (outside the segment) become zero.  Each gating thread takes four 16-byte pieces.
template <typename Tin>
__device__ __forceinline__ void v_operand(uint8_t *vt, int len, int tid)
{
    if (std::is_same<Tin, __half>::value && len == C)
        return;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int off = (tid + NA * i) * 16;
        uint4 *p = reinterpret_cast<uint4 *>(vt + off);
        const int row = (off >> 7) & 63;
        if (row >= len) {
            *p = make_uint4(0u, 0u, 0u, 0u);
        } else if (!std::is_same<Tin, __half>::value) {
            uint4 x = *p;
            x.x = In<Tin>::op(x.x);
            x.y = In<Tin>::op(x.y);
            x.z = In<Tin>::op(x.z);
            x.w = In<Tin>::op(x.w);
            *p = x;
        }
    }
}

// Everything a work item is: slot j, head h, value tile vt; sequence n, segment p, rows [bos, eos).
// itn: index among this CTA's items (state buffer itn & 1); na: index among its items with a state pass.
struct Item {
    int j, h, vt, v0, n, p, bos, eos, nchunks, nA, itn, na;
    bool last;
};

// Balanced pieces (dense batches): the chunks of the B*H (sequence, head) units, unit after unit, cut into np
// pieces at chunk c * tot / np (rounded down), tot = B*H*nc.  A unit's segment p is its part of the p-th
// piece that overlaps it; a piece is shorter than a unit, so it overlaps at most two.
__device__ __forceinline__ long long piece_bnd(const Args &a, long long c, long long tot)
{
    return c * tot / a.np;
}
// the piece holding global chunk x
__device__ __forceinline__ long long piece_of(const Args &a, long long x, long long tot)
{
    return ((x + 1) * a.np + tot - 1) / tot - 1;
}

// Slot j of head h: sequence n, segment p, rows [bos, eos) and the sequence end; false for an unused slot.
__device__ __forceinline__ bool resolve_item(const Args &a, int j, int h, int &n, int &p, int &bos, int &eos,
                                             int &send)
{
    if (!a.np)
        return resolve_slot(a, j, n, p, bos, eos, send);
    n = j / a.P;
    p = j - n * a.P;
    const long long tot = (long long)a.B * a.H * a.nc;
    const long long u0 = ((long long)n * a.H + h) * a.nc, u1 = u0 + a.nc;
    const long long c0 = piece_of(a, u0, tot);
    const long long s0 = max(u0, piece_bnd(a, c0 + p, tot)), s1 = min(u1, piece_bnd(a, c0 + p + 1, tot));
    if (s0 >= s1)
        return false;
    const int sb = n * a.T;
    send = sb + a.T;
    bos = sb + (int)(s0 - u0) * C;
    eos = min(sb + (int)(s1 - u0) * C, send);
    return true;
}

// What the start-state scan needs from the kernel (shared-memory words, barriers, the launch epoch).
struct ChainCtx {
    const float *h0;
    float *ss, *agg, *gtot;
    int *flags;
    int lb;
    uint32_t tmem, tag;
    float *wl;
    const float *gts4;        // [4][128] segment decays by state-pass item index mod 4
    volatile int *misc;       // [4] abort word, [5] look-back flag broadcast
    uint64_t *g_done, *a_done;
    int H, NV, V;
};

// Start-state scan: the start state of item `it`'s segment into TMEM state buffer `sb`.  Segments are grouped in blocks of lb;
// the first segment of a block (a boundary, p % lb == 0) publishes its end state S_out = 2^Gtot S_in + dS
// (flag 2), every other segment with a state pass publishes its contribution dS and decay Gtot (flag 1)
// as soon as the pass is done.  With p0 the last boundary before p,
//   S_in(p) = sum_{i = p-1 .. p0+1} 2^(Gtot(p-1) + ... + Gtot(i+1)) dS(i) + 2^(Gtot(p-1) + ... + Gtot(p0+1)) S_out(p0),
// summed newest first, and S_in(0) = h0.  The grouping is fixed, so the result does not depend on
// timing; lb = 1 is the plain serial chain (one tile read and one written per segment), a larger lb
// shortens the chain of dependent publications when all items run at once.
// 256 threads, lane = value column; the state group takes keys 0..63, the output group 64..127.  The two
// S' buffers (idle between an item's output pass and the next's) accumulate the sum.  Published tiles are
// key-interleaved (float4 of 4 keys per value column) so a warp reads 512 contiguous bytes per load.
// Out of line, so that its registers do not weigh on the per-chunk loops of the two groups.
__device__ __noinline__ bool chain_scan(const ChainCtx &a, const Item &it, int u, uint32_t sb, int na)
{
    const ChainCtx &cx = a;
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t tmem = cx.tmem, tag = cx.tag;
    const int H = cx.H, NV = cx.NV, V = cx.V;
    float *wl = cx.wl, *ew = cx.wl + 128, *eg = cx.wl + 256;
    volatile int *misc = cx.misc;
    volatile int *abort_w = misc + 4;
    uint64_t *g_done = cx.g_done, *a_done = cx.a_done;
    const int half = warp >= WC ? 1 : 0;
    const int b = tid - NA - half * NB;
    const int kb0 = 64 * half;
    const uint32_t lrow = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool leader = tid == NA;
    const size_t tile = (size_t)KD * VT;
    const size_t mine = ((size_t)it.j * H + it.h) * NV + it.vt;
    const int HN = H * NV;
    const int p = it.p;
    const bool boundary = p % a.lb == 0;
    const size_t soff = ((size_t)it.n * H + it.h) * KD * V + it.v0 + b;
    const float *gts = cx.gts4 + (na & 3) * 128;
    // the first segment of a sequence with a state pass stages h0 in the (idle) S' columns while the
    // pass runs, so that its end state is published without a read from memory on the critical path
    const bool h0pre = p == 0 && it.nA > 0 && a.h0 != nullptr;
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
    if (it.nA > 0)
        ok = bar_wait(&g_done[na & 3], (na >> 2) & 1, abort_w) && bar_wait(&a_done[na & 3], (na >> 2) & 1, abort_w);
    if (!team_all(ok))
        return false;
    fence_after();
    if (it.nA > 0 && !boundary) {
        float4 *dst = reinterpret_cast<float4 *>(a.agg + mine * tile);
        for (int sub = 0; sub < 4; ++sub) {
            const int k0 = kb0 + 16 * sub;
            uint32_t r[16];
            tmem_ld16(tmem + lrow + sb + k0, r);
            tmem_wait_ld(r);
#pragma unroll
            for (int w = 0; w < 4; ++w)
                __stcg(dst + (size_t)(k0 / 4 + w) * VT + b, f4(r + 4 * w));
        }
        if (b < 64)
            __stcg(a.gtot + mine * KD + kb0 + b, gts[kb0 + b]);
        sync_team();   // every thread's stores precede the leader's fence and flag
        if (leader) {
            __threadfence();
            flag_set(a.flags + u, static_cast<int>(tag << 2 | 1u));
        }
    }
    const int p0 = p > 0 ? (p - 1) / a.lb * a.lb : 0;
    if (p > 0) {
        // the predecessors publish at about the same time: wait for all of them first, newest first, then
        // read each tile with a thread's 64 keys in flight at once
        if (leader) {
            int okf = 1;
            for (int i = p - 1; i > p0 && okf; --i)
                okf = flag_wait_tag(a.flags + (u - (p - i) * HN), tag, 1, abort_w);
            misc[5] = okf ? flag_wait_tag(a.flags + (u - (p - p0) * HN), tag, 2, abort_w) : 0;
        }
        if (b < 64) {
            wl[kb0 + b] = 0.f;
            ew[kb0 + b] = 1.f;
        }
        sync_team();
        if (misc[5] == 0)
            return false;   // uniform: every thread read the same value
        for (int i = p - 1; i > p0; --i) {
            const int back = p - i;
            const size_t ti = mine - (size_t)back * HN;
            const float4 *src = reinterpret_cast<const float4 *>(a.agg + ti * tile);
            const float gi = b < 64 ? __ldcg(a.gtot + ti * KD + kb0 + b) : 0.f;
            sync_team();   // the weights of this step are in place
            for (int sub = 0; sub < 2; ++sub) {
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
                        const float4 e = *reinterpret_cast<const float4 *>(ew + k1 + 4 * w);
                        const float4 xv = x[4 * hh + w];
                        r[4 * w] = __float_as_uint(fmaf(e.x, xv.x, __uint_as_float(r[4 * w])));
                        r[4 * w + 1] = __float_as_uint(fmaf(e.y, xv.y, __uint_as_float(r[4 * w + 1])));
                        r[4 * w + 2] = __float_as_uint(fmaf(e.z, xv.z, __uint_as_float(r[4 * w + 2])));
                        r[4 * w + 3] = __float_as_uint(fmaf(e.w, xv.w, __uint_as_float(r[4 * w + 3])));
                    }
                    tmem_st16(tmem + lrow + TM_SOP + k1, r);
                }
            }
            tmem_wait_st();
            sync_team();   // every thread has used this step's weights
            if (b < 64) {
                const float w1 = wl[kb0 + b] + gi;
                wl[kb0 + b] = w1;
                ew[kb0 + b] = ex2(w1);
            }
        }
    }
    // S_in -> TMEM state buffer; a boundary segment with a state pass publishes S_out = 2^Gtot * S_in + dS
    const bool acc = p - 1 > p0;   // contributions were summed into the S' columns
    const bool pub = it.nA > 0 && boundary;
    const float4 *bsrc = reinterpret_cast<const float4 *>(a.ss + (mine - (size_t)(p - p0) * HN) * tile);
    float4 *bdst = reinterpret_cast<float4 *>(a.ss + mine * tile);
    float4 xb[16];
    if (p > 0) {
        // the boundary's end state, 64 keys in flight
#pragma unroll
        for (int w = 0; w < 16; ++w)
            xb[w] = __ldcg(bsrc + (size_t)(kb0 / 4 + w) * VT + b);
    }
    if (pub && b < 64)
        eg[kb0 + b] = ex2(gts[kb0 + b]);
    if (p > 0 || pub)
        sync_team();   // the last step's weights (and the segment's decay factors) are in place
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
        const int k1 = kb0 + 16 * hh;
        uint32_t sn[16];
        if (p > 0) {
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
                const float4 e = *reinterpret_cast<const float4 *>(ew + k1 + 4 * w);
                const float4 xv = xb[4 * hh + w];
                sn[4 * w] = __float_as_uint(fmaf(e.x, xv.x, __uint_as_float(sn[4 * w])));
                sn[4 * w + 1] = __float_as_uint(fmaf(e.y, xv.y, __uint_as_float(sn[4 * w + 1])));
                sn[4 * w + 2] = __float_as_uint(fmaf(e.z, xv.z, __uint_as_float(sn[4 * w + 2])));
                sn[4 * w + 3] = __float_as_uint(fmaf(e.w, xv.w, __uint_as_float(sn[4 * w + 3])));
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
            tmem_ld16(tmem + lrow + sb + k1, r);
            tmem_wait_ld(r);
#pragma unroll
            for (int uu = 0; uu < 16; ++uu)
                r[uu] = __float_as_uint(fmaf(eg[k1 + uu], __uint_as_float(sn[uu]), __uint_as_float(r[uu])));
#pragma unroll
            for (int w = 0; w < 4; ++w)
                __stcg(bdst + (size_t)(k1 / 4 + w) * VT + b, f4(r + 4 * w));
        }
        tmem_st16(tmem + lrow + sb + k1, sn);
    }
    tmem_wait_st();
    fence_before();
    sync_team();
    fence_after();
    if (pub && leader) {
        __threadfence();
        flag_set(a.flags + u, static_cast<int>(tag << 2 | 2u));
    }
    return true;
}

template <typename Tin, typename Tg, typename Tout, bool HF>
__global__ void __launch_bounds__(NTHREADS, 1)
    gla_fused(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_v, Args a,
              int nitems)
{
    using RG = Ring<sizeof(Tg)>;
    constexpr int NSTAGE = RG::NSTAGE, STAGE = RG::STAGE, ST_V = RG::ST_V, OFF_P = RG::OFF_P, OFF_EG = RG::OFF_EG,
                  OFF_PS = RG::OFF_PS, OFF_GT = RG::OFF_GT, OFF_WL = RG::OFF_WL, OFF_CL = RG::OFF_CL,
                  OFF_MISC = RG::OFF_MISC, OFF_BAR = RG::OFF_BAR;
    using GW = GateW<Tg>;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *full = bars + 0, *prep = bars + 3, *empty = bars + 6;        // [3] each: the stage ring
    uint64_t *ops_ready = bars + 9, *p_ready = bars + 10, *mma1 = bars + 11, *mma_st = bars + 12;
    uint64_t *mma2 = bars + 13, *o_free = bars + 14;
    uint64_t *a_done = bars + 15, *g_done = bars + 19;                     // [4] by state-pass item index
    uint64_t *item_done = bars + 23, *tmem_free = bars + 25;               // [2] by item parity
    uint64_t *item_full = bars + 27, *item_empty = bars + 31;              // [IQ]
    uint64_t *drain = bars + 35;
    uint64_t *eg_ready = bars + 36;                                        // [4]: by output chunk index
    uint64_t *sop_free = bars + 40;                                        // [2]: MMA (a) of a chunk done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBARS);
    volatile int *misc = reinterpret_cast<volatile int *>(sm + OFF_MISC);   // [0..3] queue, [4] abort, [5] flag
    volatile int *iq = misc;
    volatile int *abort_w = misc + 4;
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
            bar_init(&empty[s], 1);
        }
        bar_init(ops_ready, NB);
        bar_init(p_ready, NP);
        bar_init(mma1, 1);
        bar_init(mma_st, 1);
        bar_init(mma2, 1);
        bar_init(o_free, NC);
        for (int i = 0; i < 4; ++i) {
            bar_init(&a_done[i], 1);
            bar_init(&g_done[i], NA);
        }
        for (int i = 0; i < 2; ++i) {
            bar_init(&item_done[i], 1);
            bar_init(&tmem_free[i], NB);
        }
        for (int i = 0; i < IQ; ++i) {
            bar_init(&item_full[i], 1);
            bar_init(&item_empty[i], NA + NB + NC + NP + 1);
        }
        bar_init(drain, 1);
        for (int i = 0; i < 4; ++i)
            bar_init(&eg_ready[i], 64);
        for (int i = 0; i < 2; ++i)
            bar_init(&sop_free[i], 1);
        bar_fence_init();
        misc[4] = 0;
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_g);
        tma_prefetch_desc(&tm_v);
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;

    // Item k of this CTA from the queue (every consumer thread arrives on the slot's empty barrier once it
    // has read it); false after an abort.  u < 0 ends the loop.
    auto take_item = [&](int k, int &u) -> bool {
        if (!bar_wait(&item_full[k % IQ], (k / IQ) & 1, abort_w))
            return false;
        u = iq[k % IQ];
        bar_arrive(&item_empty[k % IQ]);
        return true;
    };
    ChainCtx cx;
    cx.h0 = a.h0;
    cx.ss = a.ss;
    cx.agg = a.agg;
    cx.gtot = a.gtot;
    cx.flags = a.flags;
    cx.lb = a.lb;
    cx.tmem = tmem;
    cx.tag = tag;
    cx.wl = wl;
    cx.gts4 = reinterpret_cast<const float *>(sm + OFF_GT);
    cx.misc = misc;
    cx.g_done = g_done;
    cx.a_done = a_done;
    cx.H = H;
    cx.NV = NV;
    cx.V = V;
    // Item u; itn and na are the role's running counts (every role counts the same items), advanced here.
    auto decode = [&](int u, Item &it, int &itn, int &na) -> bool {
        it.j = u / (H * NV);
        const int rem = u - it.j * (H * NV);
        it.h = rem / NV;
        it.vt = rem - it.h * NV;
        it.v0 = it.vt * VT;
        int send;
        if (!resolve_item(a, it.j, it.h, it.n, it.p, it.bos, it.eos, send))
            return false;   // unused varlen slot (every role sees the same)
        it.nchunks = (it.eos - it.bos + C - 1) / C;
        it.last = it.eos == send;
        it.nA = it.last ? 0 : it.nchunks;   // state-pass chunks (reverse order)
        it.itn = itn++;
        it.na = na;
        na += it.nA > 0 ? 1 : 0;
        return true;
    };

    float omax = 0.f;   // output group: running max |o| (range check)

    // Ring order: the state-pass chunks of an item (last to first), then its output-pass chunks (first to
    // last), item after item.  Every role walks its items the same way: `run_s`, then `run_o`.
#define GLA_ITEM_LOOP(VOTE, RUN_S, RUN_O)                                                                    \
    {                                                                                                        \
        int itn = 0, nac = 0;                                                                                \
        bool ok = true;                                                                                      \
        for (int k = 0; ok; ++k) {                                                                           \
            int u = -1;                                                                                      \
            ok = VOTE(take_item(k, u));                                                                      \
            if (!ok || u < 0)                                                                                \
                break;                                                                                       \
            Item cur;                                                                                        \
            if (!decode(u, cur, itn, nac))                                                                   \
                continue;                                                                                    \
            ok = RUN_S(cur) && RUN_O(cur);                                                                   \
        }                                                                                                    \
        if (!ok)                                                                                             \
            fail();                                                                                          \
    }

    if (warp == WPRD) {
        // ------------------------------------------------------------------ item claims + TMA producer
        if (lane == 0) {
            int qbase = 0, issued = 0;   // ring position; chunks whose loads were issued
            auto fail = [&]() {
                *abort_w = 1;
                report(a.status, GLA_ERR_TIMEOUT);
            };
            // the state-pass chunks (last to first) or the output-pass chunks (first to last) of an item
            auto load = [&](const Item &it, bool out) -> bool {
                const int n = out ? it.nchunks : it.nA;
                for (int q = 0; q < n; ++q) {
                    const int gq = qbase + q, s = gq % NSTAGE;
                    // the stage is free once the MMAs of the chunk three places earlier are complete
                    if (gq >= NSTAGE && !bar_wait(&empty[s], (gq / NSTAGE - 1) & 1, abort_w))
                        return false;
                    uint8_t *st = sm + s * STAGE;
                    const int row0 = it.bos + (out ? q : it.nA - 1 - q) * C;
                    // tensor-map coordinates of the chunk: (head, row) time-major, (row in sequence,
                    // sequence * H + head) head-first
                    // (a varlen pack is one batch row: its rows are global rows of that batch)
                    const int nb = a.table ? 0 : it.n;
                    const int c1 = HF ? row0 - nb * a.T : it.h, c2 = HF ? nb * H + it.h : row0;
                    bar_expect_tx(&full[s], (out ? 4 : 3) * 16384 + (int)(sizeof(Tg) - 2) * 8192);
                    if (out) {
                        tma_load_3d(st + ST_Q0, &tm_q, 0, c1, c2, &full[s]);
                        tma_load_3d(st + 16384 + ST_Q0, &tm_q, 64, c1, c2, &full[s]);
                    }
                    tma_load_3d(st + ST_K0, &tm_k, 0, c1, c2, &full[s]);
                    tma_load_3d(st + 16384 + ST_K0, &tm_k, 64, c1, c2, &full[s]);
                    tma_load_3d(st + ST_G, &tm_g, 0, c1, c2, &full[s]);
                    tma_load_3d(st + ST_V, &tm_v, it.v0, c1, c2, &full[s]);
                    tma_load_3d(st + ST_V + kHalf, &tm_v, it.v0 + 64, c1, c2, &full[s]);
                    issued = gq + 1;
                }
                qbase += n;
                return true;
            };
            // claim w: work item w, or with balanced pieces the one or two segments of piece w / NV (a
            // piece crossing into the next unit runs that unit's first segment first: its end state is
            // published early, and the previous unit's last segment then finds its start state ready)
            const long long tot = (long long)a.B * H * a.nc;
            auto claim = [&](int w, int (&us)[2]) -> int {
                if (w < 0 || w >= nitems)
                    return 0;
                if (!a.np) {
                    us[0] = w;
                    return 1;
                }
                const int c = w / NV, vt = w - c * NV;
                const long long ua = piece_bnd(a, c, tot) / a.nc, ub = (piece_bnd(a, c + 1, tot) - 1) / a.nc;
                auto id = [&](long long unit, long long p) {
                    const int n = (int)(unit / H), h = (int)(unit - (long long)n * H);
                    return ((n * a.P + (int)p) * H + h) * NV + vt;
                };
                int m = 0;
                if (ub != ua)
                    us[m++] = id(ub, 0);
                us[m++] = id(ua, c - piece_of(a, ua * a.nc, tot));
                return m;
            };
            int itn = 0, nac = 0, k = 0;
            bool ok = true;
            for (bool more = true; more && ok;) {
                int us[2];
                const int m = claim(*abort_w ? -1 : atomicAdd(a.ctr + 0, 1), us);
                more = m > 0;
                for (int i = 0; i < (more ? m : 1) && ok; ++i, ++k) {
                    if (k >= IQ && !(ok = bar_wait(&item_empty[k % IQ], ((k / IQ) - 1) & 1, abort_w)))
                        break;
                    const int u = more ? us[i] : -1;
                    iq[k % IQ] = u;
                    bar_arrive(&item_full[k % IQ]);
                    Item cur;
                    if (u >= 0 && decode(u, cur, itn, nac))
                        ok = load(cur, false) && load(cur, true);
                }
            }
            if (!ok)
                fail();
            // nothing may still be landing in shared memory when the CTA exits: wait for the last load of
            // every stage (they complete in any case; the limit only guards the wait itself)
            for (int s = 0; s < NSTAGE; ++s)
                if (issued > s)
                    bar_wait(&full[s], ((issued - 1 - s) / NSTAGE) & 1);
        }
    } else if (warp == WCTL) {
        // ------------------------------------------------------------------ MMA issue
        if (lane == 0) {
            int qbase = 0, nb = 0;
            const uint32_t pt = smem_u32(sm + OFF_P);
            auto fail = [&]() {
                *abort_w = 1;
                report(a.status, GLA_ERR_TIMEOUT);
            };
            // O^T += V^T P^T of the chunk in stage s (its P is in shared memory), then release the stage
            auto issue_d = [&](int s) {
                const uint32_t st = smem_u32(sm + s * STAGE);
                for (int kk = 0; kk < C / 16; ++kk)
                    mma_ss(tmem + TM_O, sdesc_mn_sw128(st + ST_V + kk * 2048, kHalf), sdesc_sw128(pt + kk * 32),
                           ID_D, 1u);
                mma_commit(mma2);
                mma_commit(&empty[s]);
            };
            // state pass: dS accumulated from zero into the item's state buffer
            auto run_s = [&](const Item &it) -> bool {
                if (it.nA == 0)
                    return true;
                const int buf = it.itn & 1;
                const uint32_t sb = tmem + TM_S + buf * 128;
                // the buffer was last used by item itn - 2, whose final state the state group has read
                if (it.itn >= 2 && !bar_wait(&tmem_free[buf], ((it.itn - 2) >> 1) & 1, abort_w))
                    return false;
                for (int q = 0; q < it.nA; ++q) {
                    const int s = (qbase + q) % NSTAGE;
                    const uint32_t st = smem_u32(sm + s * STAGE);
                    if (!bar_wait(&prep[s], ((qbase + q) / NSTAGE) & 1, abort_w))
                        return false;
                    fence_after();
                    for (int kk = 0; kk < C / 16; ++kk)
                        mma_ss(sb, sdesc_mn_sw128(st + ST_V + kk * 2048, kHalf),
                               sdesc_mn_sw128(st + ST_G + kk * 2048, kHalf), ID_C, (q > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&empty[s]);
                }
                mma_commit(&a_done[it.na & 3]);
                qbase += it.nA;
                return true;
            };
            // Output chunk gb needs four MMAs: (c) S += V^T k~ (needs the gating group's operands and the
            // state group's S'), (b) the scores (operands only), (a) the inter-chunk product (S' after (c), and
            // O^T free again), and later (d) O^T += V^T P^T (the P group's P).  They are issued as their inputs
            // become ready, within the order the shared buffers impose: (d) of the previous chunk before (b) of
            // this one (P in TMEM and in shared memory) and before (a) (both write O^T); (c) of a chunk before
            // its (a) and (d) (the stage is released after (d)).  Commits complete in issue order, so each also
            // covers every earlier MMA: mma_st (after (c)) tells the state group that U is ready, sop_free
            // (after (a)) that the chunk's S' buffer is free again, mma1 (after (b)) tells the P group that P
            // and the shared P tile are, mma2 (after (d)) tells the output group that O^T is.
            auto run_o = [&](const Item &it) -> bool {
                const uint32_t sb = tmem + TM_S + (it.itn & 1) * 128;
                // Item itn - 2 (same state buffer) is finished before this item's commits: without this wait,
                // items without chunks (empty sequences) would let this thread commit item_done twice for one
                // wait of the state group, which the parity of the barrier cannot tell apart.  The wait is met
                // at once in the steady state (that item's output pass completed two items ago).
                if (it.itn >= 2 && !bar_wait(&tmem_free[it.itn & 1], ((it.itn - 2) >> 1) & 1, abort_w))
                    return false;
                // Cursors: the state chain ((c) of chunk jc as soon as its operands and S' are ready) runs ahead
                // of the output chain ((b), (a), (d) of chunks jb, ja, jd), so the state recurrence does not wait
                // for the epilogue that frees O^T.  (c) of a chunk precedes its (a) and (d) (the stage is
                // released after (d)); (d) of a chunk precedes (b) and (a) of the next (P and O^T).
                const int nch = it.nchunks;
                int jb = 0, jc = 0, ja = 0, jd = 0;
                auto stage_of = [&](int j) { return (qbase + j) % NSTAGE; };
                auto ops_in = [&](int j) { return bar_test(&prep[stage_of(j)], ((qbase + j) / NSTAGE) & 1); };
                unsigned long long t0 = global_ns();
                while (jd < nch) {
                    bool progress = false;
                    if (jd < ja && bar_test(p_ready, (nb + jd) & 1)) {
                        fence_after();
                        issue_d(stage_of(jd));
                        ++jd;
                        progress = true;
                    }
                    if (jc < nch && ops_in(jc) && bar_test(ops_ready, (nb + jc) & 1)) {
                        fence_after();
                        const uint32_t st = smem_u32(sm + stage_of(jc) * STAGE);
                        for (int kk = 0; kk < C / 16; ++kk)
                            mma_ss(sb, sdesc_mn_sw128(st + ST_V + kk * 2048, kHalf),
                                   sdesc_mn_sw128(st + ST_K0 + kk * 2048, kQK), ID_C, 1u);
                        mma_commit(mma_st);
                        ++jc;
                        progress = true;
                    }
                    if (jb < nch && jb <= jd && ops_in(jb)) {
                        fence_after();
                        const uint32_t st = smem_u32(sm + stage_of(jb) * STAGE);
                        for (int kk = 0; kk < KD / 16; ++kk)
                            mma_ss(tmem + TM_P, sdesc_sw128(st + (kk >> 2) * 16384 + ST_Q0 + (kk & 3) * 32),
                                   sdesc_sw128(st + (kk >> 2) * 16384 + ST_K0 + (kk & 3) * 32), ID_N64, kk > 0);
                        mma_commit(mma1);
                        ++jb;
                        progress = true;
                    }
                    if (ja < jc && ja <= jd && (nb + ja == 0 || bar_test(o_free, (nb + ja - 1) & 1))) {
                        fence_after();
                        const int gb = nb + ja;
                        const uint32_t st = smem_u32(sm + stage_of(ja) * STAGE);
                        for (int kk = 0; kk < KD / 16; ++kk)
                            mma_ts(tmem + TM_O, tmem + TM_SOP + (gb & 1) * 64 + kk * 8,
                                   sdesc_sw128(st + (kk >> 2) * 16384 + ST_Q0 + (kk & 3) * 32), ID_N64, kk > 0);
                        mma_commit(&sop_free[gb & 1]);
                        ++ja;
                        progress = true;
                    }
                    if (progress) {
                        t0 = global_ns();
                    } else {
                        if (*abort_w)
                            return false;
                        if (global_ns() - t0 > kWaitNs) {
                            *abort_w = 1;
                            return false;
                        }
                        // idle: wait on the state chain's next hand-over (the recurrence that sets the chunk
                        // rate), waking when it completes or after a short while to look at the others
                        if (jc < nch)
                            bar_try_for(ops_ready, (nb + jc) & 1, 300);
                        else
                            bar_try_for(p_ready, (nb + jd) & 1, 300);
                    }
                }
                mma_commit(&item_done[it.itn & 1]);
                qbase += it.nchunks;
                nb += it.nchunks;
                return true;
            };
            auto one = [](bool v) { return v; };
            GLA_ITEM_LOOP(one, run_s, run_o)
            // every MMA issued is complete before TMEM is released
            mma_commit(drain);
            bar_wait(drain, 0);
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
        const float ls = log2f(a.scale);   // scale enters q~ as a power of two
        int qbase = 0, nb = 0;
        auto fail = [&]() {};
        auto gate = [&](const Item &it, bool out) -> bool {
            float *gts = reinterpret_cast<float *>(sm + OFF_GT) + (it.na & 3) * 128;
            float D0 = 0.f, D1 = 0.f;   // state pass: decay (log2) of the chunks already walked
            float P0 = 0.f, P1 = 0.f;   // output pass: G_last - G_a (log2) of the previous chunk
            const int n = out ? it.nchunks : it.nA;
            for (int q = 0; q < n; ++q) {
                const int gq = qbase + q;
                const int s = gq % NSTAGE;
                uint8_t *st = sm + s * STAGE;
                const int cq = out ? q : it.nA - 1 - q;
                const int len = min(C, it.eos - (it.bos + cq * C));
                const bool got = bar_wait(&full[s], (gq / NSTAGE) & 1, abort_w);
                typename GW::W gr[16];
                float *ps = psum + (gq & 1) * 512;
                if (got) {
                    v_operand<Tin>(st + ST_V, len, tid);
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll
                    for (int uu = 0; uu < 16; ++uu) {
                        const int t = 16 * rq + uu;
                        gr[uu] = t < len ? GW::load(st + ST_G, t, kp) : GW::zero();
                        s0 = fmaf(GW::lo(gr[uu]), L2E, s0);
                        s1 = fmaf(GW::hi(gr[uu]), L2E, s1);
                    }
                    ps[rq * 128 + key] = s0;
                    ps[rq * 128 + key + 1] = s1;
                }
                // the vote is also the barrier after which every gate row has been read (k^ goes over them)
                if (!gating_all(got))
                    return false;
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
                uint8_t *qk = st + kb * 16384;
                uint8_t *kh = st + ST_G + kb * kHalf;
                // the chunk's per-key factors go to the state group first, so that its step runs while this
                // group forms the operands: e = 2^(G_a + G_last' - G_a') (primes: the previous chunk; the
                // state buffer holds diag(2^G_a') S' + k~'^T V' after that chunk's MMA (c)) and
                // cl = 2^(G_last - G_a) (the final state of the item is diag(cl) times the buffer).  They are
                // kept by output-chunk index, not by stage: the state group waits for every output chunk in
                // turn, so each phase of these barriers is awaited in order (a stage's phases also count the
                // state-pass chunks, which the state group does not wait for)
                if (out && rq == 0) {
                    const int gb = nb + q;
                    float *eg = reinterpret_cast<float *>(sm + OFF_EG + (gb & 3) * 1024);
                    eg[key] = ex2(ga0 + P0);
                    eg[key + 1] = ex2(ga1 + P1);
                    eg[128 + key] = ex2(gl0 - ga0);
                    eg[128 + key + 1] = ex2(gl1 - ga1);
                    P0 = gl0 - ga0;
                    P1 = gl1 - ga1;
                    bar_arrive(&eg_ready[gb & 3]);
                }
                if (out) {
                    // output pass: q~ = scale q 2^(G - G_a) and k~ = k 2^(G_a - G) in place (k~ is also the
                    // state MMA's operand)
                    X0 -= ga0;
                    X1 -= ga1;
                    auto gate_rows = [&](auto full_tag) {
                        constexpr bool FULL = decltype(full_tag)::value;
#pragma unroll
                        for (int uu = 0; uu < 16; ++uu) {
                            const int t = 16 * rq + uu;
                            X0 = fmaf(GW::lo(gr[uu]), L2E, X0);
                            X1 = fmaf(GW::hi(gr[uu]), L2E, X1);
                            const uint32_t off = xo[uu & 7] + (uu >> 3) * 1024;
                            const uint32_t qw = *reinterpret_cast<const uint32_t *>(qk + ST_Q0 + off);
                            const uint32_t kw = *reinterpret_cast<const uint32_t *>(qk + ST_K0 + off);
                            float q0 = In<Tin>::lo(qw) * ex2(X0 + ls), q1 = In<Tin>::hi(qw) * ex2(X1 + ls);
                            float k0 = In<Tin>::lo(kw) * ex2(-X0), k1 = In<Tin>::hi(kw) * ex2(-X1);
                            if (!FULL && t >= len)
                                q0 = q1 = k0 = k1 = 0.f;
                            *reinterpret_cast<uint32_t *>(qk + ST_Q0 + off) = pack_h2(q0, q1);
                            *reinterpret_cast<uint32_t *>(qk + ST_K0 + off) = pack_h2(k0, k1);
                        }
                    };
                    if (len == C)
                        gate_rows(std::true_type{});
                    else
                        gate_rows(std::false_type{});
                } else {
                    // state pass: k^ = k * 2^(G_last - G + D)
                    const float e0 = gl0 + D0, e1 = gl1 + D1;
#pragma unroll
                    for (int uu = 0; uu < 16; ++uu) {
                        const int t = 16 * rq + uu;
                        X0 = fmaf(GW::lo(gr[uu]), L2E, X0);
                        X1 = fmaf(GW::hi(gr[uu]), L2E, X1);
                        const uint32_t off = xo[uu & 7] + (uu >> 3) * 1024;
                        const uint32_t kw = *reinterpret_cast<const uint32_t *>(qk + ST_K0 + off);
                        const bool in = t < len;
                        const float k0 = in ? In<Tin>::lo(kw) * ex2(e0 - X0) : 0.f;
                        const float k1 = in ? In<Tin>::hi(kw) * ex2(e1 - X1) : 0.f;
                        *reinterpret_cast<uint32_t *>(kh + off) = pack_h2(k0, k1);
                    }
                    D0 = e0;
                    D1 = e1;
                    if (q == n - 1 && rq == 0) {
                        gts[key] = D0;   // the segment's total decay, for the start-state scan
                        gts[key + 1] = D1;
                    }
                }
                fence_proxy_async();
                bar_arrive(&prep[s]);
                if (!out && q == n - 1)
                    bar_arrive(&g_done[it.na & 3]);
            }
            qbase += n;
            if (out)
                nb += n;
            return true;
        };
        auto run_s = [&](const Item &it) -> bool { return gate(it, false); };
        auto run_o = [&](const Item &it) -> bool { return gate(it, true); };
        GLA_ITEM_LOOP(gating_all, run_s, run_o)
    } else if (warp < WC) {
        // ------------------------------------------------------------------ state group
        // Per output chunk the state buffer holds U = diag(2^G_a') S' + k~'^T V' (the previous chunk's state
        // at its anchor plus its contribution, or S_in before the first chunk), so that
        //   S = diag(2^(G_last' - G_a')) U   and   S' = diag(2^G_a) S = diag(e) U:
        // one multiply per element gives S' in fp32 (written back for the MMA (c) to accumulate onto) and in
        // fp16 (the A operand of the inter-chunk MMA (a)).
        const int b = tid - NA;
        const uint32_t lrow = static_cast<uint32_t>((warp & 3) * 32) << 16;
        float *clh = reinterpret_cast<float *>(sm + OFF_CL);
        int nb = 0;
        auto fail = [&]() { report(a.status, GLA_ERR_TIMEOUT); };
        auto run_s = [](const Item &) -> bool { return true; };   // no work of this group
        auto run_o = [&](const Item &it) -> bool {
            const int buf = it.itn & 1;
            const uint32_t sb = tmem + lrow + TM_S + buf * 128;
            const bool want_ht = it.last && a.ht != nullptr;
            const int u = (it.j * H + it.h) * NV + it.vt;
            if (!chain_scan(cx, it, u, TM_S + buf * 128, it.na))
                return false;
            for (int c = 0; c < it.nchunks; ++c) {
                const int gb = nb + c;
                // U holds the previous chunk's contribution (its MMA (c) is complete); the MMA (a) two chunks
                // back, the last reader of this chunk's S' buffer, is complete; the gating group has published
                // this chunk's factors (it may still be forming the operands)
                bool got = c == 0 || bar_wait(mma_st, (gb - 1) & 1, abort_w);
                got = got && (gb < 2 || bar_wait(&sop_free[gb & 1], ((gb - 2) >> 1) & 1, abort_w));
                got = got && bar_wait(&eg_ready[gb & 3], (gb >> 2) & 1, abort_w);
                if (!__all_sync(0xffffffffu, got))
                    return false;
                fence_after();
                const float *eg = reinterpret_cast<const float *>(sm + OFF_EG + (gb & 3) * 1024);
                if (want_ht && c == it.nchunks - 1)
                    clh[buf * 128 + b] = eg[128 + b];   // the last chunk's 2^(G_last - G_a), for ht
                uint32_t ra[16], rb[16];
                auto convert = [&](uint32_t(&r)[16], int qq) {
                    uint32_t op[8];
#pragma unroll
                    for (int w = 0; w < 16; w += 4) {
                        const float4 e = *reinterpret_cast<const float4 *>(eg + qq * 16 + w);
                        r[w] = __float_as_uint(__uint_as_float(r[w]) * e.x);
                        r[w + 1] = __float_as_uint(__uint_as_float(r[w + 1]) * e.y);
                        r[w + 2] = __float_as_uint(__uint_as_float(r[w + 2]) * e.z);
                        r[w + 3] = __float_as_uint(__uint_as_float(r[w + 3]) * e.w);
                    }
#pragma unroll
                    for (int w = 0; w < 8; ++w)
                        op[w] = pack_h2(__uint_as_float(r[2 * w]), __uint_as_float(r[2 * w + 1]));
                    tmem_st8(tmem + lrow + TM_SOP + (gb & 1) * 64 + qq * 8, op);
                    tmem_st16(sb + qq * 16, r);
                };
                tmem_ld16(sb, ra);
                tmem_wait_ld(ra);
#pragma unroll 1
                for (int qq = 0; qq < KD / 16; qq += 2) {
                    tmem_ld16(sb + (qq + 1) * 16, rb);
                    convert(ra, qq);
                    tmem_wait_ld(rb);
                    if (qq + 2 < KD / 16)
                        tmem_ld16(sb + (qq + 2) * 16, ra);
                    convert(rb, qq + 1);
                    if (qq + 2 < KD / 16)
                        tmem_wait_ld(ra);
                }
                tmem_wait_st();
                fence_before();
                bar_arrive(ops_ready);
            }
            // end of the item: final state (ht for a sequence's last segment), then release the buffer
            if (!__all_sync(0xffffffffu, bar_wait(&item_done[buf], (it.itn >> 1) & 1, abort_w)))
                return false;
            if (want_ht) {
                fence_after();
                sync_state();   // every key's factor is in clh
                const float *cl = clh + buf * 128;
                const bool scaled = it.nchunks > 0;   // without chunks the buffer holds S_in itself
                float *dst = a.ht + ((size_t)it.n * H + it.h) * KD * V + it.v0 + b;
                float fmax = 0.f;
                for (int kc = 0; kc < KD / 32; ++kc) {
                    uint32_t r[32];
                    tmem_ld32(sb + kc * 32, r);
                    tmem_wait_ld(r);
#pragma unroll
                    for (int uu = 0; uu < 32; ++uu) {
                        const float x = scaled ? __uint_as_float(r[uu]) * cl[kc * 32 + uu] : __uint_as_float(r[uu]);
                        fmax = amax_nan(fmax, x);
                        dst[(size_t)(kc * 32 + uu) * V] = x;
                    }
                }
                if (!finite(fmax))
                    report(a.status, GLA_ERR_RANGE);
            }
            fence_before();
            bar_arrive(&tmem_free[buf]);
            nb += it.nchunks;
            return true;
        };
        GLA_ITEM_LOOP(team_all, run_s, run_o)
    } else if (warp < WP) {
        // ------------------------------------------------------------------ output group (epilogue)
        const int b = tid - NA - NB;
        const uint32_t lrow = static_cast<uint32_t>((warp & 3) * 32) << 16;
        Tout *go = static_cast<Tout *>(a.o);
        const size_t rstride = HF ? (size_t)V : (size_t)H * V;   // between consecutive rows of o
        int nb = 0;
        auto fail = [&]() { report(a.status, GLA_ERR_TIMEOUT); };
        auto run_s = [](const Item &) -> bool { return true; };
        auto run_o = [&](const Item &it) -> bool {
            const int u = (it.j * H + it.h) * NV + it.vt;
            if (!chain_scan(cx, it, u, TM_S + (it.itn & 1) * 128, it.na))
                return false;
            for (int c = 0; c < it.nchunks; ++c) {
                const int gb = nb + c;
                const int row0 = it.bos + c * C;
                const int len = min(C, it.eos - row0);
                if (!output_all(bar_wait(mma2, gb & 1, abort_w)))
                    return false;
                fence_after();
                // O^T rows (lane = value column) straight from TMEM to global memory (q~ carries the scale):
                // for every row t the warp stores 32 consecutive values of o, one coalesced line per
                // instruction
                const uint32_t ob = tmem + lrow + TM_O;
                Tout *orow = go + row_head(row0, it.h, H, a.T, HF ? 1 : 0) * V + it.v0 + b;
                for (int half = 0; half < 2; ++half) {
                    uint32_t r[32];
                    tmem_ld32(ob + half * 32, r);
                    tmem_wait_ld(r);
                    if (half == 1) {
                        fence_before();
                        bar_arrive(o_free);   // all of O^T is in registers: the MMA (a) of the next chunk may run
                    }
                    Tout *orh = orow + (size_t)(32 * half) * rstride;
                    if (len == C) {
#pragma unroll
                        for (int uu = 0; uu < 32; ++uu) {
                            const float x = __uint_as_float(r[uu]);
                            omax = amax_nan(omax, x);
                            orh[(size_t)uu * rstride] = to_out<Tout>(x);
                        }
                    } else {
#pragma unroll
                        for (int uu = 0; uu < 32; ++uu) {
                            const float x = __uint_as_float(r[uu]);
                            if (32 * half + uu < len) {
                                omax = amax_nan(omax, x);
                                orh[(size_t)uu * rstride] = to_out<Tout>(x);
                            }
                        }
                    }
                }
            }
            nb += it.nchunks;
            return true;
        };
        GLA_ITEM_LOOP(team_all, run_s, run_o)
        if (!finite(omax))
            report(a.status, GLA_ERR_RANGE);
    } else if (warp < WCTL) {
        // ------------------------------------------------------------------ P group (2 warps)
        // P = q~ k~^T (TMEM lanes 0..63 = rows t) masked to s <= t (inclusive diagonal, by select), as the
        // fp16 K-major B operand of MMA (d).  MMA (b) of a chunk is issued after MMA (d) of the previous one,
        // so the completion of (b) also means the shared P tile is free again.
        const int t = tid - NA - NB - NC;
        const uint32_t lrow = static_cast<uint32_t>((warp & 3) * 32) << 16;
        int nb = 0;
        auto fail = [&]() { report(a.status, GLA_ERR_TIMEOUT); };
        auto run_s = [](const Item &) -> bool { return true; };
        auto run_o = [&](const Item &it) -> bool {
            for (int c = 0; c < it.nchunks; ++c) {
                const int gb = nb + c;
                if (!p_all(bar_wait(mma1, gb & 1, abort_w)))
                    return false;
                fence_after();
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + lrow + TM_P, r0);
                tmem_ld32(tmem + lrow + TM_P + 32, r1);
                tmem_wait_ld(r0);
                tmem_wait_ld(r1);
#pragma unroll
                for (int sc = 0; sc < 2; ++sc) {
#pragma unroll
                    for (int u0 = 0; u0 < 32; u0 += 8) {
                        uint32_t pk[4];
#pragma unroll
                        for (int w = 0; w < 8; w += 2) {
                            const int sa = sc * 32 + u0 + w;
                            const uint32_t x0 = sc ? r1[u0 + w] : r0[u0 + w];
                            const uint32_t x1 = sc ? r1[u0 + w + 1] : r0[u0 + w + 1];
                            const float p0 = sa <= t ? __uint_as_float(x0) : 0.f;
                            const float p1 = sa + 1 <= t ? __uint_as_float(x1) : 0.f;
                            pk[w / 2] = pack_h2(p0, p1);
                        }
                        *reinterpret_cast<uint4 *>(sm + OFF_P + sw128(t, sc * 32 + u0)) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
                fence_proxy_async();
                fence_before();
                bar_arrive(p_ready);
            }
            nb += it.nchunks;
            return true;
        };
        GLA_ITEM_LOOP(p_all, run_s, run_o)
    }
#undef GLA_ITEM_LOOP

    // let the last CTA out reset the work counters for the next call
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

template <typename Tin, typename Tg, typename Tout, bool HF>
cudaError_t launch_fused_t(const Plan &pl, const Args &a, cudaStream_t s, int sms)
{
    constexpr int SMEM_BYTES = Ring<sizeof(Tg)>::SMEM_BYTES;
    const long long rows = pl.varlen ? (long long)pl.T : (long long)pl.B * pl.T;
    const CUtensorMapDataType tin =
        std::is_same<Tin, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapDataType tg = std::is_same<Tg, float>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : tin;
    CUtensorMap mq, mk, mg, mv;
    const bool hf = HF;
    if (!encode_rows(&mq, a.q, pl.K, pl.H, rows, 64, C, true, tin, hf, pl.T) ||
        !encode_rows(&mk, a.k, pl.K, pl.H, rows, 64, C, true, tin, hf, pl.T) ||
        !encode_rows(&mg, a.g, pl.K, pl.H, rows, 128, C, false, tg, hf, pl.T) ||
        !encode_rows(&mv, a.v, pl.V, pl.H, rows, 64, C, true, tin, hf, pl.T))
        return cudaErrorInvalidValue;
    auto f = gla_fused<Tin, Tg, Tout, HF>;
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
    // work claims: items, or pieces per value tile
    int nitems = pl.np ? pl.np * (pl.V / VT) : pl.J * pl.H * (pl.V / VT);
    // scan block length: when every item runs at once the chain of end-state publications is the critical
    // path, so only every 8th segment publishes one; with several waves a block of 2 halves the chain of
    // dependent publications for one extra tile read on every other segment
    Args ka = a;
    ka.lb = nitems <= sms ? 8 : 2;
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
    void *args[] = {&mq, &mk, &mg, &mv, &ka, &nitems};
    cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(f), args);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(int dtype, int K, int V)
{
    // 16-bit q, k, v; g 16-bit or fp32
    return (dtype == GLA_BF16 || dtype == GLA_BF16_OBF16 || dtype == GLA_F16 || dtype == GLA_BF16_GF32 ||
            dtype == GLA_F16_GF32) &&
           K == KD && V % VT == 0 && V <= 256;
}

cudaError_t launch_fused_tc(const Plan &pl, const Args &a, cudaStream_t s, int sms)
{
    // the layout is a template parameter, so the time-major kernel carries no layout branches
    switch (pl.dtype) {
    case GLA_BF16_OBF16:
        return a.hf ? launch_fused_t<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16, true>(pl, a, s, sms)
                    : launch_fused_t<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16, false>(pl, a, s, sms);
    case GLA_F16:
        return a.hf ? launch_fused_t<__half, __half, float, true>(pl, a, s, sms)
                    : launch_fused_t<__half, __half, float, false>(pl, a, s, sms);
    case GLA_BF16_GF32:
        return a.hf ? launch_fused_t<__nv_bfloat16, float, float, true>(pl, a, s, sms)
                    : launch_fused_t<__nv_bfloat16, float, float, false>(pl, a, s, sms);
    case GLA_F16_GF32:
        return a.hf ? launch_fused_t<__half, float, float, true>(pl, a, s, sms)
                    : launch_fused_t<__half, float, float, false>(pl, a, s, sms);
    default:
        return a.hf ? launch_fused_t<__nv_bfloat16, __nv_bfloat16, float, true>(pl, a, s, sms)
                    : launch_fused_t<__nv_bfloat16, __nv_bfloat16, float, false>(pl, a, s, sms);
    }
}

}  // namespace gla
