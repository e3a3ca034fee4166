// Backward gradients of one chunk on the tensor cores (bf16 inputs, K = V = 128; page
// "fla/ops/gla/fused_chunk.py": bwd_inner_chunk and fused_chunk_gla_bwd_kernel, whose per-chunk products these
// are).  With G the chunk-local inclusive cumsum of the gates, the anchor row a = 31, q~ = q e^{G - G_a},
// k~ = k e^{G_a - G}, S_c the chunk-start state and R_c the chunk-end adjoint (both from the backward scan):
//
//   AM = scale mask(q~ k~^T),  BM = scale mask(do v^T)            (mask: column <= row, inclusive diagonal)
//   dq = e^{G - G_a} (BM k~ + do S'^T),        S' = scale diag(e^{G_a}) S_c
//   dk = e^{G_a - G} (BM^T q~ + v R'^T),       R' = diag(e^{G_l - G_a}) R_c
//   dv = AM^T do + k~ R'
//   dg (chunk-local) = suffix sums over rows of q dq - k dk,  and the chunk total for the carry scan.
//
// Every product is a tcgen05 kind::f16 MMA with bf16 operands and fp32 accumulation in TMEM, M = 128.  The
// three results are accumulated transposed (dq^T, dk^T with lane = key, dv^T with lane = value column), so
// every accumulator fills all 128 lanes and the epilogue thread that owns a key takes that key's cumsum and the
// dg suffix sums on its own.  Every operand is used in the layout it is stored in (K-major or MN-major
// descriptors, 128-byte swizzle): nothing is transposed.  q, k, v and do are exact in bf16; the computed
// operands (q~, k~, AM, BM, S', R') are split exactly into three bf16 terms x = x1 + x2 + x3:
// a product of two split operands takes the six term products above the third order (x1 y1, x1 y2, x2 y1,
// x1 y3, x2 y2, x3 y1), a split operand times an exact one three, so the result carries fp32-level error.
// Rows past the end of a chunk are zero in every operand.
//
// Persistent CTAs (one per SM, about 226 KB of shared memory) walk the (chunk, head) items.  Warps 0-7 form
// the operands and issue the products (thread 0 issues); warps 8-11 are the epilogue, one thread per TMEM
// lane.  The gating thread of a key and row half also leaves, in TMEM, that key's factors 2^(G - G_a) and
// 2^(G_a - G) on its rows and the raw q and k there (packed), so the epilogue reads TMEM only (and needs no
// exponentials) and writes the gradients while the operand
// warps go on to the next item's gating and score products.  The next item's q, k and g rows are copied in as
// soon as the current gating has read its own, its v and do rows as soon as the current products are
// complete.  The state tiles are read into registers while the products before them run: R' first (its
// products are the longer phase, under which S_c is read), then S'.
#include <algorithm>
#include <atomic>

#include <cuda_bf16.h>

#include "gla_internal.h"
#include "tc_ptx.cuh"

namespace gla {

namespace {

constexpr int CT = kChunk;    // 64 rows per chunk
constexpr int KD = 128;       // keys = value columns
constexpr int NMAIN = 256;    // warps 0-7: operands and products
constexpr int NEPI = 128;     // warps 8-11: epilogue
constexpr int NT = NMAIN + NEPI;
constexpr float L2E = 1.4426950408889634f;

// shared memory (offsets from a 1024-byte aligned base); a [64 rows][128] bf16 tile is two 64-column halves of
// 8 KB, a [128 rows][128] tile two halves of 16 KB, both 128-byte swizzled
constexpr int Q3 = 0;          // q~, three terms of 16 KB
constexpr int AM3 = 49152;     // AM, three terms of 8 KB ([64 rows i][64 columns j]); the gating's partial sums
                               // live here before AM is formed
constexpr int BM3 = 73728;     // BM, three terms of 8 KB
constexpr int ST3 = 0;         // R', then S': three terms of 32 KB ([128 keys][128 v]) over Q3 .. BM3
constexpr int K3 = 98304;      // k~, three terms of 16 KB
constexpr int DO = 147456;     // do [64 rows][128 v]
constexpr int VV = 163840;     // v
constexpr int RQ = 180224;     // raw rows, 256 bytes each: q
constexpr int RK = 196608;     // k
constexpr int RG = 212992;     // g
constexpr int MISC = 229376;   // FA[128] = scale 2^(G_a), FR[128] = 2^(G_l - G_a)
constexpr int BAR = MISC + 1024;   // mma, acc_full, acc_empty, xq_full, xq_free, TMEM address, abort word
constexpr int SMEM_BYTES = BAR + 64 + 1024;
// TMEM columns (lane = key or value column): the score tiles (lanes 0..63 = rows), for the epilogue the
// factors 2^(G - G_a), 2^(G_a - G) and the packed raw q | k per row, the accumulators dq^T, dk^T, dv^T
// (column = row)
constexpr uint32_t TM_AM = 0, TM_BM = 64, TM_EP = 128, TM_QK = 192, TM_DQ = 256, TM_DK = 320, TM_DV = 384,
                   TM_EM = 448;
constexpr uint32_t TM_COLS = 512;

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t ID = idesc_bf16(128, 64);


__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(tc::smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all_but_newest() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// barrier 1 over the 256 threads of warps 0-7; the second form also ANDs a predicate over them
__device__ __forceinline__ void main_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool main_and(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, 256, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v)
                 : "memory");
    return r != 0;
}

// Two fp32 values -> three bf16x2 words with x = x1 + x2 + x3 exactly for each: x1 is x rounded to 8
// significant bits (half-way cases away from zero) by an integer carry into the bits it keeps, x2 the
// remainder (exact, by Sterbenz's lemma) rounded the same way, and x3 the rest, which has at most 8
// significant bits.  Every term is a bf16 value without a conversion instruction; |x2| <= 2^-8 |x| and
// |x3| <= 2^-16 |x|.  The low halves of the words hold a's terms, the high halves b's.
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

__device__ __forceinline__ float lo16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// 4x4 transpose inside each quad of lanes: on entry lane p holds a[i] = element (key p, row i) of its quad's
// block, on exit a[i] = element (key i, row p), so that a lane can store four consecutive keys of one row.
__device__ __forceinline__ void quad_transpose(float (&a)[4], int p)
{
#pragma unroll
    for (int b = 1; b <= 2; b <<= 1) {
        const bool hi = (p & b) != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i & b)
                continue;
            const float send = hi ? a[i] : a[i | b];
            const float got = __shfl_xor_sync(0xffffffffu, send, b);
            if (hi)
                a[i] = got;
            else
                a[i | b] = got;
        }
    }
}

// K-major operand whose K index runs over two 64-element halves `hs` bytes apart: K step kk (16 elements)
// Shared-memory descriptors of the operand tiles, formed from bases computed once: K-major (step kk of 16 keys:
// 32 bytes inside a 128-byte row, 64-key halves `hs` bytes apart) and MN-major (step kk: 16 rows of 128 bytes;
// 64-element blocks `lbo` bytes apart).  The start-address field holds address >> 4 and shared addresses stay
// below 2^18, so adding an offset cannot carry out of it; with the MMA loops unrolled the offsets are constants
// and an issuing thread spends about half the cycles per tcgen05.mma that forming each descriptor anew costs.
struct Descs {
    uint64_t k, m8, m16;
    __device__ __forceinline__ uint64_t kd(uint32_t ofs, int kk, uint32_t hs) const
    {
        return k + ((ofs + (kk >> 2) * hs + (kk & 3) * 32) >> 4);
    }
    __device__ __forceinline__ uint64_t md8(uint32_t ofs, int kk) const { return m8 + ((ofs + kk * 2048) >> 4); }
    __device__ __forceinline__ uint64_t md16(uint32_t ofs, int kk) const { return m16 + ((ofs + kk * 2048) >> 4); }
};

// One (chunk, head) item: rows [bos, bos + len) of head h; row t of the chunk is row-head index rb + t * rs.
struct Item {
    int j, h, len;
    size_t rb;
};

// The first used item at or after u on this CTA's stride (items u = j * H + h), or -1.
__device__ __forceinline__ int next_item(const BwdArgs &a, int u, int nitems, Item &it)
{
    for (; u < nitems; u += gridDim.x) {
        const int j = u / a.H, h = u - j * a.H;
        int bos, eos;
        if (a.table) {
            const int4 e = a.table[j];
            if (e.x < 0)
                continue;
            bos = e.z;
            eos = e.w;
        } else {
            const int n = j / a.NC, c = j - n * a.NC;
            bos = n * a.T + c * CT;
            eos = min(bos + CT, n * a.T + a.T);
        }
        it.j = j;
        it.h = h;
        it.len = eos - bos;
        it.rb = row_head(bos, h, a.H, a.T, a.hf);
        return u;
    }
    return -1;
}

__global__ void __launch_bounds__(NT, 1) bwd_grads_tc(BwdArgs a, int nitems)
{
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char *sm = smraw + ((1024u - (tc::smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t *bar_mma = reinterpret_cast<uint64_t *>(sm + BAR);
    uint64_t *acc_full = bar_mma + 1, *acc_empty = bar_mma + 2, *xq_full = bar_mma + 3, *xq_free = bar_mma + 4;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + BAR + 40);
    volatile int *abort_w = reinterpret_cast<volatile int *>(sm + BAR + 44);
    float *FA = reinterpret_cast<float *>(sm + MISC), *FR = FA + 128;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, H = a.H;
    const int rs = a.hf ? 1 : H;

    if (tid == 0) {
        tc::bar_init(bar_mma, 1);
        tc::bar_init(acc_full, 1);
        tc::bar_init(acc_empty, NEPI);
        tc::bar_init(xq_full, NMAIN);
        tc::bar_init(xq_free, NEPI);
        *abort_w = 0;
        tc::bar_fence_init();
    }
    if (warp == 0)
        tc::tmem_alloc(tslot, TM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t sb = tc::smem_u32(sm);

    if (warp < 8) {
        // ================================ operands and products ================================
        // copies of an item's rows (rows past its end are zero-filled): q, k, g as plain 256-byte rows;
        // v and do straight into their swizzled operand tiles
        auto copy_rows = [&](const Item &it, bool raw) {
#pragma unroll
            for (int w = 0; w < 3; ++w) {
                if (!raw && w == 2)
                    break;
                const int which = raw ? w : 3 + w;
                const void *src = which == 0 ? a.q : which == 1 ? a.k : which == 2 ? a.g : which == 3 ? a.v : a.dout;
                const int dst = which == 0 ? RQ : which == 1 ? RK : which == 2 ? RG : which == 3 ? VV : DO;
#pragma unroll
                for (int r = tid; r < CT * 16; r += NMAIN) {
                    const int t = r >> 4, c = r & 15;
                    const bool in = t < it.len;
                    const size_t ld = which < 3 ? (size_t)KD : (size_t)a.ldv;   // v and do: the caller's stride
                    const unsigned char *s = static_cast<const unsigned char *>(src) +
                                             ((it.rb + (size_t)(in ? t : 0) * rs) * ld + 8 * c) * 2;
                    const uint32_t off = which < 3 ? (uint32_t)(t * 256 + 16 * c)
                                                   : (uint32_t)((c >> 3) * 8192) + tc::sw128(t, 8 * (c & 7));
                    cp_async16(sm + dst + off, s, in ? 16u : 0u);
                }
            }
        };

        bool ok = true;
        uint32_t mph = 0;   // completed waits on bar_mma
        const Descs dsc{tc::sdesc_sw128(sb), tc::sdesc_mn_sw128(sb, 8192), tc::sdesc_mn_sw128(sb, 16384)};
        auto wait_mma = [&]() {
            const bool got = tc::bar_wait(bar_mma, mph & 1, abort_w);
            ++mph;
            ok = main_and(got && ok);
            tc::fence_after();
        };
        auto publish = [&]() {   // generic-proxy stores of all main threads -> visible to the next MMAs
            tc::fence_proxy_async();
            tc::fence_before();
            main_sync();
            tc::fence_after();
        };

        // the state tiles [128 keys][128 v] fp32 of an item (its slot in the workspace): into registers,
        // then key-scaled and split into three bf16 terms over the q~ / AM / BM space
        float4 st[16];
        auto fetch_state = [&](const float *src, const Item &it) {
            const size_t tile = ((size_t)it.j * H + it.h) * KD * KD;
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const int e = tid + v * NMAIN, key = e >> 4, c = e & 15;
                const float4 *p = reinterpret_cast<const float4 *>(src + tile + (size_t)key * KD + 8 * c);
                st[2 * v] = __ldcg(p);
                st[2 * v + 1] = __ldcg(p + 1);
            }
        };
        auto split_state = [&](const float *f) {
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const int e = tid + v * NMAIN, key = e >> 4, c = e & 15;
                const float fk = f[key];
                const float4 x0 = st[2 * v], x1 = st[2 * v + 1];
                uint32_t w1[4], w2[4], w3[4];
                split3(fk * x0.x, fk * x0.y, w1[0], w2[0], w3[0]);
                split3(fk * x0.z, fk * x0.w, w1[1], w2[1], w3[1]);
                split3(fk * x1.x, fk * x1.y, w1[2], w2[2], w3[2]);
                split3(fk * x1.z, fk * x1.w, w1[3], w2[3], w3[3]);
                const uint32_t off = (uint32_t)((c >> 3) * 16384) + tc::sw128(key, 8 * (c & 7));
                *reinterpret_cast<uint4 *>(sm + ST3 + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
                *reinterpret_cast<uint4 *>(sm + ST3 + 32768 + off) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
                *reinterpret_cast<uint4 *>(sm + ST3 + 65536 + off) = make_uint4(w3[0], w3[1], w3[2], w3[3]);
            }
            publish();
        };

        Item cur, nxt;
        int u = next_item(a, blockIdx.x, nitems, cur);
        if (u >= 0)
            copy_rows(cur, true);
        cp_commit();
        if (u >= 0)
            copy_rows(cur, false);
        cp_commit();
        for (int nit = 0; u >= 0; ++nit) {
            const int un = next_item(a, u + gridDim.x, nitems, nxt);
            const int len = cur.len;
            cp_wait_all_but_newest();   // this item's q, k, g
            main_sync();

            // ---- gating: thread (key k, row half rh); cumsum in log2 units, the halves' sums exchanged
            const int gk = 32 * (warp & 3) + lane, rh = warp >> 2, gr0 = 32 * rh;
            const uint32_t glane = (uint32_t)(32 * (warp & 3)) << 16;
            uint32_t ep[32], em[32], qk[32];   // 2^(G - G_a), 2^(G_a - G) and raw q | k on the half's rows
            {
                const unsigned short *rgp = reinterpret_cast<const unsigned short *>(sm + RG);
                const unsigned short *rqp = reinterpret_cast<const unsigned short *>(sm + RQ);
                const unsigned short *rkp = reinterpret_cast<const unsigned short *>(sm + RK);
                float *psum = reinterpret_cast<float *>(sm + AM3);
                float gv[32], sum = 0.f;
#pragma unroll
                for (int v = 0; v < 32; ++v) {
                    const int t = gr0 + v;
                    gv[v] = t < len ? __uint_as_float(static_cast<uint32_t>(rgp[t * KD + gk]) << 16) * L2E : 0.f;
                    sum += gv[v];
                }
                psum[rh * KD + gk] = sum;
                main_sync();
                const float ga = psum[gk], gl = ga + psum[KD + gk];
                if (rh == 0) {
                    FA[gk] = a.scale * tc::ex2(ga);
                    FR[gk] = tc::ex2(gl - ga);
                }
                float G = rh ? ga : 0.f;
                const int kb = gk >> 6, kc = gk & 63;
#pragma unroll
                for (int v = 0; v < 32; ++v) {
                    const int t = gr0 + v;
                    G += gv[v];
                    const float X = G - ga, fp = tc::ex2(X), fm = tc::ex2(-X);
                    ep[v] = __float_as_uint(fp);
                    em[v] = __float_as_uint(fm);
                    const bool in = t < len;
                    const uint32_t qr = rqp[t * KD + gk], kr = rkp[t * KD + gk];
                    qk[v] = in ? (qr << 16) | kr : 0u;
                    const float qt = in ? __uint_as_float(qr << 16) * fp : 0.f;
                    const float kt = in ? __uint_as_float(kr << 16) * fm : 0.f;
                    const uint32_t off = (uint32_t)(kb * 8192) + tc::sw128(t, kc);
                    uint32_t w[3];   // (q~, k~) term pairs: q~ in the low halves, k~ in the high ones
                    split3(qt, kt, w[0], w[1], w[2]);
#pragma unroll
                    for (int e = 0; e < 3; ++e) {
                        *reinterpret_cast<unsigned short *>(sm + Q3 + e * 16384 + off) = (unsigned short)(w[e] & 0xFFFFu);
                        *reinterpret_cast<unsigned short *>(sm + K3 + e * 16384 + off) = (unsigned short)(w[e] >> 16);
                    }
                }
            }
            main_sync();   // the raw rows are read: the next item's q, k, g may come in
            if (un >= 0)
                copy_rows(nxt, true);
            cp_commit();
            // the factors and q | k to TMEM for the epilogue, once it has read the previous item's
            if (nit == 0 || tc::bar_wait(xq_free, (nit - 1) & 1, abort_w)) {
                tc::fence_after();
                tc::tmem_st32(tmem + glane + TM_EP + gr0, ep);
                tc::tmem_st32(tmem + glane + TM_EM + gr0, em);
                tc::tmem_st32(tmem + glane + TM_QK + gr0, qk);
                tc::tmem_wait_st();
            }
            tc::fence_before();
            tc::bar_arrive(xq_full);
            cp_wait_all_but_newest();   // this item's v, do
            publish();

            // ---- AM = q~ k~^T (six term products), BM = do v^T
            if (tid == 0) {
#pragma unroll
                for (int ta = 0; ta < 3; ++ta)
                    for (int tb = 0; ta + tb < 3; ++tb)
                        for (int kk = 0; kk < 8; ++kk)
                            tc::mma_ss(tmem + TM_AM, dsc.kd(Q3 + ta * 16384, kk, 8192),
                                       dsc.kd(K3 + tb * 16384, kk, 8192), ID, (ta | tb | kk) ? 1u : 0u);
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_ss(tmem + TM_BM, dsc.kd(DO, kk, 8192), dsc.kd(VV, kk, 8192), ID, kk ? 1u : 0u);
                tc::mma_commit(bar_mma);
            }
            wait_mma();
            if (!ok)
                break;

            // ---- AM, BM (TMEM lanes 0..63 = rows i, columns j) -> scale, inclusive causal mask, three bf16
            //      terms in their [i][j] tiles: warps 0, 1 take AM, warps 4, 5 BM
            if ((warp & 2) == 0) {
                const int i = 32 * (warp & 1) + lane;
                const bool isb = warp >= 4;
                const uint32_t col = isb ? TM_BM : TM_AM;
                const int dst = isb ? BM3 : AM3;
                uint32_t r0[32], r1[32];
                tc::tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + col, r0);
                tc::tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + col + 32, r1);
                tc::tmem_wait_ld(r0);
                tc::tmem_wait_ld(r1);
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    uint32_t w1[4], w2[4], w3[4];
#pragma unroll
                    for (int pr = 0; pr < 4; ++pr) {
                        const int jj = 8 * c8 + 2 * pr;
                        const uint32_t xa = c8 < 4 ? r0[jj & 31] : r1[jj & 31];
                        const uint32_t xb = c8 < 4 ? r0[(jj + 1) & 31] : r1[(jj + 1) & 31];
                        const float va = jj <= i ? a.scale * __uint_as_float(xa) : 0.f;
                        const float vb = jj + 1 <= i ? a.scale * __uint_as_float(xb) : 0.f;
                        split3(va, vb, w1[pr], w2[pr], w3[pr]);
                    }
                    const uint32_t off = tc::sw128(i, 8 * c8);
                    *reinterpret_cast<uint4 *>(sm + dst + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
                    *reinterpret_cast<uint4 *>(sm + dst + 8192 + off) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
                    *reinterpret_cast<uint4 *>(sm + dst + 16384 + off) = make_uint4(w3[0], w3[1], w3[2], w3[3]);
                }
            }
            publish();

            // ---- the products with the score tiles, into the accumulators once the epilogue has drained the
            //      previous item's: dq^T = k~^T BM^T, dk^T = q~^T BM, dv^T = do^T AM
            const uint32_t acc = tmem;
            if (tid == 0 && (nit == 0 || tc::bar_wait(acc_empty, (nit - 1) & 1, abort_w))) {
                tc::fence_after();
#pragma unroll
                for (int ta = 0; ta < 3; ++ta)
                    for (int tb = 0; ta + tb < 3; ++tb)
                        for (int kk = 0; kk < 4; ++kk)
                            tc::mma_ss(acc + TM_DQ, dsc.md8(K3 + ta * 16384, kk),
                                       dsc.kd(BM3 + tb * 8192, kk, 0), ID | tc::kIdescAMajorMN,
                                       (ta | tb | kk) ? 1u : 0u);
#pragma unroll
                for (int ta = 0; ta < 3; ++ta)
                    for (int tb = 0; ta + tb < 3; ++tb)
                        for (int kk = 0; kk < 4; ++kk)
                            tc::mma_ss(acc + TM_DK, dsc.md8(Q3 + ta * 16384, kk),
                                       dsc.md8(BM3 + tb * 8192, kk),
                                       ID | tc::kIdescAMajorMN | tc::kIdescBMajorMN, (ta | tb | kk) ? 1u : 0u);
#pragma unroll
                for (int t = 0; t < 3; ++t)
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_ss(acc + TM_DV, dsc.md8(DO, kk), dsc.md8(AM3 + t * 8192, kk),
                                   ID | tc::kIdescAMajorMN | tc::kIdescBMajorMN, (t | kk) ? 1u : 0u);
                tc::mma_commit(bar_mma);
            }
            fetch_state(a.dR, cur);
            wait_mma();
            if (!ok)
                break;

            // ---- R' = 2^(G_l - G_a) R_c: dk^T += R' v^T, dv^T += R'^T k~^T
            split_state(FR);
            if (tid == 0) {
#pragma unroll
                for (int t = 0; t < 3; ++t)
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma_ss(acc + TM_DK, dsc.kd(ST3 + t * 32768, kk, 16384), dsc.kd(VV, kk, 8192),
                                   ID, 1u);
#pragma unroll
                for (int ta = 0; ta < 3; ++ta)
                    for (int tb = 0; ta + tb < 3; ++tb)
                        for (int kk = 0; kk < 8; ++kk)
                            tc::mma_ss(acc + TM_DV, dsc.md16(ST3 + ta * 32768, kk),
                                       dsc.kd(K3 + tb * 16384, kk, 8192), ID | tc::kIdescAMajorMN, 1u);
                tc::mma_commit(bar_mma);
            }
            fetch_state(a.dS, cur);
            wait_mma();
            if (!ok)
                break;

            // ---- S' = scale 2^(G_a) S_c: dq^T += S' do^T; the accumulator set goes to the epilogue
            split_state(FA);
            if (tid == 0) {
#pragma unroll
                for (int t = 0; t < 3; ++t)
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma_ss(acc + TM_DQ, dsc.kd(ST3 + t * 32768, kk, 16384), dsc.kd(DO, kk, 8192),
                                   ID, 1u);
                tc::mma_commit(bar_mma);
                tc::mma_commit(acc_full);
            }
            wait_mma();   // every operand tile is free again
            if (!ok)
                break;
            if (un >= 0)
                copy_rows(nxt, false);
            cp_commit();
            cur = nxt;
            u = un;
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
    } else {
        // ================================ epilogue ================================
        // Thread = TMEM lane k: key k of dq^T and dk^T, value column k of dv^T.  Rows 32..63 first, then
        // 0..31, so that the dg suffix sums run from the last row in one pass.  Results go out as 16-byte
        // stores of four consecutive keys of one row, after a transpose inside each quad of lanes.
        const int k = 32 * (warp & 3) + lane, p = lane & 3, kq = k - p;
        const uint32_t lrow = (uint32_t)(32 * (warp & 3)) << 16;
        Item it;
        for (int u = next_item(a, blockIdx.x, nitems, it), nit = 0; u >= 0;
             u = next_item(a, u + gridDim.x, nitems, it), ++nit) {
            const int len = it.len;
            const size_t rb = it.rb;
            // rows r0 + 4 g + p (g = 0..7) of v[]: four keys from kq on, one 16-byte store each (rows ld apart;
            // added to what is there when acc)
            auto store_rows = [&](float *out, const uint32_t (&v)[32], int r0, size_t ld, int acc) {
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    float q4[4] = {__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                                   __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3])};
                    quad_transpose(q4, p);
                    const int t = r0 + 4 * g + p;
                    if (t < len) {
                        float4 *dst = reinterpret_cast<float4 *>(out + (rb + (size_t)t * rs) * ld + kq);
                        float4 x = make_float4(q4[0], q4[1], q4[2], q4[3]);
                        if (acc) {
                            const float4 o = *dst;
                            x.x += o.x;
                            x.y += o.y;
                            x.z += o.z;
                            x.w += o.w;
                        }
                        *dst = x;
                    }
                }
            };
            if (!tc::bar_wait(acc_full, nit & 1, abort_w) || !tc::bar_wait(xq_full, nit & 1, abort_w))
                break;
            tc::fence_after();
            const uint32_t tl = tmem + lrow;
            float run = 0.f;
#pragma unroll 1
            for (int half = 1; half >= 0; --half) {
                const int r0 = 32 * half;
                float pd[32];
                uint32_t f[32], qk[32], r[32];   // f: a factor; r: an accumulator, then the results in its place
                tc::tmem_ld32(tl + TM_EM + r0, f);
                tc::tmem_ld32(tl + TM_QK + r0, qk);
                tc::tmem_ld32(tl + TM_DK + r0, r);
                tc::tmem_wait_ld(f);
                tc::tmem_wait_ld(qk);
                tc::tmem_wait_ld(r);
#pragma unroll
                for (int v = 0; v < 32; ++v) {
                    const float dk = __uint_as_float(f[v]) * __uint_as_float(r[v]);
                    pd[v] = -lo16(qk[v]) * dk;
                    r[v] = __float_as_uint(dk);
                }
                store_rows(a.dk, r, r0, KD, a.acc);
                tc::tmem_ld32(tl + TM_EP + r0, f);
                tc::tmem_ld32(tl + TM_DQ + r0, r);
                tc::tmem_wait_ld(f);
                tc::tmem_wait_ld(r);
                if (half == 0) {   // the factors and q | k are read: the next item's may come in
                    tc::fence_before();
                    tc::bar_arrive(xq_free);
                }
#pragma unroll
                for (int v = 0; v < 32; ++v) {
                    const float dq = __uint_as_float(f[v]) * __uint_as_float(r[v]);
                    pd[v] = fmaf(hi16(qk[v]), dq, pd[v]);
                    r[v] = __float_as_uint(dq);
                }
                store_rows(a.dq, r, r0, KD, a.acc);
#pragma unroll
                for (int v = 31; v >= 0; --v) {
                    run += r0 + v < len ? pd[v] : 0.f;
                    r[v] = __float_as_uint(run);
                }
                store_rows(a.dg, r, r0, KD, a.acc);
                tc::tmem_ld32(tl + TM_DV + r0, r);
                tc::tmem_wait_ld(r);
                if (half == 0) {   // the accumulators are read: the next item's products may start
                    tc::fence_before();
                    tc::bar_arrive(acc_empty);
                }
                store_rows(a.dv, r, r0, a.ldv, 0);
            }
            a.dgt[((size_t)it.j * H + it.h) * KD + k] = run;
        }
    }

    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (tid == 0 && *abort_w)
        report(a.status, GLA_ERR_TIMEOUT);
    if (warp == 0)
        tc::tmem_dealloc(tmem, TM_COLS);
}

}  // namespace

bool bwd_grads_tc_supported(int dtype, int K, int V)
{
    return dtype == GLA_BF16 && K == KD && V == KD;
}

cudaError_t launch_bwd_grads_tc(const BwdArgs &a, int J, cudaStream_t s)
{
    static std::atomic<uint64_t> ready{0};   // per-device shared-memory opt-in and SM count, done once
    static std::atomic<int> sm_count[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(ready.load(std::memory_order_acquire) & bit)) {
        if ((e = cudaFuncSetAttribute(bwd_grads_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)) !=
            cudaSuccess)
            return e;
        int sms = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        sm_count[dev & 63].store(sms, std::memory_order_relaxed);
        ready.fetch_or(bit, std::memory_order_release);
    }
    const int nitems = J * a.H;
    const int grid = std::min(nitems, sm_count[dev & 63].load(std::memory_order_relaxed));
    if (grid <= 0)
        return cudaSuccess;
    bwd_grads_tc<<<grid, NT, SMEM_BYTES, s>>>(a, nitems);
    return cudaGetLastError();
}

}  // namespace gla
