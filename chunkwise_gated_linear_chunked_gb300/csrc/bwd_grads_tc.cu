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
// One CTA (8 warps) per (chunk, head).  Every product is a tcgen05 kind::f16 MMA with bf16 operands and fp32
// accumulation in TMEM, M = 128.  The three results are accumulated transposed (dq^T, dk^T with lane = key,
// dv^T with lane = value column), so every accumulator fills all 128 lanes and the epilogue thread that owns a
// key recomputes that key's cumsum and takes the dg suffix sums on its own.  Every operand is used in the
// layout it is stored in (K-major or MN-major descriptors, 128-byte swizzle): nothing is transposed.  q, k,
// v and do are exact in bf16; the computed operands (q~, k~, AM, BM, S', R') are split into three bf16 terms
// x = x1 + x2 + x3 (exact to fp32 rounding): a product of two split operands takes the six term products
// above the third order (x1 y1, x1 y2, x2 y1, x1 y3, x2 y2, x3 y1), a split operand times an exact one three,
// so the result carries fp32-level error.  The state tiles S' and R' (three 32 KB terms each) are formed in
// turn in the space of q~, AM and BM once the products that read those are complete.  Rows past the end of a
// chunk are zero in every operand.  About 226 KB of shared memory: one CTA per SM.
#include <atomic>

#include <cuda_bf16.h>

#include "gla_internal.h"
#include "tc_ptx.cuh"

namespace gla {

namespace {

constexpr int CT = kChunk;   // 64 rows per chunk
constexpr int KD = 128;      // keys = value columns
constexpr int NT = 256;      // threads per CTA
constexpr float L2E = 1.4426950408889634f;

// shared memory (offsets from a 1024-byte aligned base); a [64 rows][128] bf16 tile is two 64-column halves of
// 8 KB, a [128 rows][128] tile two halves of 16 KB, both 128-byte swizzled
constexpr int Q3 = 0;          // q~, three terms of 16 KB
constexpr int AM3 = 49152;     // AM, three terms of 8 KB ([64 rows i][64 columns j]); the gating's partial sums
                               // live here before AM is formed
constexpr int BM3 = 73728;     // BM, three terms of 8 KB
constexpr int ST3 = 0;         // S', then R': three terms of 32 KB ([128 keys][128 v]) over Q3 .. BM3
constexpr int K3 = 98304;      // k~, three terms of 16 KB
constexpr int DO = 147456;     // do [64 rows][128 v]
constexpr int VV = 163840;     // v
constexpr int RQ = 180224;     // raw rows, 256 bytes each: q
constexpr int RK = 196608;     // k
constexpr int RG = 212992;     // g
constexpr int MISC = 229376;   // FA[128] = scale 2^(G_a), FR[128] = 2^(G_l - G_a); the dg partial totals in FA's
                               // place in the epilogue
constexpr int BAR = MISC + 1536;
constexpr int SMEM_BYTES = BAR + 16 + 1024;
constexpr uint32_t TM_AM = 0, TM_BM = 64, TM_DQ = 128, TM_DK = 192, TM_DV = 256, TM_COLS = 512;

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t ID = idesc_bf16(128, 64);

// term pairs of a product of two split operands (i + j <= 2)
__device__ constexpr int PA[6] = {0, 0, 1, 0, 1, 2};
__device__ constexpr int PB[6] = {0, 1, 0, 2, 1, 0};

__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(tc::smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// Two fp32 values -> three bf16x2 words (x = x1 + x2 + x3 for each, exact to fp32 rounding).
__device__ __forceinline__ void split3(float a, float b, uint32_t &w1, uint32_t &w2, uint32_t &w3)
{
    const __nv_bfloat162 x1 = __floats2bfloat162_rn(a, b);
    const float2 y1 = __bfloat1622float2(x1);
    const float ra = a - y1.x, rb = b - y1.y;
    const __nv_bfloat162 x2 = __floats2bfloat162_rn(ra, rb);
    const float2 y2 = __bfloat1622float2(x2);
    const __nv_bfloat162 x3 = __floats2bfloat162_rn(ra - y2.x, rb - y2.y);
    w1 = *reinterpret_cast<const uint32_t *>(&x1);
    w2 = *reinterpret_cast<const uint32_t *>(&x2);
    w3 = *reinterpret_cast<const uint32_t *>(&x3);
}

__device__ __forceinline__ float lo16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf(const unsigned short *p) { return __uint_as_float(static_cast<uint32_t>(*p) << 16); }

// K-major operand whose K index runs over two 64-element halves `hs` bytes apart: K step kk (16 elements)
__device__ __forceinline__ uint64_t kdesc(uint32_t base, int kk, uint32_t hs)
{
    return tc::sdesc_sw128(base + (kk >> 2) * hs + (kk & 3) * 32);
}
// MN-major operand (MN blocks of 64 `lbo` bytes apart, K = rows of 128 bytes): K step kk (16 rows)
__device__ __forceinline__ uint64_t mdesc(uint32_t base, int kk, uint32_t lbo)
{
    return tc::sdesc_mn_sw128(base + kk * 2048, lbo);
}

__global__ void __launch_bounds__(NT, 1) bwd_grads_tc(BwdArgs a)
{
    extern __shared__ __align__(16) unsigned char smraw[];
    unsigned char *sm = smraw + ((1024u - (tc::smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + BAR + 8);
    float *FA = reinterpret_cast<float *>(sm + MISC), *FR = FA + 128;
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
    (void)n;
    const int len = eos - bos, H = a.H;
    const size_t rb = row_head(bos, h, H, a.T, a.hf);   // row t of the chunk: row-head index rb + t * rs
    const int rs = a.hf ? 1 : H;

    // ---- rows of the chunk by 16-byte asynchronous copies (rows past the end are zero-filled): q, k, g as
    //      plain 256-byte rows; v and do straight into their swizzled operand tiles
    {
#pragma unroll
        for (int which = 0; which < 5; ++which) {
            const void *src = which == 0 ? a.q : which == 1 ? a.k : which == 2 ? a.g : which == 3 ? a.v : a.dout;
            const int dst = which == 0 ? RQ : which == 1 ? RK : which == 2 ? RG : which == 3 ? VV : DO;
            for (int r = tid; r < CT * 16; r += NT) {
                const int t = r >> 4, c = r & 15;
                const bool in = t < len;
                const unsigned char *s =
                    static_cast<const unsigned char *>(src) + ((rb + (size_t)(in ? t : 0) * rs) * KD + 8 * c) * 2;
                const uint32_t off = which < 3 ? (uint32_t)(t * 256 + 16 * c)
                                               : (uint32_t)((c >> 3) * 8192) + tc::sw128(t, 8 * (c & 7));
                cp_async16(sm + dst + off, s, in ? 16u : 0u);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    if (tid == 0) {
        tc::bar_init(bar, 1);
        tc::bar_fence_init();
    }
    if (warp == 0)
        tc::tmem_alloc(tslot, TM_COLS);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t sb = tc::smem_u32(sm);

    // ---- gating: thread (key pair kp, row quarter rq); cumsum in log2 units, partial sums exchanged
    {
        const int kp = tid & 63, rq = tid >> 6, key = 2 * kp, kb = key >> 6, kc = key & 63;
        float *psum = reinterpret_cast<float *>(sm + AM3);
        uint32_t gr[16];
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int t = 16 * rq + u;
            gr[u] = t < len ? *reinterpret_cast<const uint32_t *>(sm + RG + t * 256 + kp * 4) : 0u;
            s0 = fmaf(lo16(gr[u]), L2E, s0);
            s1 = fmaf(hi16(gr[u]), L2E, s1);
        }
        psum[rq * 128 + key] = s0;
        psum[rq * 128 + key + 1] = s1;
        __syncthreads();
        float p0[4], p1[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            p0[r] = psum[r * 128 + key];
            p1[r] = psum[r * 128 + key + 1];
        }
        const float ga0 = p0[0] + p0[1], ga1 = p1[0] + p1[1];
        const float gl0 = ga0 + p0[2] + p0[3], gl1 = ga1 + p1[2] + p1[3];
        if (rq == 0) {
            FA[key] = a.scale * tc::ex2(ga0);
            FA[key + 1] = a.scale * tc::ex2(ga1);
            FR[key] = tc::ex2(gl0 - ga0);
            FR[key + 1] = tc::ex2(gl1 - ga1);
        }
        float X0 = (rq >= 1 ? p0[0] : 0.f) + (rq >= 2 ? p0[1] : 0.f) + (rq >= 3 ? p0[2] : 0.f) - ga0;
        float X1 = (rq >= 1 ? p1[0] : 0.f) + (rq >= 2 ? p1[1] : 0.f) + (rq >= 3 ? p1[2] : 0.f) - ga1;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int t = 16 * rq + u;
            X0 = fmaf(lo16(gr[u]), L2E, X0);
            X1 = fmaf(hi16(gr[u]), L2E, X1);
            const uint32_t qw = *reinterpret_cast<const uint32_t *>(sm + RQ + t * 256 + kp * 4);
            const uint32_t kw = *reinterpret_cast<const uint32_t *>(sm + RK + t * 256 + kp * 4);
            const bool in = t < len;
            const float eq0 = tc::ex2(X0), eq1 = tc::ex2(X1), ek0 = tc::ex2(-X0), ek1 = tc::ex2(-X1);
            const float q0 = in ? lo16(qw) * eq0 : 0.f, q1 = in ? hi16(qw) * eq1 : 0.f;
            const float k0 = in ? lo16(kw) * ek0 : 0.f, k1 = in ? hi16(kw) * ek1 : 0.f;
            const uint32_t off = (uint32_t)(kb * 8192) + tc::sw128(t, kc);
            uint32_t w1, w2, w3;
            split3(q0, q1, w1, w2, w3);
            *reinterpret_cast<uint32_t *>(sm + Q3 + off) = w1;
            *reinterpret_cast<uint32_t *>(sm + Q3 + 16384 + off) = w2;
            *reinterpret_cast<uint32_t *>(sm + Q3 + 32768 + off) = w3;
            split3(k0, k1, w1, w2, w3);
            *reinterpret_cast<uint32_t *>(sm + K3 + off) = w1;
            *reinterpret_cast<uint32_t *>(sm + K3 + 16384 + off) = w2;
            *reinterpret_cast<uint32_t *>(sm + K3 + 32768 + off) = w3;
        }
    }
    tc::fence_proxy_async();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();

    bool ok = true;
    uint32_t phase = 0;
    auto wait_mma = [&]() {
        const bool got = tc::bar_wait(bar, phase & 1);
        ++phase;
        ok = __syncthreads_and(got && ok) != 0;
        tc::fence_after();
    };

    // ---- AM = q~ k~^T (six term products), BM = do v^T
    if (tid == 0) {
        for (int p = 0; p < 6; ++p)
            for (int kk = 0; kk < 8; ++kk)
                tc::mma_ss(tmem + TM_AM, kdesc(sb + Q3 + PA[p] * 16384, kk, 8192),
                           kdesc(sb + K3 + PB[p] * 16384, kk, 8192), ID, (p | kk) ? 1u : 0u);
        for (int kk = 0; kk < 8; ++kk)
            tc::mma_ss(tmem + TM_BM, kdesc(sb + DO, kk, 8192), kdesc(sb + VV, kk, 8192), ID, kk ? 1u : 0u);
        tc::mma_commit(bar);
    }
    wait_mma();

    // ---- AM, BM (TMEM lanes 0..63 = rows i, columns j) -> scale, inclusive causal mask, three bf16 terms in
    //      their [i][j] tiles: warps 0, 1 take AM, warps 4, 5 BM
    if (ok && (warp & 3) < 2 && (warp & 2) == 0) {
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
    tc::fence_proxy_async();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();

    // ---- the products with the score tiles: dq^T = k~^T BM^T, dk^T = q~^T BM, dv^T = do^T AM
    if (ok && tid == 0) {
        for (int p = 0; p < 6; ++p)
            for (int kk = 0; kk < 4; ++kk)
                tc::mma_ss(tmem + TM_DQ, mdesc(sb + K3 + PA[p] * 16384, kk, 8192),
                           kdesc(sb + BM3 + PB[p] * 8192, kk, 0), ID | tc::kIdescAMajorMN, (p | kk) ? 1u : 0u);
        for (int p = 0; p < 6; ++p)
            for (int kk = 0; kk < 4; ++kk)
                tc::mma_ss(tmem + TM_DK, mdesc(sb + Q3 + PA[p] * 16384, kk, 8192),
                           mdesc(sb + BM3 + PB[p] * 8192, kk, 8192), ID | tc::kIdescAMajorMN | tc::kIdescBMajorMN,
                           (p | kk) ? 1u : 0u);
        for (int t = 0; t < 3; ++t)
            for (int kk = 0; kk < 4; ++kk)
                tc::mma_ss(tmem + TM_DV, mdesc(sb + DO, kk, 8192), mdesc(sb + AM3 + t * 8192, kk, 8192),
                           ID | tc::kIdescAMajorMN | tc::kIdescBMajorMN, (t | kk) ? 1u : 0u);
        tc::mma_commit(bar);
    }
    if (ok)
        wait_mma();

    // ---- a state tile [128 keys][128 v] fp32 (this chunk's slot in the workspace) -> key-scaled, three bf16
    //      terms over the q~ / AM / BM space (free now)
    const size_t tile = ((size_t)j * H + h) * KD * KD;
    auto split_state = [&](const float *src, const float *f) {
        for (int e = tid; e < KD * 16; e += NT) {
            const int key = e >> 4, c = e & 15;
            const float4 x0 = __ldcg(reinterpret_cast<const float4 *>(src + tile + (size_t)key * KD + 8 * c));
            const float4 x1 = __ldcg(reinterpret_cast<const float4 *>(src + tile + (size_t)key * KD + 8 * c + 4));
            const float fk = f[key];
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
        tc::fence_proxy_async();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
    };
    if (ok) {
        split_state(a.dS, FA);   // S' = scale 2^(G_a) S_c
        if (tid == 0) {
            for (int t = 0; t < 3; ++t)
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_ss(tmem + TM_DQ, kdesc(sb + ST3 + t * 32768, kk, 16384), kdesc(sb + DO, kk, 8192), ID, 1u);
            tc::mma_commit(bar);
        }
        wait_mma();
    }
    if (ok) {
        split_state(a.dR, FR);   // R' = 2^(G_l - G_a) R_c
        if (tid == 0) {
            for (int t = 0; t < 3; ++t)
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_ss(tmem + TM_DK, kdesc(sb + ST3 + t * 32768, kk, 16384), kdesc(sb + VV, kk, 8192), ID, 1u);
            for (int p = 0; p < 6; ++p)
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_ss(tmem + TM_DV, mdesc(sb + ST3 + PA[p] * 32768, kk, 16384),
                               kdesc(sb + K3 + PB[p] * 16384, kk, 8192), ID | tc::kIdescAMajorMN, 1u);
            tc::mma_commit(bar);
        }
        wait_mma();
    }

    // ---- epilogue.  Warp w owns TMEM lanes 32 (w % 4) .. + 31 (keys for dq^T, dk^T; value columns for dv^T)
    //      and rows 32 (w / 4) .. + 31 of the chunk.
    if (ok) {
        const int k = 32 * (warp & 3) + lane, half = warp >> 2, r0 = 32 * half;
        const uint32_t lrow = (uint32_t)(32 * (warp & 3)) << 16;
        const unsigned short *rq = reinterpret_cast<const unsigned short *>(sm + RQ);
        const unsigned short *rk = reinterpret_cast<const unsigned short *>(sm + RK);
        const unsigned short *rg = reinterpret_cast<const unsigned short *>(sm + RG);
        // this key's cumsum (log2) up to row 31 (the anchor) and up to the row before this warp's rows
        float ga = 0.f, pre = 0.f;
        for (int t = 0; t < CT / 2; ++t)
            ga += t < len ? bf(rg + t * KD + k) * L2E : 0.f;
        pre = half ? ga : 0.f;
        uint32_t aq[32], ak[32];
        tc::tmem_ld32(tmem + lrow + TM_DQ + r0, aq);
        tc::tmem_ld32(tmem + lrow + TM_DK + r0, ak);
        tc::tmem_wait_ld(aq);
        tc::tmem_wait_ld(ak);
        float pd[32];
        float G = pre;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int t = r0 + u;
            const bool in = t < len;
            G += in ? bf(rg + t * KD + k) * L2E : 0.f;
            const float dq = tc::ex2(G - ga) * __uint_as_float(aq[u]);
            const float dk = tc::ex2(ga - G) * __uint_as_float(ak[u]);
            pd[u] = in ? bf(rq + t * KD + k) * dq - bf(rk + t * KD + k) * dk : 0.f;
            if (in) {
                const size_t row = rb + (size_t)t * rs;
                a.dq[row * KD + k] = dq;
                a.dk[row * KD + k] = dk;
            }
        }
        uint32_t av[32];
        tc::tmem_ld32(tmem + lrow + TM_DV + r0, av);
        tc::tmem_wait_ld(av);
#pragma unroll
        for (int u = 0; u < 32; ++u)
            if (r0 + u < len)
                a.dv[(rb + (size_t)(r0 + u) * rs) * KD + k] = __uint_as_float(av[u]);
        // suffix sums of q dq - k dk over the rows: the later rows' warps first, their totals to FA's place
        float run = 0.f;
        if (half) {
#pragma unroll
            for (int u = 31; u >= 0; --u) {
                run += pd[u];
                if (r0 + u < len)
                    a.dg[(rb + (size_t)(r0 + u) * rs) * KD + k] = run;
            }
        }
        __syncthreads();   // every thread of the CTA reaches this barrier (ok is uniform)
        if (half)
            FA[k] = run;
        __syncthreads();
        if (!half) {
            run = FA[k];
#pragma unroll
            for (int u = 31; u >= 0; --u) {
                run += pd[u];
                if (u < len)
                    a.dg[(rb + (size_t)u * rs) * KD + k] = run;
            }
            a.dgt[((size_t)j * H + h) * KD + k] = run;
        }
    } else if (tid == 0) {
        report(a.status, GLA_ERR_TIMEOUT);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
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
    static std::atomic<uint64_t> ready{0};   // per-device shared-memory opt-in, done once
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (!(ready.load(std::memory_order_acquire) & (1ull << (dev & 63)))) {
        if ((e = cudaFuncSetAttribute(bwd_grads_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)) !=
            cudaSuccess)
            return e;
        ready.fetch_or(1ull << (dev & 63), std::memory_order_release);
    }
    bwd_grads_tc<<<dim3(J, a.H), NT, SMEM_BYTES, s>>>(a);
    return cudaGetLastError();
}

}  // namespace gla
