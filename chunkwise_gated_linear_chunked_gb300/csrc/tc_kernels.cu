// Tensor-core (tcgen05) kernels of the chunkwise GLA forward for bf16 inputs, K = 128, V a multiple of 128.
//
// Method (page "fla/ops/gla/fused_chunk.py"): per chunk of C = 64 rows with chunk-local cumsum G of the
// gates (FusedChunkGLAFunction.forward, kernel a), the state contribution (k*exp(G_last-G))^T V
// (prepare_qg_kg, fused_chunk_gla_fwd_kernel: kernel b), and the output = inter-chunk term (q*exp(G)) S plus
// the causally masked intra-chunk term with the inclusive diagonal (fwd_inner_chunk, the A @ v product of
// FusedChunkGLAFunction.forward: kernel d), with scale applied to the sum.
//
// One CTA owns one (segment, head, 128-wide value tile).  The K x V state lives in TMEM transposed
// (lane = value column v, column = key dimension), so every MMA has M = 128:
//   (a) O^T  = S'^T  q~^T      A = S' from TMEM (fp16),        B = q~  [t][key]   (K-major, smem)
//   (b) P    = q~    k~^T      A = q~ (rows 64..127 unused),   B = k~  [s][key]   (K-major, smem)
//   (c) S^T += V^T   k^^T     A = V^T [v][t]  (K-major, smem), B = k^^T [key][t] (K-major, smem)
//   (d) O^T += V^T   P^T      A = V^T [v][s],                  B = P   [t][s]     (K-major, smem)
// with q~ = q*exp(G-G_a), k~ = k*exp(G_a-G), k^ = k*exp(G_last-G), S' = diag(exp(G_a)) S, the anchor a in
// the middle of the chunk.  Operands are fp16 (bf16 inputs widen exactly; 11-bit significands keep the
// result within the parity bounds where single-rounded bf16 operands do not), accumulation is fp32 in TMEM.
//
// Roles: warps 0-3 (128 threads) form the compute group — in the gating pass thread i owns key column i
// (and value column i), elsewhere thread i owns TMEM lane i; warp 4 lane 0 issues the TMA loads (two raw
// stages of q, k, g, v tiles) and the MMAs.  Every mbarrier wait is bounded; on timeout the kernel records
// GLA_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "gla_internal.h"
#include "tc_ptx.cuh"

namespace gla {
namespace {

using namespace tc;

constexpr int C = 64;            // chunk rows
constexpr int KD = 128;          // key dimension handled by this path
constexpr int VT = 128;          // value tile = TMEM lanes
constexpr int NCOMP = 128;       // compute threads
constexpr int NTHREADS = NCOMP + 32;
constexpr float L2E = 1.4426950408889634f;

// shared memory (byte offsets from a 1024-aligned base)
constexpr int RAW_TILE = C * 128 * 2;          // one [64][128] bf16 tile
constexpr int RAW_STAGE = 4 * RAW_TILE;        // q, k, g, v
constexpr int OFF_RAW = 0;                     // two stages
constexpr int OFF_QK = 2 * RAW_STAGE;          // [q~ kb0 | k~ kb0 | q~ kb1 | k~ kb1], 8 KB each
constexpr int OFF_KH = OFF_QK + 32768;         // k^^T [key][t]
constexpr int OFF_VT = OFF_KH + 16384;         // V^T  [v][t]
constexpr int OFF_P = OFF_VT + 16384;          // P    [t][s]
constexpr int OFF_EG = OFF_P + 8192;           // exp(G_a)[128], exp(G_last)[128]
constexpr int OFF_BAR = OFF_EG + 1024;         // mbarriers + TMEM address slot
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;

// TMEM columns (fp32 unless noted)
constexpr uint32_t TM_S = 0;      // S^T accumulator: 128 columns (key)
constexpr uint32_t TM_SOP = 128;  // S'^T fp16 operand: 64 columns (key pairs)
constexpr uint32_t TM_O = 192;    // O^T: 64 columns (t)
constexpr uint32_t TM_P = 256;    // P: 64 columns (s), lanes t
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t ID_N64 = idesc_f16_f32(128, 64);
constexpr uint32_t ID_N128 = idesc_f16_f32(128, 128);

__device__ __forceinline__ float bf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <typename T>
__device__ __forceinline__ T to_out(float x);
template <>
__device__ __forceinline__ float to_out<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ void named_sync_compute() { asm volatile("bar.sync 1, %0;" ::"n"(NCOMP) : "memory"); }

template <bool OUT, typename Tout>
__global__ void __launch_bounds__(NTHREADS, 1)
    gla_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_v, Args a,
           int multi)
{
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *raw_full = bars + 0, *raw_empty = bars + 2, *ops_ready = bars + 4, *p_ready = bars + 5;
    uint64_t *mma1 = bars + 6, *mma2 = bars + 7, *fin = bars + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 10);
    float *eGa = reinterpret_cast<float *>(sm + OFF_EG), *eGl = eGa + 128;

    const int vt = blockIdx.x, h = blockIdx.y, j = blockIdx.z;
    int n, p, bos, eos, send;
    if (!resolve_slot(a, j, n, p, bos, eos, send))
        return;
    if (!OUT && eos == send)
        return;   // state contributions are needed for non-final segments only
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, V = a.V, v0 = vt * VT;
    const int nchunks = (eos - bos + C - 1) / C;

    if (warp == 0)
        tmem_alloc(tmem_slot, TM_COLS);
    if (tid == NCOMP) {
        bar_init(&raw_full[0], 1);
        bar_init(&raw_full[1], 1);
        bar_init(&raw_empty[0], NCOMP);
        bar_init(&raw_empty[1], NCOMP);
        bar_init(ops_ready, NCOMP);
        bar_init(p_ready, NCOMP);
        bar_init(mma1, 1);
        bar_init(mma2, 1);
        bar_init(fin, 1);
        bar_fence_init();
        if (OUT)
            tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_g);
        tma_prefetch_desc(&tm_v);
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ------------------------------------------------------------ control: TMA + MMA issue
        if (lane == 0) {
            bool ok = true;
            constexpr uint32_t tx = (OUT ? 4 : 3) * RAW_TILE;
            int last_issued[2] = {-1, -1};
            auto issue = [&](int c) {
                const int s = c & 1;
                uint8_t *st = sm + OFF_RAW + s * RAW_STAGE;
                const int row0 = bos + c * C;
                bar_expect_tx(&raw_full[s], tx);
                if (OUT)
                    tma_load_3d(st, &tm_q, 0, h, row0, &raw_full[s]);
                tma_load_3d(st + RAW_TILE, &tm_k, 0, h, row0, &raw_full[s]);
                tma_load_3d(st + 2 * RAW_TILE, &tm_g, 0, h, row0, &raw_full[s]);
                tma_load_3d(st + 3 * RAW_TILE, &tm_v, v0, h, row0, &raw_full[s]);
                last_issued[s] = c;
            };
            if (nchunks > 0)
                issue(0);
            if (nchunks > 1)
                issue(1);
            const uint32_t qk = smem_u32(sm + OFF_QK), kh = smem_u32(sm + OFF_KH);
            const uint32_t vtile = smem_u32(sm + OFF_VT), pt = smem_u32(sm + OFF_P);
            for (int c = 0; c < nchunks; ++c) {
                const uint32_t ph = c & 1;
                if (!(ok = bar_wait(ops_ready, ph)))
                    break;
                fence_after();
                if (OUT) {
                    // (a) O^T = S'^T q~^T : A = S' (TMEM), B = q~ rows t, K = key
                    for (int k = 0; k < KD / 16; ++k)
                        mma_ts(tmem + TM_O, tmem + TM_SOP + k * 8,
                               sdesc_sw128(qk + (k >> 2) * 16384 + (k & 3) * 32), ID_N64, k > 0);
                    // (b) P = q~ k~^T : A = q~ (128-row view), B = k~ rows s
                    for (int k = 0; k < KD / 16; ++k)
                        mma_ss(tmem + TM_P, sdesc_sw128(qk + (k >> 2) * 16384 + (k & 3) * 32),
                               sdesc_sw128(qk + (k >> 2) * 16384 + 8192 + (k & 3) * 32), ID_N64, k > 0);
                }
                // (c) S^T += V^T k^^T : K = t
                for (int k = 0; k < C / 16; ++k)
                    mma_ss(tmem + TM_S, sdesc_sw128(vtile + k * 32), sdesc_sw128(kh + k * 32), ID_N128, 1);
                mma_commit(mma1);
                if (c + 2 < nchunks) {
                    if (!(ok = bar_wait(&raw_empty[c & 1], (c >> 1) & 1)))
                        break;
                    issue(c + 2);
                }
                if (OUT) {
                    if (!(ok = bar_wait(p_ready, ph)))
                        break;
                    fence_after();
                    // (d) O^T += V^T P^T : K = s
                    for (int k = 0; k < C / 16; ++k)
                        mma_ss(tmem + TM_O, sdesc_sw128(vtile + k * 32), sdesc_sw128(pt + k * 32), ID_N64, 1);
                }
                mma_commit(mma2);
            }
            // drain: every MMA issued by this thread, and the last copy into each raw stage
            mma_commit(fin);
            bool drained = bar_wait(fin, 0);
            for (int s = 0; s < 2; ++s)
                if (last_issued[s] >= 0)
                    drained &= bar_wait(&raw_full[s], (last_issued[s] >> 1) & 1);
            if (!ok || !drained)
                report(a.status, GLA_ERR_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ compute group (128 threads)
        const int i = tid;
        const uint32_t lrow = static_cast<uint32_t>(warp * 32) << 16;   // this warp's TMEM lane quarter
        bool ok = true;
        float amax = 0.f;   // largest magnitude converted to an fp16 operand
        float gsum = 0.f;   // total log-decay of the segment for key i (state pass)

        // initial state -> TMEM (thread = lane v); S^T[v][key] = S[key][v]
        {
            const float *src = nullptr;
            if (OUT)
                src = multi ? a.ss + ((size_t)j * H + h) * KD * V
                            : (a.h0 ? a.h0 + ((size_t)n * H + h) * KD * V : nullptr);
            for (int kc = 0; kc < KD / 32; ++kc) {
                uint32_t r[32];
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    r[u] = __float_as_uint(src ? __ldg(src + (size_t)(kc * 32 + u) * V + v0 + i) : 0.f);
                tmem_st32(tmem + lrow + TM_S + kc * 32, r);
            }
            tmem_wait_st();
        }

        for (int c = 0; c < nchunks; ++c) {
            const int s = c & 1;
            const uint32_t ph = c & 1;
            const int row0 = bos + c * C;
            const int len = min(C, eos - row0);
            const uint8_t *st = sm + OFF_RAW + s * RAW_STAGE;
            const __nv_bfloat16 *rq = reinterpret_cast<const __nv_bfloat16 *>(st);
            const __nv_bfloat16 *rk = rq + C * 128, *rg = rk + C * 128, *rv = rg + C * 128;
            if (!(ok = bar_wait(&raw_full[s], (c >> 1) & 1)))
                break;

            // pass 1: chunk-local cumsum of column i -> G at the anchor and at the last valid row
            const int ra = min(C / 2 - 1, len - 1);
            float G = 0.f, Ga = 0.f;
            for (int t = 0; t < len; ++t) {
                G += bf(rg + t * 128 + i);
                if (t == ra)
                    Ga = G;
            }
            const float Gl = G;
            gsum += Gl;
            // the previous chunk's MMAs must be done before its operand buffers are overwritten
            if (c > 0 && !(ok = bar_wait(mma2, (c - 1) & 1)))
                break;

            // pass 2: gated operands (thread i = key column i; value column i for V^T)
            const float cl = exp2f((Gl - Ga) * L2E);
            G = 0.f;
            uint8_t *qk = sm + OFF_QK + (i >> 6) * 16384;
            const int ic = i & 63;
#pragma unroll 1
            for (int t0 = 0; t0 < C; t0 += 8) {
                uint32_t khp[4], vp[4];
#pragma unroll
                for (int u = 0; u < 8; u += 2) {
                    float kh2[2], vv2[2];
#pragma unroll
                    for (int w = 0; w < 2; ++w) {
                        const int t = t0 + u + w;
                        float qt = 0.f, kt = 0.f, kk = 0.f, vv = 0.f;
                        if (t < len) {
                            G += bf(rg + t * 128 + i);
                            const float kv = bf(rk + t * 128 + i);
                            vv = bf(rv + t * 128 + i);
                            if (OUT) {
                                const float qv = bf(rq + t * 128 + i);
                                qt = qv * exp2f((G - Ga) * L2E);
                                kt = kv * exp2f((Ga - G) * L2E);
                                kk = kt * cl;
                            } else {
                                kk = kv * exp2f((Gl - G) * L2E);
                            }
                        }
                        if (OUT) {
                            *reinterpret_cast<__half *>(qk + sw128(t, ic)) = __float2half_rn(qt);
                            *reinterpret_cast<__half *>(qk + 8192 + sw128(t, ic)) = __float2half_rn(kt);
                            amax = fmaxf(amax, fmaxf(fabsf(qt), fabsf(kt)));
                        }
                        amax = fmaxf(amax, fmaxf(fabsf(kk), fabsf(vv)));
                        kh2[w] = kk;
                        vv2[w] = vv;
                    }
                    khp[u / 2] = pack_h2(kh2[0], kh2[1]);
                    vp[u / 2] = pack_h2(vv2[0], vv2[1]);
                }
                *reinterpret_cast<uint4 *>(sm + OFF_KH + sw128(i, t0)) = make_uint4(khp[0], khp[1], khp[2], khp[3]);
                *reinterpret_cast<uint4 *>(sm + OFF_VT + sw128(i, t0)) = make_uint4(vp[0], vp[1], vp[2], vp[3]);
            }
            eGa[i] = exp2f(Ga * L2E);
            eGl[i] = exp2f(Gl * L2E);
            fence_proxy_async();
            bar_arrive(&raw_empty[s]);
            named_sync_compute();   // eGa / eGl complete

            // state: S' = diag(exp(G_a)) S (fp16 operand), S <- diag(exp(G_last)) S (thread = lane v)
            for (int kc = 0; kc < KD / 32; ++kc) {
                uint32_t r[32];
                tmem_ld32(tmem + lrow + TM_S + kc * 32, r);
                tmem_wait_ld();
                if (OUT) {
                    uint32_t op[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const float s0 = __uint_as_float(r[2 * u]) * eGa[kc * 32 + 2 * u];
                        const float s1 = __uint_as_float(r[2 * u + 1]) * eGa[kc * 32 + 2 * u + 1];
                        amax = fmaxf(amax, fmaxf(fabsf(s0), fabsf(s1)));
                        op[u] = pack_h2(s0, s1);
                    }
                    tmem_st16(tmem + lrow + TM_SOP + kc * 16, op);
                }
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    r[u] = __float_as_uint(__uint_as_float(r[u]) * eGl[kc * 32 + u]);
                tmem_st32(tmem + lrow + TM_S + kc * 32, r);
            }
            tmem_wait_st();
            fence_before();
            bar_arrive(ops_ready);

            if (OUT) {
                // masked scores -> fp16 P[t][s] (thread = lane t, t < 64)
                if (!(ok = bar_wait(mma1, ph)))
                    break;
                fence_after();
                if (warp < 2) {
                    const int t = i;
                    for (int sc = 0; sc < 2; ++sc) {
                        uint32_t r[32];
                        tmem_ld32(tmem + lrow + TM_P + sc * 32, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int u0 = 0; u0 < 32; u0 += 8) {
                            uint32_t pk[4];
#pragma unroll
                            for (int u = 0; u < 8; u += 2) {
                                const int sa = sc * 32 + u0 + u;
                                const float p0 = sa <= t ? __uint_as_float(r[u0 + u]) : 0.f;
                                const float p1 = sa + 1 <= t ? __uint_as_float(r[u0 + u + 1]) : 0.f;
                                amax = fmaxf(amax, fmaxf(fabsf(p0), fabsf(p1)));
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

                // output (thread = lane v): o[t, v] = scale * O^T[v][t]
                if (!(ok = bar_wait(mma2, ph)))
                    break;
                fence_after();
                Tout *go = static_cast<Tout *>(a.o);
                for (int oc = 0; oc < 2; ++oc) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lrow + TM_O + oc * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        const int t = oc * 32 + u;
                        if (t < len) {
                            const float val = a.scale * __uint_as_float(r[u]);
                            go[((size_t)(row0 + t) * H + h) * V + v0 + i] = to_out<Tout>(val);
                        }
                    }
                }
                fence_before();
            }
        }

        // final state of the segment: ht (output pass, last segment) or the contribution (state pass)
        if (ok && nchunks > 0)
            ok = bar_wait(mma2, (nchunks - 1) & 1);
        if (ok) {
            fence_after();
            float *dst = nullptr;
            if (OUT)
                dst = (eos == send && a.ht) ? a.ht + ((size_t)n * H + h) * KD * V : nullptr;
            else
                dst = a.ss + ((size_t)j * H + h) * KD * V;
            if (dst) {
                for (int kc = 0; kc < KD / 32; ++kc) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lrow + TM_S + kc * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int u = 0; u < 32; ++u)
                        dst[(size_t)(kc * 32 + u) * V + v0 + i] = __uint_as_float(r[u]);
                }
            }
            if (!OUT && vt == 0)
                a.gtot[((size_t)j * H + h) * KD + i] = gsum;
        }
        if (!ok)
            report(a.status, GLA_ERR_TIMEOUT);
        if (!(amax <= 65000.f))
            report(a.status, GLA_ERR_RANGE);
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

// [rows][H][D] bf16 tensor, box = 128 (inner) x 1 head x 64 rows.
bool encode_rows(CUtensorMap *m, const void *ptr, int D, int H, long long rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {128, 1, (cuuint32_t)C};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool OUT, typename Tout>
cudaError_t launch_one(const Plan &pl, const Args &a, cudaStream_t s)
{
    const long long rows = pl.varlen ? (long long)pl.T : (long long)pl.B * pl.T;
    CUtensorMap mq, mk, mg, mv;
    if (!encode_rows(&mq, a.q, pl.K, pl.H, rows) || !encode_rows(&mk, a.k, pl.K, pl.H, rows) ||
        !encode_rows(&mg, a.g, pl.K, pl.H, rows) || !encode_rows(&mv, a.v, pl.V, pl.H, rows))
        return cudaErrorInvalidValue;
    auto f = gla_tc<OUT, Tout>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess)
            return e;
        attr = true;
    }
    dim3 grid(pl.V / VT, pl.H, pl.J);
    f<<<grid, NTHREADS, SMEM_BYTES, s>>>(mq, mk, mg, mv, a, pl.multi ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(int dtype, int K, int V)
{
    return dtype != GLA_F32 && K == KD && V % VT == 0 && V <= 256;
}

cudaError_t launch_state_tc(const Plan &pl, const Args &a, cudaStream_t s)
{
    return launch_one<false, float>(pl, a, s);
}

cudaError_t launch_out_tc(const Plan &pl, const Args &a, cudaStream_t s)
{
    if (pl.dtype == GLA_BF16_OBF16)
        return launch_one<true, __nv_bfloat16>(pl, a, s);
    return launch_one<true, float>(pl, a, s);
}

}  // namespace gla
