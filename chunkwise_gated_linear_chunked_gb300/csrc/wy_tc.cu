// WY representation forward of the gated delta rule on the tensor cores (bf16 inputs; page
// "fla/ops/gated_delta_rule/backends/triton_ascend/wy_fast.py": recompute_w_u_fwd_kernel_npu):
//     u = A (v * beta),   w = A (k * beta * 2^g)      per chunk of BT rows and value head.
//
// Per work item (chunk, value head) the product is computed transposed, D^T = X^T A^T, with tcgen05
// kind::f16 MMAs (bf16 operands, fp32 accumulation in TMEM):
//   * M = 128 columns of X = [k*beta*2^g | v*beta] per block (K + V = 128 or 256: one or two blocks);
//   * N = BT rows of the chunk;  K = BT (the chunk's columns s), in steps of 16.
// The B operand (N x K, K-major) is A itself: row t of the chunk's matrix is stored contiguously over s, so
// its raw bf16 rows are copied straight into a 128-byte-swizzled tile.  The A operand X^T (M x K, K-major)
// is formed on chip: X is scaled in fp32 and split into two bf16 terms x = x1 + x2 + e, x1 = RN(x),
// x2 = RN(x - x1), |e| <= 2^-18 |x| (within the fp32 outputs' 1e-5 relative bound, since A is exact), each
// written transposed into its own swizzled tile; the two MMA groups accumulate into the same TMEM columns.
// A work item is one 128-column block of one (chunk, value
// head), so that three CTAs (58 KB each) fit on an SM and one's conversion overlaps the others' MMAs and
// stores.  A and the raw k | v columns of the next item arrive by 16-byte asynchronous copies while the
// current item is stored; the epilogue reads D^T from TMEM (lane = column of w or u) and each warp
// stores 32 consecutive columns of a row per instruction.
//
// Persistent: three CTAs per SM walk the items blockIdx.x, blockIdx.x + gridDim.x, ...  Rows past the end of a
// sequence: X^T is zero there (so A's columns for them contribute nothing) and their outputs are not stored.
#include <atomic>

#include "gla_internal.h"
#include "io.cuh"
#include "tc_ptx.cuh"

namespace gla {

namespace {

constexpr int NTC = 256;   // threads per CTA (8 warps)

template <int BT, int KV>
struct WyTcSmem {
    static constexpr int NBLK = KV / 128;                      // 128-column blocks of X (one per work item)
    static constexpr int XT_TILE = 128 * 128;                  // bytes: 128 rows (columns of X) x 64 s slots
    static constexpr int A_TILE = BT * 128;                    // bytes: BT rows (t) x 64 s slots
    static constexpr int A_STRIDE = (A_TILE + 1023) / 1024 * 1024;
    static constexpr int XT = 0;                               // [2 terms] X^T tiles of the block (1024-aligned)
    static constexpr int AB = XT + 2 * XT_TILE;                // A tile (B operand)
    static constexpr int RAW = AB + A_STRIDE;                  // [BT][128] raw columns of the block (bf16)
    static constexpr int F = RAW + BT * 128 * 2;               // [2][BT] row factors (k part, v part)
    static constexpr int BAR = F + 2 * BT * 4;                 // mbarrier (MMA done)
    static constexpr int TSLOT = BAR + 8;                      // TMEM base address
    static constexpr int BYTES = TSLOT + 8;
    static constexpr int TCOLS = BT <= 32 ? 32 : 64;
};

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 accumulation, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T>
__device__ __forceinline__ T to_out_tc(float x);
template <>
__device__ __forceinline__ float to_out_tc<float>(float x)
{
    return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 to_out_tc<__nv_bfloat16>(float x)
{
    return __float2bfloat16_rn(x);
}

// Resolve work item `it` = ((chunk slot j, value head hv), column block cb) to (cb, hv, first row, valid
// rows); false if it has no rows.
__device__ __forceinline__ bool wy_item(const WyArgs &a, int it, int BT, int nblk, int &cb, int &hv, int &bos,
                                        int &m)
{
    const int jh = it / nblk;
    cb = it - jh * nblk;
    const int j = jh / a.HV;
    hv = jh - j * a.HV;
    int eos;
    if (a.table) {
        const int4 e = a.table[j];
        if (e.x < 0)
            return false;
        bos = e.z;
        eos = e.w;
    } else {
        const int n = j / a.NT, p = j - n * a.NT;
        bos = n * a.T + p * BT;
        eos = min(bos + BT, n * a.T + a.T);
    }
    m = eos - bos;
    return m > 0;
}

template <typename Tout, int BT, int K, int V>
__global__ void __launch_bounds__(NTC, 3) wy_fwd_tc(WyArgs a, int items)
{
    constexpr int KV = K + V;
    using L = WyTcSmem<BT, KV>;
    constexpr int NBLK = L::NBLK, CPR = BT / 8;   // 16-byte chunks per row of A
    extern __shared__ __align__(16) unsigned char smraw[];
    // swizzled tiles need 1024-byte alignment: the launch adds 1024 bytes of slack for this offset
    unsigned char *sm = smraw + ((1024u - (tc::smem_u32(smraw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + L::TSLOT);
    float *F = reinterpret_cast<float *>(sm + L::F);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const __nv_bfloat16 *A = static_cast<const __nv_bfloat16 *>(a.A);
    const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(a.beta);
    const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(a.k);
    const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(a.v);
    const int HV = a.HV;
    if (tid == 0) {
        tc::bar_init(bar, 1);
        tc::bar_fence_init();
    }
    if (warp == 0)
        tc::tmem_alloc(tslot, L::TCOLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;

    // ---- asynchronous copies of item `it` into buffer `b`: A's valid rows into the swizzled B tile, the
    //      k | v rows into the raw buffer (one commit group per item, even when it has no rows)
    auto copy_item = [&](int it) {
        int cb, hv, bos, m;
        if (it < items && wy_item(a, it, BT, NBLK, cb, hv, bos, m)) {
            const int hk = hv / (HV / a.H);
            unsigned char *at = sm + L::AB;
            for (int e = tid; e < BT * CPR; e += NTC) {
                const int t = e / CPR, c = e - t * CPR;
                if (t < m)
                    cp_async16(at + tc::sw128(t, 8 * c), A + ((size_t)(bos + t) * HV + hv) * BT + 8 * c);
            }
            __nv_bfloat16 *raw = reinterpret_cast<__nv_bfloat16 *>(sm + L::RAW);
            for (int e = tid; e < BT * 16; e += NTC) {   // 16 copies of 8 columns per row of the block
                const int s = e >> 4, cg = cb * 128 + 8 * (e & 15);
                if (s < m) {
                    const size_t row = (size_t)(bos + s);
                    cp_async16(raw + s * 128 + 8 * (e & 15),
                               cg < K ? k + (row * a.H + hk) * K + cg : v + (row * HV + hv) * V + (cg - K));
                }
            }
        }
        cp_commit();
    };
    // row factors of item `it` (plain loads; threads < BT)
    auto load_factors = [&](int it, float &fk, float &fv) {
        fk = fv = 0.f;
        int cb, hv, bos, m;
        if (tid < BT && it < items && wy_item(a, it, BT, NBLK, cb, hv, bos, m) && tid < m) {
            const size_t row = (size_t)(bos + tid);
            fv = __bfloat162float(beta[row * HV + hv]);
            fk = a.g ? fv * exp2f(a.g[row * HV + hv]) : fv;
        }
    };

    const int first = blockIdx.x, step = gridDim.x;
    copy_item(first);
    float fk, fv;
    load_factors(first, fk, fv);
    if (tid < BT) {
        F[tid] = fk;
        F[BT + tid] = fv;
    }
    volatile int abort_flag = 0;
    int n = 0;
    for (int it = first; it < items; it += step, ++n) {
        float nfk, nfv;
        load_factors(it + step, nfk, nfv);   // the next item's factors, used after this item
        cp_wait<0>();                        // this item's copies
        __syncthreads();
        int cb, hv, bos, m;
        const bool live = wy_item(a, it, BT, NBLK, cb, hv, bos, m);
        if (live) {
            // ---- X^T terms: task (column c, s-group j of 8 rows); lanes take consecutive columns
            const __nv_bfloat16 *raw = reinterpret_cast<const __nv_bfloat16 *>(sm + L::RAW);
            const float *Fb = F;
            for (int e = tid; e < 128 * CPR; e += NTC) {
                const int j = e >> 7, c = e & 127;
                const float *fr = Fb + (cb * 128 + c < K ? 0 : BT);
                uint32_t p1[4], p2[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {   // rows s0, s0 + 1 of the group, two at a time
                    const int s0 = 8 * j + 2 * q;
                    const float2 x = make_float2(s0 < m ? __bfloat162float(raw[s0 * 128 + c]) * fr[s0] : 0.f,
                                                 s0 + 1 < m ? __bfloat162float(raw[(s0 + 1) * 128 + c]) * fr[s0 + 1] : 0.f);
                    const __nv_bfloat162 x1 = __float22bfloat162_rn(x);
                    const float2 y1 = __bfloat1622float2(x1);
                    const __nv_bfloat162 x2 = __float22bfloat162_rn(make_float2(x.x - y1.x, x.y - y1.y));
                    p1[q] = *reinterpret_cast<const uint32_t *>(&x1);
                    p2[q] = *reinterpret_cast<const uint32_t *>(&x2);
                }
                const uint32_t off = tc::sw128(c, 8 * j);
                *reinterpret_cast<uint4 *>(sm + L::XT + 0 * L::XT_TILE + off) = make_uint4(p1[0], p1[1], p1[2], p1[3]);
                *reinterpret_cast<uint4 *>(sm + L::XT + 1 * L::XT_TILE + off) = make_uint4(p2[0], p2[1], p2[2], p2[3]);
            }
            tc::fence_proxy_async();   // generic-proxy writes of the tiles -> visible to the MMAs
        }
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        if (live && tid == 0) {
            const uint32_t at = tc::smem_u32(sm + L::AB);
            constexpr uint32_t idesc = idesc_bf16_f32(128, BT);
#pragma unroll
            for (int term = 0; term < 2; ++term)
#pragma unroll
                for (int ks = 0; ks < BT / 16; ++ks) {
                    const uint32_t xa = tc::smem_u32(sm + L::XT + term * L::XT_TILE) + 32 * ks;
                    tc::mma_ss(tmem, tc::sdesc_sw128(xa), tc::sdesc_sw128(at + 32 * ks), idesc, (term | ks) ? 1u : 0u);
                }
            tc::mma_commit(bar);
        }
        if (live && !tc::bar_wait(bar, n & 1)) {   // bounded: 1 s
            if (tid == 0)
                report(a.status, GLA_ERR_TIMEOUT);
            abort_flag = 1;
        }
        if (!live && tid == 0)
            tc::mma_commit(bar);   // keep one phase per item (no MMAs issued: arrives at once)
        if (!live && !tc::bar_wait(bar, n & 1))
            abort_flag = 1;
        tc::fence_after();
        // the MMAs no longer read the A tile and the conversion is done with the raw rows: fetch the next
        // item while this one is stored (and the SM's other CTAs work)
        __syncthreads();
        copy_item(it + step);
        if (tid < BT) {   // factors of the next item
            F[tid] = nfk;
            F[BT + tid] = nfv;
        }
        // ---- epilogue: lane = column of the block; warp group g = warp / 4 takes the 32-row chunks g, g + 2,
        //      ...; a warp stores 32 consecutive columns of one row per instruction
        if (live && !abort_flag) {
            constexpr int TL = BT < 32 ? BT : 32, NT = BT / TL;
            Tout *w = static_cast<Tout *>(a.w), *u = static_cast<Tout *>(a.u);
            const int c = cb * 128 + 32 * (warp & 3) + lane;
            Tout *dst = c < K ? w + (size_t)hv * K + c : u + (size_t)hv * V + (c - K);
            const size_t rstride = (size_t)HV * (c < K ? K : V);
            for (int task = warp >> 2; task < NT; task += 2) {
                const int t0 = task * TL;
                const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)t0;
                uint32_t r[32];
                if constexpr (TL == 32) {
                    tc::tmem_ld32(taddr, r);
                    tc::tmem_wait_ld(r);
                } else {
                    uint32_t r16[16];
                    tc::tmem_ld16(taddr, r16);
                    tc::tmem_wait_ld(r16);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        r[i] = r16[i];
                }
#pragma unroll
                for (int i = 0; i < TL; ++i)
                    if (t0 + i < m)
                        dst[(size_t)(bos + t0 + i) * rstride] = to_out_tc<Tout>(__uint_as_float(r[i]));
            }
        }
        tc::fence_before();
    }
    cp_wait<0>();
    __syncthreads();
    tc::fence_after();
    if (warp == 0)
        tc::tmem_dealloc(tmem, L::TCOLS);
}

template <typename Tout, int BT, int K, int V>
cudaError_t launch_tc_t(const WyArgs &a, int J, cudaStream_t s)
{
    using L = WyTcSmem<BT, K + V>;
    auto f = wy_fwd_tc<Tout, BT, K, V>;
    const size_t bytes = L::BYTES + 1024;
    // per-device one-time setup (shared-memory opt-in, SM count); repeating it is harmless
    static std::atomic<uint64_t> ready{0};
    static int sm_count[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(ready.load(std::memory_order_acquire) & bit)) {
        if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sm_count[dev & 63], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        ready.fetch_or(bit, std::memory_order_release);
    }
    const int sms = sm_count[dev & 63];
    const int items = J * a.HV * L::NBLK;
    const int grid = items < 3 * sms ? items : 3 * sms;   // three CTAs per SM
    f<<<grid, NTC, bytes, s>>>(a, items);
    return cudaGetLastError();
}

template <typename Tout, int BT>
cudaError_t launch_tc_bt(const WyArgs &a, int J, cudaStream_t s)
{
    if (a.K == 64)
        return launch_tc_t<Tout, BT, 64, 64>(a, J, s);
    return launch_tc_t<Tout, BT, 128, 128>(a, J, s);
}

template <typename Tout>
cudaError_t launch_tc_out(const WyArgs &a, int J, cudaStream_t s)
{
    if (a.BT == 16)
        return launch_tc_bt<Tout, 16>(a, J, s);
    if (a.BT == 32)
        return launch_tc_bt<Tout, 32>(a, J, s);
    return launch_tc_bt<Tout, 64>(a, J, s);
}

}  // namespace

bool wy_tc_supported(int dtype, int K, int V)
{
    return (dtype == GLA_BF16 || dtype == GLA_BF16_OBF16) && K == V && (K == 64 || K == 128);
}

cudaError_t launch_wy_fwd_tc(const WyArgs &a, int J, int dtype, cudaStream_t s)
{
    if (dtype == GLA_BF16_OBF16)
        return launch_tc_out<__nv_bfloat16>(a, J, s);
    return launch_tc_out<float>(a, J, s);
}

}  // namespace gla
