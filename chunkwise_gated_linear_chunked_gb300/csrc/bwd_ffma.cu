// CUDA-core (fp32) kernels of the chunkwise GLA backward.
//
// Method (page "fla/ops/gla/fused_chunk.py": fused_chunk_gla_bwd_kernel, bwd_inner_chunk and
// FusedChunkGLAFunction.backward).  Per chunk c of C = 64 rows with chunk-local inclusive cumsum G of the
// gates (natural log), G_l its last valid row and the loss L = sum(o * do) + sum(ht * dht):
//
//   chunk-start state     S_c      (forward: S_{c+1} = diag(e^{G_l}) S_c + sum_j (k_j e^{G_l - G_j})^T v_j,
//                                   S_0 = h0)
//   chunk-end adjoint     R_c      (reverse: R_{c-1} = diag(e^{G_l}) R_c + scale sum_i (q_i e^{G_i})^T do_i,
//                                   R_last = dht, dh0 = R_{-1})
//   dq_i = scale e^{G_i} (S_c do_i^T) + scale sum_{j<=i} (do_i . v_j) k_j e^{G_i - G_j}
//   dk_j = e^{G_l - G_j} (R_c v_j^T) + scale sum_{i>=j} (do_i . v_j) q_i e^{G_i - G_j}
//   dv_j = (k_j e^{G_l - G_j}) R_c + scale sum_{i>=j} (q_i k_j e^{G_i - G_j} summed over keys) do_i
//   dg_t = sum_{s>=t} (q_s dq_s - k_s dk_s) + sum_v ht dht        (reverse cumsum over the sequence)
//
// The pairwise e^{G_i - G_j} is factorised around the anchor row a = 31 (q~ = q e^{G - G_a},
// k~ = k e^{G_a - G}), which makes q dq = q~ acc and k dk = k~ acc for the kernels' accumulators: the
// gate-gradient terms need no further exponentials.  Launch sequence: [varlen: chunk table] ->
// bwd_chunk_sums (per chunk: dS, dR, G_l) -> bwd_scan (S_c, R_c, ht, dh0) -> bwd_grads (dq, dk, dv, chunk-
// local suffix sums of q dq - k dk) -> bwd_dg_scan (carry over chunks) -> bwd_dg_add.
#include "gla_internal.h"
#include "io.cuh"

namespace gla {

namespace {

constexpr int C = kChunk;   // 64
constexpr int NTB = 256;    // threads per CTA
constexpr int AROW = 31;    // anchor row of the factorisation

// Store four floats, or add them to what is there (a later value slice of the same gradient).
__device__ __forceinline__ void put4(float *p, float4 x, int acc)
{
    if (acc) {
        const float4 o = *reinterpret_cast<const float4 *>(p);
        x.x += o.x;
        x.y += o.y;
        x.z += o.z;
        x.w += o.w;
    }
    *reinterpret_cast<float4 *>(p) = x;
}

__device__ __forceinline__ bool bwd_slot(const BwdArgs &a, int j, int &n, int &bos, int &eos)
{
    if (a.table) {
        const int4 e = a.table[j];
        if (e.x < 0)
            return false;
        n = e.x;
        bos = e.z;
        eos = e.w;
        return true;
    }
    n = j / a.NC;
    const int c = j - n * a.NC;
    bos = n * a.T + c * C;
    eos = min(bos + C, n * a.T + a.T);
    return true;
}

// ------------------------------------------------------------------------------------------------
// per chunk and 64-wide value tile: dS = sum_j (k_j e^{G_l - G_j})^T v_j, dR = scale sum_i (q_i e^{G_i})^T do_i
// ------------------------------------------------------------------------------------------------
template <typename Tin, int K, typename Tg>
__global__ void __launch_bounds__(NTB) bwd_chunk_sums(BwdArgs a)
{
    extern __shared__ float sm[];
    float *QE = sm;              // [C][K] G, then q e^{G}
    float *KL = QE + C * K;      // [C][K] k e^{G_l - G}
    float *VS = KL + C * K;      // [C][64] v tile
    float *DS = VS + C * 64;     // [C][64] do tile
    float *GL = DS + C * 64;     // [K]
    const int j = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * 64, tid = threadIdx.x;
    int n, bos, eos;
    if (!bwd_slot(a, j, n, bos, eos))
        return;
    const int len = eos - bos, H = a.H, V = a.V;
    const size_t rb = row_head(bos, h, H, a.T, a.hf);   // row t of the chunk: row-head index rb + t * rs
    const int rs = a.hf ? 1 : H;
    const Tin *q = static_cast<const Tin *>(a.q), *k = static_cast<const Tin *>(a.k);
    const Tg *g = static_cast<const Tg *>(a.g);
    const Tin *v = static_cast<const Tin *>(a.v);
    const Tin *dout = static_cast<const Tin *>(a.dout);
    if (tid < K) {
        float run = 0.f;
        for (int i = 0; i < C; ++i) {
            run += i < len ? IO<Tg>::load1(g + (rb + (size_t)i * rs) * K + tid) : 0.f;
            QE[i * K + tid] = run;
        }
        GL[tid] = run;
    }
    for (int e = tid; e < C * 16; e += NTB) {
        const int i = e >> 4, c4 = (e & 15) * 4;
        const size_t o = (rb + (size_t)i * rs) * a.ldv + v0 + c4;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(VS + i * 64 + c4) = i < len ? IO<Tin>::load4(v + o) : z;
        *reinterpret_cast<float4 *>(DS + i * 64 + c4) = i < len ? IO<Tin>::load4(dout + o) : z;
    }
    __syncthreads();
    for (int e = tid; e < C * K; e += NTB) {
        const int i = e / K, kk = e - i * K;
        const size_t o = (rb + (size_t)i * rs) * K + kk;
        const float G = QE[e];
        const float qv = i < len ? IO<Tin>::load1(q + o) : 0.f;
        const float kv = i < len ? IO<Tin>::load1(k + o) : 0.f;
        QE[e] = qv * expf(G);
        KL[e] = kv * expf(GL[kk] - G);
    }
    __syncthreads();
    constexpr int R = K / 16;
    const int tx = tid & 15, ty = tid >> 4;
    float aS[R][4], aR[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c)
            aS[r][c] = aR[r][c] = 0.f;
    for (int i = 0; i < C; ++i) {
        const float4 vv = *reinterpret_cast<const float4 *>(VS + i * 64 + 4 * tx);
        const float4 dd = *reinterpret_cast<const float4 *>(DS + i * 64 + 4 * tx);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float kl = KL[i * K + ty * R + r], qe = QE[i * K + ty * R + r];
            aS[r][0] = fmaf(kl, vv.x, aS[r][0]);
            aS[r][1] = fmaf(kl, vv.y, aS[r][1]);
            aS[r][2] = fmaf(kl, vv.z, aS[r][2]);
            aS[r][3] = fmaf(kl, vv.w, aS[r][3]);
            aR[r][0] = fmaf(qe, dd.x, aR[r][0]);
            aR[r][1] = fmaf(qe, dd.y, aR[r][1]);
            aR[r][2] = fmaf(qe, dd.z, aR[r][2]);
            aR[r][3] = fmaf(qe, dd.w, aR[r][3]);
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const size_t o = (((size_t)j * H + h) * K + ty * R + r) * V + v0 + 4 * tx;
        *reinterpret_cast<float4 *>(a.dS + o) = make_float4(aS[r][0], aS[r][1], aS[r][2], aS[r][3]);
        *reinterpret_cast<float4 *>(a.dR + o) =
            make_float4(a.scale * aR[r][0], a.scale * aR[r][1], a.scale * aR[r][2], a.scale * aR[r][3]);
    }
    if (blockIdx.z == 0 && tid < K)
        a.gl[((size_t)j * H + h) * K + tid] = GL[tid];
}

// ------------------------------------------------------------------------------------------------
// per (sequence, head, key, value) element: chunk-start states forward, chunk-end adjoints backward
// ------------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(NTB) bwd_scan(BwdArgs a)
{
    const int e = blockIdx.x * NTB + threadIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int K = a.K, V = a.V, H = a.H;
    if (e >= K * V)
        return;
    const int kk = e / V;
    int first, cnt;
    if (a.seqinfo) {
        const int2 si = a.seqinfo[n];
        first = si.x;
        cnt = si.y;
    } else {
        first = n * a.NC;
        cnt = a.NC;
    }
    const size_t st = ((size_t)n * H + h) * K * V + e;                 // ht in the workspace
    const size_t su = (((size_t)n * H + h) * K + kk) * a.lds + (e - kk * V);   // h0, dht, dh0 of the caller
    const size_t hs = (size_t)H * K * V;                               // slot stride of dS / dR
    float *__restrict__ dS = a.dS + ((size_t)first * H + h) * K * V + e;
    float *__restrict__ dR = a.dR + ((size_t)first * H + h) * K * V + e;
    const float *__restrict__ gl = a.gl + ((size_t)first * H + h) * K + kk;
    const size_t gs = (size_t)H * K;
    // The forward scan (chunk-start states, in place of dS, oldest first) and the backward scan (chunk-end
    // adjoints, in place of dR, newest first) run in the same loop, in batches of D chunks whose loads are
    // all issued before the batch's in-place stores, so both directions' loads overlap.
    constexpr int D = 16;
    float S = a.h0 ? a.h0[su] : 0.f;
    float R = a.dht ? a.dht[su] : 0.f;
    for (int c0 = 0; c0 < cnt; c0 += D) {
        const int c1 = cnt - 1 - c0;   // the backward scan's first chunk of this batch
        float ts[D], es[D], tr[D], er[D];
#pragma unroll
        for (int u = 0; u < D; ++u)
            if (c0 + u < cnt) {
                ts[u] = dS[(size_t)(c0 + u) * hs];
                es[u] = gl[(size_t)(c0 + u) * gs];
                tr[u] = dR[(size_t)(c1 - u) * hs];
                er[u] = gl[(size_t)(c1 - u) * gs];
            }
#pragma unroll
        for (int u = 0; u < D; ++u)
            if (c0 + u < cnt) {
                dS[(size_t)(c0 + u) * hs] = S;
                S = fmaf(expf(es[u]), S, ts[u]);
                dR[(size_t)(c1 - u) * hs] = R;
                R = fmaf(expf(er[u]), R, tr[u]);
            }
    }
    a.ht[st] = S;
    if (a.dh0)
        a.dh0[su] = R;
}

// ------------------------------------------------------------------------------------------------
// per chunk: dq, dk, dv and the chunk-local suffix sums of q dq - k dk
// ------------------------------------------------------------------------------------------------

// 64 x N block product: thread (tx, ty) accumulates rows 4ty .. 4ty+3 and columns {4tx .. 4tx+3} (and
// {64+4tx ..} when N == 128).  A(i, m) is A[i*lda + m], or A[m*lda + i] when A_T (then four rows are one
// float4); B(m, c) is B[m*ldb + c], or, when SWZ (N == 64, a transposed copy written by transpose_swz), the
// float4 group c/4 of row m sits at group (c/4) ^ (m & 7).
template <int N, bool A_T, bool SWZ = false>
__device__ __forceinline__ void mm(float (&acc)[4][N / 16], const float *A, int lda, const float *B, int ldb,
                                   int M, int ty, int tx)
{
    const int i0 = 4 * ty;
#pragma unroll 4
    for (int m = 0; m < M; ++m) {
        float av[4];
        if (A_T) {
            const float4 t = *reinterpret_cast<const float4 *>(A + m * lda + i0);
            av[0] = t.x;
            av[1] = t.y;
            av[2] = t.z;
            av[3] = t.w;
        } else {
#pragma unroll
            for (int r = 0; r < 4; ++r)
                av[r] = A[(i0 + r) * lda + m];
        }
#pragma unroll
        for (int half = 0; half < N / 64; ++half) {
            const int grp = SWZ ? (tx ^ (m & 7)) : tx;
            const float4 b = *reinterpret_cast<const float4 *>(B + m * ldb + 64 * half + 4 * grp);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                acc[r][4 * half + 0] = fmaf(av[r], b.x, acc[r][4 * half + 0]);
                acc[r][4 * half + 1] = fmaf(av[r], b.y, acc[r][4 * half + 1]);
                acc[r][4 * half + 2] = fmaf(av[r], b.z, acc[r][4 * half + 2]);
                acc[r][4 * half + 3] = fmaf(av[r], b.w, acc[r][4 * half + 3]);
            }
        }
    }
}

// dst[r][i] = src[i][r] for i < C rows of src (pitch R) and r < R, dst pitch C, float4 groups of each dst
// row XOR-swizzled by (r & 7): a warp covers 8 consecutive r x 4 consecutive i, so the stores are
// conflict-free (the loads are 4-way).
template <int R>
__device__ __forceinline__ void transpose_swz(float *dst, const float *src)
{
    for (int e = threadIdx.x; e < C * R; e += NTB) {
        const int i4 = e & 3, rlo = (e >> 2) & 7, ihi = (e >> 5) & 15, rhi = e >> 9;
        const int r = rhi * 8 + rlo, i = ihi * 4 + i4;
        dst[r * C + ((ihi ^ rlo) << 2) + i4] = src[i * R + r];
    }
}

template <int N>
__device__ __forceinline__ void zero(float (&acc)[4][N / 16])
{
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < N / 16; ++c)
            acc[r][c] = 0.f;
}

// column of accumulator entry c for thread tx
__device__ __forceinline__ int col_of(int c, int tx) { return 64 * (c >> 2) + 4 * tx + (c & 3); }

template <int K, int V>
struct BwdSmem {
    static constexpr int SCR = (K > V ? K : V) * C;   // scratch: a transposed [K|V][C] copy or a state tile
    static constexpr int Q = 0;                         // [C][K] q~ = q e^{G - G_a}
    static constexpr int KA = Q + C * K;                // [C][K] k~ = k e^{G_a - G}
    static constexpr int G = KA + C * K;                // [C][K] G
    static constexpr int VV = G + C * K;                // [C][V] v
    static constexpr int DO = VV + C * V;               // [C][V] do, later q dq - k dk ([C][K])
    static constexpr int S6 = DO + C * (K > V ? K : V); // scratch
    static constexpr int BM = S6 + SCR;                 // [C][C] scale * masked do v^T
    static constexpr int AM = BM + C * C;               // [C][C] scale * masked q~ k~^T
    static constexpr int GA = AM + C * C;               // [K] G_a
    static constexpr int EGA = GA + K;                  // [K] e^{G_a}
    static constexpr int ELA = EGA + K;                 // [K] e^{G_l - G_a}
    static constexpr int PART = ELA + K;                // [NTB] partial cumsums
    static constexpr int FLOATS = PART + NTB;
};

template <typename Tin, int K, int V, typename Tg>
__global__ void __launch_bounds__(NTB, 1) bwd_grads(BwdArgs a)
{
    using L = BwdSmem<K, V>;
    extern __shared__ __align__(16) float sm[];
    float *Q = sm + L::Q, *KA = sm + L::KA, *G = sm + L::G, *VV = sm + L::VV, *DO = sm + L::DO;
    float *S6 = sm + L::S6, *BM = sm + L::BM, *AM = sm + L::AM;
    float *GA = sm + L::GA, *EGA = sm + L::EGA, *ELA = sm + L::ELA, *PART = sm + L::PART;
    const int j = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    int n, bos, eos;
    if (!bwd_slot(a, j, n, bos, eos))
        return;
    const int len = eos - bos, H = a.H;
    const size_t rb = row_head(bos, h, H, a.T, a.hf);   // row t of the chunk: row-head index rb + t * rs
    const int rs = a.hf ? 1 : H;
    const Tin *q = static_cast<const Tin *>(a.q), *k = static_cast<const Tin *>(a.k);
    const Tg *g = static_cast<const Tg *>(a.g);
    const Tin *v = static_cast<const Tin *>(a.v);
    const Tin *dout = static_cast<const Tin *>(a.dout);
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);

    // ---- load the chunk (rows >= len are zero; their gate is 0, so G stays at G_l there)
    for (int e = tid; e < C * K / 4; e += NTB) {
        const int i = e / (K / 4), c4 = (e - i * (K / 4)) * 4;
        const size_t o = (rb + (size_t)i * rs) * K + c4;
        const bool in = i < len;
        *reinterpret_cast<float4 *>(Q + i * K + c4) = in ? IO<Tin>::load4(q + o) : z4;
        *reinterpret_cast<float4 *>(KA + i * K + c4) = in ? IO<Tin>::load4(k + o) : z4;
        *reinterpret_cast<float4 *>(G + i * K + c4) = in ? IO<Tg>::load4(g + o) : z4;
    }
    for (int e = tid; e < C * V / 4; e += NTB) {
        const int i = e / (V / 4), c4 = (e - i * (V / 4)) * 4;
        const size_t o = (rb + (size_t)i * rs) * a.ldv + c4;
        const bool in = i < len;
        *reinterpret_cast<float4 *>(VV + i * V + c4) = in ? IO<Tin>::load4(v + o) : z4;
        *reinterpret_cast<float4 *>(DO + i * V + c4) = in ? IO<Tin>::load4(dout + o) : z4;
    }
    __syncthreads();
    // ---- chunk-local cumsum: NTB/K threads per key, each over C/(NTB/K) rows, then the partial prefix
    {
        constexpr int PARTS = NTB / K, RP = C / PARTS;
        const int kk = tid % K, part = tid / K;
        float run = 0.f;
        for (int r = 0; r < RP; ++r) {
            run += G[(part * RP + r) * K + kk];
            G[(part * RP + r) * K + kk] = run;
        }
        PART[part * K + kk] = run;
        __syncthreads();
        float off = 0.f;
        for (int p = 0; p < part; ++p)
            off += PART[p * K + kk];
        if (part > 0)
            for (int r = 0; r < RP; ++r)
                G[(part * RP + r) * K + kk] += off;
        __syncthreads();
        if (tid < K) {
            const float ga = G[AROW * K + tid], gl = G[(C - 1) * K + tid];
            GA[tid] = ga;
            EGA[tid] = expf(ga);
            ELA[tid] = expf(gl - ga);
        }
        __syncthreads();
    }
    // ---- q~, k~ in place
    for (int e = tid; e < C * K; e += NTB) {
        const int kk = e % K;
        const float d = G[e] - GA[kk];
        Q[e] *= expf(d);
        KA[e] *= expf(-d);
    }
    __syncthreads();

    // ---- AM = scale * mask(q~ k~^T), BM = scale * mask(do v^T)  (mask: column <= row)
    transpose_swz<K>(S6, KA);   // S6 <- k~^T  [K][C]
    __syncthreads();
    {
        float acc[4][4];
        zero<64>(acc);
        mm<64, false, true>(acc, Q, K, S6, C, K, ty, tx);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = 4 * ty + r, jj = 4 * tx + c;
                AM[i * C + jj] = jj <= i ? a.scale * acc[r][c] : 0.f;
            }
    }
    __syncthreads();
    transpose_swz<V>(S6, VV);   // S6 <- v^T  [V][C]
    __syncthreads();
    {
        float acc[4][4];
        zero<64>(acc);
        mm<64, false, true>(acc, DO, V, S6, C, V, ty, tx);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = 4 * ty + r, jj = 4 * tx + c;
                BM[i * C + jj] = jj <= i ? a.scale * acc[r][c] : 0.f;
            }
    }
    __syncthreads();

    const size_t tile = ((size_t)j * H + h) * K * V;   // this chunk's S_c / R_c [K][V]
    // ---- dv_j = (k~_j e^{G_l - G_a}) R_c + sum_i AM_ij do_i
    {
        float acc[4][V / 16];
        zero<V>(acc);
        mm<V, true>(acc, AM, C, DO, V, C, ty, tx);
        constexpr int KT = L::SCR / V;   // key rows of R_c per tile
        for (int k0 = 0; k0 < K; k0 += KT) {
            __syncthreads();
            for (int e = tid; e < KT * V / 4; e += NTB) {
                const int kr = e / (V / 4), c4 = (e - kr * (V / 4)) * 4;
                float4 x = *reinterpret_cast<const float4 *>(a.dR + tile + (size_t)(k0 + kr) * V + c4);
                const float f = ELA[k0 + kr];
                x.x *= f;
                x.y *= f;
                x.z *= f;
                x.w *= f;
                *reinterpret_cast<float4 *>(S6 + kr * V + c4) = x;
            }
            __syncthreads();
            mm<V, false>(acc, KA + k0, K, S6, V, KT, ty, tx);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int jj = 4 * ty + r;
            if (jj < len) {
                float *row = a.dv + (rb + (size_t)jj * rs) * a.ldv;
#pragma unroll
                for (int c = 0; c < V / 16; c += 4)
                    *reinterpret_cast<float4 *>(row + col_of(c, tx)) =
                        make_float4(acc[r][c], acc[r][c + 1], acc[r][c + 2], acc[r][c + 3]);
            }
        }
    }
    // ---- dq_i = e^{G_i - G_a} (sum_j BM_ij k~_j + scale e^{G_a} S_c do_i^T); q dq = q~ (that sum)
    float accq[4][K / 16];
    zero<K>(accq);
    mm<K, false>(accq, BM, C, KA, K, C, ty, tx);
    {
        constexpr int VT = L::SCR / K;   // value rows of S_c^T per tile
        for (int w0 = 0; w0 < V; w0 += VT) {
            __syncthreads();
            for (int e = tid; e < VT * K; e += NTB) {
                const int kk = e % K, vr = e / K;   // consecutive threads: consecutive keys (smem rows)
                S6[vr * K + kk] = a.dS[tile + (size_t)kk * V + w0 + vr] * a.scale * EGA[kk];
            }
            __syncthreads();
            mm<K, false>(accq, DO + w0, V, S6, K, VT, ty, tx);
        }
    }
    __syncthreads();   // every thread is done with do: its region becomes q dq - k dk
    float *PD = DO;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = 4 * ty + r;
#pragma unroll
        for (int c = 0; c < K / 16; ++c) {
            const int kk = col_of(c, tx);
            const float x = accq[r][c];
            PD[i * K + kk] = Q[i * K + kk] * x;
            accq[r][c] = x * expf(G[i * K + kk] - GA[kk]);
        }
        if (i < len) {
            float *row = a.dq + (rb + (size_t)i * rs) * K;
#pragma unroll
            for (int c = 0; c < K / 16; c += 4)
                put4(row + col_of(c, tx), make_float4(accq[r][c], accq[r][c + 1], accq[r][c + 2], accq[r][c + 3]),
                     a.acc);
        }
    }
    // ---- dk_j = e^{G_a - G_j} (sum_i BM_ij q~_i + e^{G_l - G_a} R_c v_j^T); k dk = k~ (that sum)
    float acck[4][K / 16];
    zero<K>(acck);
    mm<K, true>(acck, BM, C, Q, K, C, ty, tx);
    {
        constexpr int VT = L::SCR / K;
        for (int w0 = 0; w0 < V; w0 += VT) {
            __syncthreads();
            for (int e = tid; e < VT * K; e += NTB) {
                const int kk = e % K, vr = e / K;
                S6[vr * K + kk] = a.dR[tile + (size_t)kk * V + w0 + vr] * ELA[kk];
            }
            __syncthreads();
            mm<K, false>(acck, VV + w0, V, S6, K, VT, ty, tx);
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = 4 * ty + r;
#pragma unroll
        for (int c = 0; c < K / 16; ++c) {
            const int kk = col_of(c, tx);
            const float x = acck[r][c];
            PD[i * K + kk] -= KA[i * K + kk] * x;
            acck[r][c] = x * expf(GA[kk] - G[i * K + kk]);
        }
        if (i < len) {
            float *row = a.dk + (rb + (size_t)i * rs) * K;
#pragma unroll
            for (int c = 0; c < K / 16; c += 4)
                put4(row + col_of(c, tx), make_float4(acck[r][c], acck[r][c + 1], acck[r][c + 2], acck[r][c + 3]),
                     a.acc);
        }
    }
    __syncthreads();
    // ---- chunk-local suffix sums of q dq - k dk into dg; the chunk total for the carry scan
    if (tid < K) {
        float run = 0.f;
        for (int i = len - 1; i >= 0; --i) {
            run += PD[i * K + tid];
            float *d = a.dg + (rb + (size_t)i * rs) * K + tid;
            *d = a.acc ? *d + run : run;
        }
        a.dgt[((size_t)j * H + h) * K + tid] = run;
    }
}

// per (sequence, head, key): carry of every chunk = sum over later chunks + sum_v ht dht
__global__ void __launch_bounds__(NTB) bwd_dg_scan(BwdArgs a)
{
    const int kk = blockIdx.x * NTB + threadIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int K = a.K, V = a.V, H = a.H;
    if (kk >= K)
        return;
    int first, cnt;
    if (a.seqinfo) {
        const int2 si = a.seqinfo[n];
        first = si.x;
        cnt = si.y;
    } else {
        first = n * a.NC;
        cnt = a.NC;
    }
    float carry = 0.f;
    if (a.dht) {   // sum over v of ht * dht for this key: one contiguous row of V floats per thread
        const size_t st = (((size_t)n * H + h) * K + kk) * V;
        const float4 *x4 = reinterpret_cast<const float4 *>(a.ht + st);
        const float4 *y4 = reinterpret_cast<const float4 *>(a.dht + (((size_t)n * H + h) * K + kk) * a.lds);
#pragma unroll 8
        for (int i = 0; i < V / 4; ++i) {
            const float4 x = x4[i], y = y4[i];
            carry = fmaf(x.x, y.x, carry);
            carry = fmaf(x.y, y.y, carry);
            carry = fmaf(x.z, y.z, carry);
            carry = fmaf(x.w, y.w, carry);
        }
    }
    // reverse carry over the chunks, loads batched D chunks ahead of the in-place stores
    float *__restrict__ dgt = a.dgt + ((size_t)first * H + h) * K + kk;
    const size_t cs = (size_t)H * K;
    constexpr int D = 16;
    for (int c1 = cnt - 1; c1 >= 0; c1 -= D) {
        float t[D];
#pragma unroll
        for (int u = 0; u < D; ++u)
            if (c1 - u >= 0)
                t[u] = dgt[(size_t)(c1 - u) * cs];
#pragma unroll
        for (int u = 0; u < D; ++u)
            if (c1 - u >= 0) {
                dgt[(size_t)(c1 - u) * cs] = carry;
                carry += t[u];
            }
    }
}

__global__ void __launch_bounds__(128) bwd_dg_add(BwdArgs a)
{
    const int j = blockIdx.x, h = blockIdx.y, kk = threadIdx.x + blockIdx.z * 128;
    int n, bos, eos;
    if (kk >= a.K || !bwd_slot(a, j, n, bos, eos))
        return;
    const float carry = a.dgt[((size_t)j * a.H + h) * a.K + kk];
    const size_t rb = row_head(bos, h, a.H, a.T, a.hf);
    const int rs = a.hf ? 1 : a.H, len = eos - bos;
    float *__restrict__ dg = a.dg + rb * a.K + kk;
    const size_t st = (size_t)rs * a.K;
    constexpr int D = 8;   // rows per batch: all loads of a batch before its stores
    for (int t0 = 0; t0 < len; t0 += D) {
        float x[D];
#pragma unroll
        for (int u = 0; u < D; ++u)
            if (t0 + u < len)
                x[u] = dg[(size_t)(t0 + u) * st];
#pragma unroll
        for (int u = 0; u < D; ++u)
            if (t0 + u < len)
                dg[(size_t)(t0 + u) * st] = x[u] + carry;
    }
}

template <typename F>
cudaError_t smem_optin(F *f, size_t bytes)
{
    return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename Tin, int K, typename Tg = Tin>
cudaError_t launch_sums_t(const BwdArgs &a, int J, cudaStream_t s)
{
    const size_t bytes = sizeof(float) * ((size_t)2 * C * K + 2 * C * 64 + K);
    auto f = bwd_chunk_sums<Tin, K, Tg>;
    cudaError_t e = smem_optin(f, bytes);
    if (e != cudaSuccess)
        return e;
    f<<<dim3(J, a.H, a.V / 64), NTB, bytes, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, int K, int V, typename Tg>
cudaError_t launch_grads_t(const BwdArgs &a, int J, cudaStream_t s)
{
    const size_t bytes = sizeof(float) * BwdSmem<K, V>::FLOATS;
    auto f = bwd_grads<Tin, K, V, Tg>;
    cudaError_t e = smem_optin(f, bytes);
    if (e != cudaSuccess)
        return e;
    f<<<dim3(J, a.H), NTB, bytes, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, typename Tg = Tin>
cudaError_t launch_grads_kv(const BwdArgs &a, int J, cudaStream_t s)
{
    if (a.K == 64 && a.V == 64)
        return launch_grads_t<Tin, 64, 64, Tg>(a, J, s);
    if (a.K == 64 && a.V == 128)
        return launch_grads_t<Tin, 64, 128, Tg>(a, J, s);
    if (a.K == 128 && a.V == 64)
        return launch_grads_t<Tin, 128, 64, Tg>(a, J, s);
    return launch_grads_t<Tin, 128, 128, Tg>(a, J, s);
}

}  // namespace

bool bwd_supported(int dtype, int K, int V)
{
    return (dtype == GLA_F32 || dtype == GLA_BF16 || dtype == GLA_F16 || dtype == GLA_BF16_GF32 ||
            dtype == GLA_F16_GF32) &&
           (K == 64 || K == 128) && (V == 64 || V == 128);
}

cudaError_t launch_bwd_sums(const BwdArgs &a, int J, int dtype, cudaStream_t s)
{
    if (dtype == GLA_F32)
        return a.K == 64 ? launch_sums_t<float, 64>(a, J, s) : launch_sums_t<float, 128>(a, J, s);
    if (dtype == GLA_F16)
        return a.K == 64 ? launch_sums_t<__half, 64>(a, J, s) : launch_sums_t<__half, 128>(a, J, s);
    if (dtype == GLA_BF16_GF32)
        return a.K == 64 ? launch_sums_t<__nv_bfloat16, 64, float>(a, J, s)
                         : launch_sums_t<__nv_bfloat16, 128, float>(a, J, s);
    if (dtype == GLA_F16_GF32)
        return a.K == 64 ? launch_sums_t<__half, 64, float>(a, J, s) : launch_sums_t<__half, 128, float>(a, J, s);
    return a.K == 64 ? launch_sums_t<__nv_bfloat16, 64>(a, J, s) : launch_sums_t<__nv_bfloat16, 128>(a, J, s);
}

cudaError_t launch_bwd_scan(const BwdArgs &a, cudaStream_t s)
{
    bwd_scan<<<dim3((a.K * a.V + NTB - 1) / NTB, a.H, a.N), NTB, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_grads(const BwdArgs &a, int J, int dtype, cudaStream_t s)
{
    if (dtype == GLA_F16)
        return launch_grads_kv<__half>(a, J, s);
    if (dtype == GLA_BF16_GF32)
        return launch_grads_kv<__nv_bfloat16, float>(a, J, s);
    if (dtype == GLA_F16_GF32)
        return launch_grads_kv<__half, float>(a, J, s);
    return dtype == GLA_F32 ? launch_grads_kv<float>(a, J, s) : launch_grads_kv<__nv_bfloat16>(a, J, s);
}

cudaError_t launch_bwd_dg(const BwdArgs &a, int J, cudaStream_t s)
{
    bwd_dg_scan<<<dim3((a.K + NTB - 1) / NTB, a.H, a.N), NTB, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || J == 0)
        return e;
    bwd_dg_add<<<dim3(J, a.H, (a.K + 127) / 128), 128, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace gla
