// CUDA-core (fp32 FMA) kernels of the chunkwise GLA forward: the exact fp32 path, and the path every
// dtype takes for shapes the tensor-core kernels do not cover.
//
// Method (page "fla/ops/gla/fused_chunk.py"): per chunk of C rows with chunk-local cumsum G of the gates
// (FusedChunkGLAFunction.forward), the output is the inter-chunk term (q*exp(G)*scale) S plus the
// intra-chunk term sum_{s<=t} (q_t*exp(G_t-G_s)*scale . k_s) v_s with the inclusive diagonal
// (fwd_inner_chunk), and the state advances as S <- diag(exp(G_last)) S + (k*exp(G_last-G))^T V
// (fused_chunk_gla_fwd_kernel, prepare_qg_kg).
//
// Differences from the page's design: the pairwise exp(G_t-G_s) of fwd_inner_chunk is factorised as
// exp(G_t-G_a) * exp(G_a-G_s) around an anchor row a in the middle of the chunk (2*C*K exps per chunk
// instead of C*C*K), with exp(G_a) folded into the state operand; and sequences are cut into segments
// whose contributions are combined by a decayed scan, so few-head long sequences still fill the GPU.
#include "gla_internal.h"
#include "io.cuh"

namespace gla {

namespace {

constexpr int NT = 256;       // threads per CTA
constexpr int C = kChunk;     // 64
constexpr int BV = 64;        // value tile
constexpr int QS = C + 4;     // padded row stride of the transposed [K][C] tiles (keeps float4 alignment)

template <int K>
struct Smem {
    // floats
    static constexpr int G = 0;                  // [C][K]   G, then k^ = k*exp(G_last - G)
    static constexpr int QT = G + C * K;         // [K][QS]  q~^T = (scale*q*exp(G - G_a))^T
    static constexpr int KT = QT + K * QS;       // [K][QS]  k~^T = (k*exp(G_a - G))^T
    static constexpr int PT = KT + K * QS;       // [C][QS]  P^T (masked scores, [s][t])
    static constexpr int VS = PT + C * QS;       // [C][BV]  v tile
    static constexpr int SP = VS + C * BV;       // [K][BV]  S' = diag(exp(G_a)) S
    static constexpr int GA = SP + K * BV;       // [K]      G at the anchor row
    static constexpr int GL = GA + K;            // [K]      G at the last valid row
    static constexpr int TOT = GL + K;           // [NT/K][K] partial column sums of the cumsum
    static constexpr int OUT_FLOATS = TOT + NT;
    // the state-only kernel uses G, VS (placed right after G), GL and TOT
    static constexpr int S_VS = C * K;
    static constexpr int S_GL = S_VS + C * BV;
    static constexpr int S_TOT = S_GL + K;
    static constexpr int STATE_FLOATS = S_TOT + NT;
};

// Chunk-local inclusive cumsum of g for the chunk's rows t < len into Gs[C][K] (rows >= len get the
// running total, i.e. g = 0 there); row t of the chunk is row-head index rb + t * rs (layout-dependent).
// NT/K threads share a column; each scans C/(NT/K) rows in registers.
template <typename Tg, int K>
__device__ __forceinline__ void chunk_cumsum(const Tg *__restrict__ g, size_t rb, int rs, int len,
                                             float *Gs, float *Tot)
{
    constexpr int PARTS = NT / K, RPP = C / PARTS;
    const int col = threadIdx.x % K, part = threadIdx.x / K;
    float vals[RPP];
    float run = 0.f;
#pragma unroll
    for (int r = 0; r < RPP; ++r) {
        const int t = part * RPP + r;
        const float x = t < len ? IO<Tg>::load1(g + (rb + (size_t)t * rs) * K + col) : 0.f;
        run += x;
        vals[r] = run;
    }
    Tot[part * K + col] = run;
    __syncthreads();
    float off = 0.f;
    for (int q = 0; q < part; ++q)
        off += Tot[q * K + col];
#pragma unroll
    for (int r = 0; r < RPP; ++r)
        Gs[(part * RPP + r) * K + col] = vals[r] + off;
}

// Load the [C][BV] value tile (rows >= len zero) into Vs.
template <typename Tin>
__device__ __forceinline__ void load_v(const Tin *__restrict__ v, size_t rb, int rs, int V, int v0, int len,
                                       float *Vs)
{
    for (int e = threadIdx.x; e < C * BV / 4; e += NT) {
        const int t = (e * 4) / BV, c = (e * 4) % BV;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < len)
            x = IO<Tin>::load4(v + (rb + (size_t)t * rs) * V + v0 + c);
        *reinterpret_cast<float4 *>(Vs + t * BV + c) = x;
    }
}

// S (rows sk0..sk0+KPT-1, cols sv0..sv0+3 of the K x BV state tile) <- diag(exp(Gl)) S + Kh^T Vs.
template <int K>
__device__ __forceinline__ void advance_state(float (&S)[K / 16][4], const float *Gs, const float *Vs,
                                              const float *Gl, int sk0, int sv0, int len)
{
    constexpr int KPT = K / 16;
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
        const float d = expf(Gl[sk0 + i]);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            S[i][c] *= d;
    }
    for (int s = 0; s < len; ++s) {
        float kh[KPT];
#pragma unroll
        for (int i = 0; i < KPT; i += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(Gs + s * K + sk0 + i);
            kh[i] = x.x;
            kh[i + 1] = x.y;
            kh[i + 2] = x.z;
            kh[i + 3] = x.w;
        }
        const float4 vv = *reinterpret_cast<const float4 *>(Vs + s * BV + sv0);
#pragma unroll
        for (int i = 0; i < KPT; ++i) {
            S[i][0] = fmaf(kh[i], vv.x, S[i][0]);
            S[i][1] = fmaf(kh[i], vv.y, S[i][1]);
            S[i][2] = fmaf(kh[i], vv.z, S[i][2]);
            S[i][3] = fmaf(kh[i], vv.w, S[i][3]);
        }
    }
}

// Segment state contribution (kernel b) for every non-final segment: dS = sum over the segment's chunks
// of the decayed k^T v, starting from zero, plus the segment's total log-decay (kernel a fused in).
template <typename Tin, int K, typename Tg = Tin>
__global__ void __launch_bounds__(NT) state_ffma(Args a)
{
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    using L = Smem<K>;
    float *Gs = sm + L::G, *Vs = sm + L::S_VS, *Gl = sm + L::S_GL, *Tot = sm + L::S_TOT;
    constexpr int KPT = K / 16;
    const int vt = blockIdx.x, h = blockIdx.y, j = blockIdx.z;
    int n, p, bos, eos, send;
    if (!resolve_slot(a, j, n, p, bos, eos, send) || eos == send)
        return;
    const Tin *__restrict__ gk = static_cast<const Tin *>(a.k);
    const Tg *__restrict__ gg = static_cast<const Tg *>(a.g);
    const Tin *__restrict__ gv = static_cast<const Tin *>(a.v);
    const int H = a.H, V = a.V, v0 = vt * BV;
    const int sk0 = (threadIdx.x / 16) * KPT, sv0 = (threadIdx.x % 16) * 4;
    float S[KPT][4] = {};
    float gsum = 0.f;
    for (int c0 = bos; c0 < eos; c0 += C) {
        const int len = min(C, eos - c0);
        const size_t rb = row_head(c0, h, H, a.T, a.hf);
        const int rs = a.hf ? 1 : H;
        chunk_cumsum<Tg, K>(gg, rb, rs, len, Gs, Tot);
        load_v<Tin>(gv, rb, rs, V, v0, len, Vs);
        __syncthreads();
        if (threadIdx.x < K) {
            Gl[threadIdx.x] = Gs[(len - 1) * K + threadIdx.x];
            gsum += Gl[threadIdx.x];
        }
        __syncthreads();
        for (int e = threadIdx.x; e < C * K / 4; e += NT) {
            const int t = (e * 4) / K, kk = (e * 4) % K;
            float4 kv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < len)
                kv = IO<Tin>::load4(gk + (rb + (size_t)t * rs) * K + kk);
            float4 G4 = *reinterpret_cast<float4 *>(Gs + t * K + kk);
            G4.x = kv.x * expf(Gl[kk] - G4.x);
            G4.y = kv.y * expf(Gl[kk + 1] - G4.y);
            G4.z = kv.z * expf(Gl[kk + 2] - G4.z);
            G4.w = kv.w * expf(Gl[kk + 3] - G4.w);
            *reinterpret_cast<float4 *>(Gs + t * K + kk) = G4;
        }
        __syncthreads();
        advance_state<K>(S, Gs, Vs, Gl, sk0, sv0, len);
        __syncthreads();
    }
    float *dst = a.ss + ((size_t)j * H + h) * K * V;
#pragma unroll
    for (int i = 0; i < KPT; ++i)
        *reinterpret_cast<float4 *>(dst + (size_t)(sk0 + i) * V + v0 + sv0) =
            make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
    if (vt == 0 && threadIdx.x < K)
        a.gtot[((size_t)j * H + h) * K + threadIdx.x] = gsum;
}

// Fused output (kernel d): per (value tile, head, slot) run the chunk loop of the segment with the state
// in registers.  o_t = q~_t S' + sum_{s<=t} (q~_t . k~_s) v_s;  S <- diag(exp(G_last)) S + k^^T V.
template <typename Tin, typename Tout, int K, typename Tg = Tin>
__global__ void __launch_bounds__(NT, 1) out_ffma(Args a, int multi)
{
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    using L = Smem<K>;
    float *Gs = sm + L::G, *QtT = sm + L::QT, *KtT = sm + L::KT, *PT = sm + L::PT, *Vs = sm + L::VS;
    float *Sp = sm + L::SP, *Ga = sm + L::GA, *Gl = sm + L::GL, *Tot = sm + L::TOT;
    constexpr int KPT = K / 16;
    const int vt = blockIdx.x, h = blockIdx.y, j = blockIdx.z;
    int n, p, bos, eos, send;
    if (!resolve_slot(a, j, n, p, bos, eos, send))
        return;
    const Tin *__restrict__ gq = static_cast<const Tin *>(a.q);
    const Tin *__restrict__ gk = static_cast<const Tin *>(a.k);
    const Tg *__restrict__ gg = static_cast<const Tg *>(a.g);
    const Tin *__restrict__ gv = static_cast<const Tin *>(a.v);
    Tout *__restrict__ go = static_cast<Tout *>(a.o);
    const int H = a.H, V = a.V, v0 = vt * BV;
    const int tid = threadIdx.x;
    const int sk0 = (tid / 16) * KPT, sv0 = (tid % 16) * 4;
    const int ty = tid / 16, tx = tid % 16;

    float S[KPT][4];
    {
        const float *src = multi ? a.ss + ((size_t)j * H + h) * K * V
                                 : (a.h0 ? a.h0 + ((size_t)n * H + h) * K * V : nullptr);
#pragma unroll
        for (int i = 0; i < KPT; ++i) {
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (src)
                x = *reinterpret_cast<const float4 *>(src + (size_t)(sk0 + i) * V + v0 + sv0);
            S[i][0] = x.x;
            S[i][1] = x.y;
            S[i][2] = x.z;
            S[i][3] = x.w;
        }
    }

    for (int c0 = bos; c0 < eos; c0 += C) {
        const int len = min(C, eos - c0);
        const size_t rb = row_head(c0, h, H, a.T, a.hf);
        const int rs = a.hf ? 1 : H;
        chunk_cumsum<Tg, K>(gg, rb, rs, len, Gs, Tot);
        load_v<Tin>(gv, rb, rs, V, v0, len, Vs);
        __syncthreads();
        const int ra = min(C / 2 - 1, len - 1);
        if (tid < K) {
            Ga[tid] = Gs[ra * K + tid];
            Gl[tid] = Gs[(len - 1) * K + tid];
        }
        __syncthreads();
        // gated operands; k^ overwrites G in place (each element read and written by one thread)
        for (int e = tid; e < C * K / 4; e += NT) {
            const int t = (e * 4) / K, kk = (e * 4) % K;
            float4 qv = make_float4(0.f, 0.f, 0.f, 0.f), kv = qv;
            if (t < len) {
                qv = IO<Tin>::load4(gq + (rb + (size_t)t * rs) * K + kk);
                kv = IO<Tin>::load4(gk + (rb + (size_t)t * rs) * K + kk);
            }
            float4 G4 = *reinterpret_cast<float4 *>(Gs + t * K + kk);
            float kh[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float Gt = at(G4, i);
                QtT[(kk + i) * QS + t] = a.scale * at(qv, i) * expf(Gt - Ga[kk + i]);
                KtT[(kk + i) * QS + t] = at(kv, i) * expf(Ga[kk + i] - Gt);
                kh[i] = at(kv, i) * expf(Gl[kk + i] - Gt);
            }
            *reinterpret_cast<float4 *>(Gs + t * K + kk) = make_float4(kh[0], kh[1], kh[2], kh[3]);
        }
#pragma unroll
        for (int i = 0; i < KPT; ++i) {
            const float d = expf(Ga[sk0 + i]);
            *reinterpret_cast<float4 *>(Sp + (sk0 + i) * BV + sv0) =
                make_float4(d * S[i][0], d * S[i][1], d * S[i][2], d * S[i][3]);
        }
        __syncthreads();

        // intra scores P[t][s] = q~_t . k~_s, masked to s <= t (select, so inf/NaN above never leaks)
        {
            const int t0 = ty * 4, s0 = tx * 4;
            float acc[4][4] = {};
            for (int kk = 0; kk < K; ++kk) {
                const float4 qa = *reinterpret_cast<const float4 *>(QtT + kk * QS + t0);
                const float4 kb = *reinterpret_cast<const float4 *>(KtT + kk * QS + s0);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        acc[i][c] = fmaf(at(qa, i), at(kb, c), acc[i][c]);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int s = s0 + c;
                float4 col;
                col.x = s <= t0 + 0 ? acc[0][c] : 0.f;
                col.y = s <= t0 + 1 ? acc[1][c] : 0.f;
                col.z = s <= t0 + 2 ? acc[2][c] : 0.f;
                col.w = s <= t0 + 3 ? acc[3][c] : 0.f;
                *reinterpret_cast<float4 *>(PT + s * QS + t0) = col;
            }
        }
        __syncthreads();

        // output tile rows t0..t0+3, cols v0+c0v..+3: inter (q~ S') + intra (P V)
        {
            const int t0 = ty * 4, cv = tx * 4;
            float acc[4][4] = {};
            for (int kk = 0; kk < K; ++kk) {
                const float4 qa = *reinterpret_cast<const float4 *>(QtT + kk * QS + t0);
                const float4 sb = *reinterpret_cast<const float4 *>(Sp + kk * BV + cv);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        acc[i][c] = fmaf(at(qa, i), at(sb, c), acc[i][c]);
            }
            for (int s = 0; s < len; ++s) {
                const float4 pa = *reinterpret_cast<const float4 *>(PT + s * QS + t0);
                const float4 vb = *reinterpret_cast<const float4 *>(Vs + s * BV + cv);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        acc[i][c] = fmaf(at(pa, i), at(vb, c), acc[i][c]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (t0 + i < len)
                    IO<Tout>::store4(go + (rb + (size_t)(t0 + i) * rs) * V + v0 + cv,
                                     make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
        }

        advance_state<K>(S, Gs, Vs, Gl, sk0, sv0, len);
        __syncthreads();
    }

    if (eos == send && a.ht) {
        float *dst = a.ht + ((size_t)n * H + h) * K * V;
#pragma unroll
        for (int i = 0; i < KPT; ++i)
            *reinterpret_cast<float4 *>(dst + (size_t)(sk0 + i) * V + v0 + sv0) =
                make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
    }
}

// Decayed scan over the segments of each sequence (kernel c), parallel over (n, h, k, v):
//   ss[j0+p] <- S_in(p);  S_in(0) = h0 (or 0);  S_in(p+1) = diag(exp(gtot[p])) S_in(p) + dS(p).
__global__ void __launch_bounds__(256) scan_segments(Args a)
{
    const int KV = a.K * a.V;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    const int h = blockIdx.y, n = blockIdx.z;
    if (e >= KV)
        return;
    int j0, cnt;
    if (a.seqinfo) {
        const int2 si = a.seqinfo[n];
        j0 = si.x;
        cnt = si.y;
    } else {
        j0 = n * a.P;
        cnt = a.P;
    }
    const int kk = e / a.V;
    float carry = a.h0 ? a.h0[((size_t)n * a.H + h) * KV + e] : 0.f;
    int p = 0;
    // batches of 4 segments: issue the independent loads first, then run the dependent chain
    for (; p + 4 <= cnt - 1; p += 4) {
        float x[4], d[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t j = (size_t)(j0 + p + u);
            x[u] = a.ss[(j * a.H + h) * KV + e];
            d[u] = a.gtot[(j * a.H + h) * a.K + kk];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const size_t j = (size_t)(j0 + p + u);
            a.ss[(j * a.H + h) * KV + e] = carry;
            carry = fmaf(expf(d[u]), carry, x[u]);
        }
    }
    for (; p < cnt - 1; ++p) {
        const size_t j = (size_t)(j0 + p);
        const float x = a.ss[(j * a.H + h) * KV + e];
        const float d = a.gtot[(j * a.H + h) * a.K + kk];
        a.ss[(j * a.H + h) * KV + e] = carry;
        carry = fmaf(expf(d), carry, x);
    }
    if (cnt > 0)
        a.ss[((size_t)(j0 + cnt - 1) * a.H + h) * KV + e] = carry;
}

// Varlen plan (one CTA): validate cu_seqlens, give each sequence max(1, ceil(len/L)) slots, fill the
// slot table and per-sequence (first slot, count).  For the tensor-core kernel (a.sms > 0) the segment length
// follows the pack (see below) and, for up to 1024 sequences, the slots are ordered longest sequence first.
// Invalid offsets: report and leave every slot unused.
__global__ void __launch_bounds__(1024) plan_varlen(Args a)
{
    __shared__ int warp_sums[32];
    __shared__ long long wsum[32];
    __shared__ int wmax[32];
    __shared__ int bad, seg_len;
    __shared__ int lens[1024];   // ordered plan: the lengths, then the segment counts by rank
    int4 *table = const_cast<int4 *>(a.table);
    int2 *seqinfo = const_cast<int2 *>(a.seqinfo);
    const int tid = threadIdx.x, N = a.N, lane = tid & 31, w = tid >> 5, nw = blockDim.x >> 5;
    if (tid == 0)
        bad = (a.cu[0] != 0 || a.cu[N] != a.T) ? 1 : 0;
    __syncthreads();
    for (int n = tid; n < N; n += blockDim.x)
        if (a.cu[n + 1] < a.cu[n])
            bad = 1;
    __syncthreads();
    if (bad) {
        if (tid == 0)
            report(a.status, GLA_ERR_INVALID_ARG);
        for (int j = tid; j < a.J; j += blockDim.x)
            table[j] = make_int4(-1, 0, 0, 0);
        for (int n = tid; n < N; n += blockDim.x)
            seqinfo[n] = make_int2(0, 0);
        return;
    }
    // exclusive block-wide scan of one int per thread (every thread calls it); returns the total in *total
    auto block_scan = [&](int cnt, int &total) -> int {
        int x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += y;
        }
        if (lane == 31)
            warp_sums[w] = x;
        __syncthreads();
        if (w == 0) {
            int s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o)
                    s += y;
            }
            warp_sums[lane] = s;
        }
        __syncthreads();
        const int incl = x + (w > 0 ? warp_sums[w - 1] : 0);
        total = warp_sums[nw - 1];
        __syncthreads();
        return incl - cnt;
    };
    auto segments = [&](int len, int L, int &seg) {
        seg = L;
        int cnt = len > 0 ? (len + L - 1) / L : 1;
        if (a.seg_cap > 0 && cnt > a.seg_cap) {
            // longer segments for this sequence (a multiple of the chunk), at most seg_cap of them
            seg = ((len + a.seg_cap - 1) / a.seg_cap + kChunk - 1) / kChunk * kChunk;
            cnt = (len + seg - 1) / seg;
        }
        return cnt;
    };

    // Segment length.  Fixed (L rows) unless the tensor-core kernel's SM count is given: then, with the
    // average load of a CTA in chunks A = (sum of the sequences' chunks) x H x value tiles / SMs, no sequence
    // is cut when the longest is at most 1.25 A (its one item is then not much longer than an average CTA's
    // work, and nothing runs a state pass); otherwise segments of about A / 1.7 chunks (a cut segment runs a
    // state pass as well as its output pass), never shorter than L rows.
    int L = a.L;
    if (a.sms > 0) {
        long long csum = 0;
        int cmax = 0;
        for (int n = tid; n < N; n += blockDim.x) {
            const int len = a.cu[n + 1] - a.cu[n];
            const int c = len > 0 ? (len + kChunk - 1) / kChunk : 1;
            csum += c;
            cmax = max(cmax, c);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            csum += __shfl_xor_sync(0xffffffffu, csum, o);
            cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
        }
        if (lane == 0) {
            wsum[w] = csum;
            wmax[w] = cmax;
        }
        __syncthreads();
        if (tid == 0) {
            long long tot = 0;
            int mx = 0;
            for (int i = 0; i < nw; ++i) {
                tot += wsum[i];
                mx = max(mx, wmax[i]);
            }
            const double load = (double)tot * a.H * (a.V / 128) / a.sms;
            long long lr;
            if (mx <= 1.25 * load)
                lr = (long long)mx * kChunk;
            else
                lr = max((long long)a.L, (long long)ceil(load / 1.7) * kChunk);
            seg_len = (int)min(lr, (long long)(a.T > 0 ? (a.T + kChunk - 1) / kChunk * kChunk : kChunk));
        }
        __syncthreads();
        L = max(seg_len, kChunk);
    }

    if (a.sms > 0 && N <= (int)blockDim.x) {
        // sequences longest first (ties by index), so that the longest items are claimed in the first wave; the
        // segments of a sequence stay consecutive and in order (the scan's predecessors are claimed earlier)
        const int n = tid;
        const int len = n < N ? a.cu[n + 1] - a.cu[n] : 0;
        if (n < N)
            lens[n] = len;
        __syncthreads();
        int rank = 0;
        if (n < N)
            for (int m = 0; m < N; ++m) {
                const int lm = lens[m];
                rank += lm > len || (lm == len && m < n);
            }
        int seg = L;
        const int cnt = n < N ? segments(len, L, seg) : 0;
        __syncthreads();
        if (n < N)
            lens[rank] = cnt;
        __syncthreads();
        int total = 0;
        const int mine = tid < N ? lens[tid] : 0;
        const int excl = block_scan(mine, total);
        if (tid < N)
            lens[tid] = excl;   // first slot of the sequence of rank tid
        __syncthreads();
        if (n < N) {
            const int first = lens[rank];
            seqinfo[n] = make_int2(first, cnt);
            const int bos = a.cu[n], eos = a.cu[n + 1];
            for (int q = 0; q < cnt; ++q)
                table[first + q] = make_int4(n, q, min(bos + q * seg, eos), min(bos + (q + 1) * seg, eos));
        }
        for (int j = total + tid; j < a.J; j += blockDim.x)
            table[j] = make_int4(-1, 0, 0, 0);
        return;
    }

    int base = 0;
    for (int n0 = 0; n0 < N; n0 += blockDim.x) {
        const int n = n0 + tid;
        int cnt = 0, seg = L;
        if (n < N)
            cnt = segments(a.cu[n + 1] - a.cu[n], L, seg);
        int total = 0;
        const int first = base + block_scan(cnt, total);
        if (n < N) {
            seqinfo[n] = make_int2(first, cnt);
            const int bos = a.cu[n], eos = a.cu[n + 1];
            for (int q = 0; q < cnt; ++q)
                table[first + q] = make_int4(n, q, min(bos + q * seg, eos), min(bos + (q + 1) * seg, eos));
        }
        base += total;
    }
    for (int j = base + tid; j < a.J; j += blockDim.x)
        table[j] = make_int4(-1, 0, 0, 0);
}

// Standalone chunk-local cumsum (gla_chunk_local_cumsum): CTA per (row block of `chunk`, head), one
// thread per key dimension.  A block's first row may sit inside a chunk that began in the previous block;
// the thread then re-sums from that chunk's first row.
template <typename Tin>
__global__ void chunk_cumsum_standalone(const Tin *__restrict__ g, float *__restrict__ G,
                                        const int32_t *__restrict__ cu, int N, int T, int rows, int H,
                                        int K, int chunk)
{
    const int r0 = blockIdx.x * chunk, h = blockIdx.y;
    const int r1 = min(r0 + chunk, rows);
    auto seq_start = [&](int r) -> int {
        if (!cu)
            return (r / T) * T;
        int lo = 0, hi = N;   // largest n with cu[n] <= r
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cu[mid] <= r)
                lo = mid;
            else
                hi = mid - 1;
        }
        return cu[lo];
    };
    for (int kk = threadIdx.x; kk < K; kk += blockDim.x) {
        const int b0 = seq_start(r0);
        int u = b0 + ((r0 - b0) / chunk) * chunk;
        float run = 0.f;
        int bcur = b0;
        for (; u < r1; ++u) {
            const int b = u >= r0 ? seq_start(u) : bcur;
            if (b != bcur || (u - b) % chunk == 0) {
                run = 0.f;
                bcur = b;
            }
            run += IO<Tin>::load1(g + ((size_t)u * H + h) * K + kk);
            if (u >= r0)
                G[((size_t)u * H + h) * K + kk] = run;
        }
    }
}

template <typename F>
cudaError_t set_smem(F *f, size_t bytes)
{
    return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_plan_varlen(const Plan &pl, const Args &a, cudaStream_t s)
{
    plan_varlen<<<1, 1024, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_state_ffma(const Plan &pl, const Args &a, cudaStream_t s)
{
    dim3 grid(pl.NV, pl.H, pl.J);
    const bool bf = pl.dtype == GLA_BF16 || pl.dtype == GLA_BF16_OBF16, hf = pl.dtype == GLA_F16;
#define GLA_STATE(TIN, KK, ...)                                                             \
    {                                                                                       \
        auto f = state_ffma<TIN, KK, ##__VA_ARGS__>;                                        \
        const size_t sm = Smem<KK>::STATE_FLOATS * sizeof(float);                           \
        cudaError_t e = set_smem(f, sm);                                                    \
        if (e != cudaSuccess)                                                               \
            return e;                                                                       \
        f<<<grid, NT, sm, s>>>(a);                                                          \
        return cudaGetLastError();                                                          \
    }
    if (pl.dtype == GLA_BF16_GF32) {
        if (pl.K == 64) GLA_STATE(__nv_bfloat16, 64, float) else GLA_STATE(__nv_bfloat16, 128, float)
    }
    if (pl.dtype == GLA_F16_GF32) {
        if (pl.K == 64) GLA_STATE(__half, 64, float) else GLA_STATE(__half, 128, float)
    }
    if (pl.K == 64) {
        if (bf) GLA_STATE(__nv_bfloat16, 64) else if (hf) GLA_STATE(__half, 64) else GLA_STATE(float, 64)
    } else {
        if (bf) GLA_STATE(__nv_bfloat16, 128) else if (hf) GLA_STATE(__half, 128) else GLA_STATE(float, 128)
    }
#undef GLA_STATE
}

cudaError_t launch_scan(const Plan &pl, const Args &a, cudaStream_t s)
{
    dim3 grid((pl.K * pl.V + 255) / 256, pl.H, pl.N);
    scan_segments<<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_out_ffma(const Plan &pl, const Args &a, cudaStream_t s)
{
    dim3 grid(pl.NV, pl.H, pl.J);
    const int multi = pl.multi ? 1 : 0;
#define GLA_OUT(TIN, TOUT, KK, ...)                                                         \
    {                                                                                       \
        auto f = out_ffma<TIN, TOUT, KK, ##__VA_ARGS__>;                                    \
        const size_t sm = Smem<KK>::OUT_FLOATS * sizeof(float);                             \
        cudaError_t e = set_smem(f, sm);                                                    \
        if (e != cudaSuccess)                                                               \
            return e;                                                                       \
        f<<<grid, NT, sm, s>>>(a, multi);                                                   \
        return cudaGetLastError();                                                          \
    }
    if (pl.dtype == GLA_F32) {
        if (pl.K == 64) GLA_OUT(float, float, 64) else GLA_OUT(float, float, 128)
    } else if (pl.dtype == GLA_BF16) {
        if (pl.K == 64) GLA_OUT(__nv_bfloat16, float, 64) else GLA_OUT(__nv_bfloat16, float, 128)
    } else if (pl.dtype == GLA_F16) {
        if (pl.K == 64) GLA_OUT(__half, float, 64) else GLA_OUT(__half, float, 128)
    } else if (pl.dtype == GLA_BF16_GF32) {
        if (pl.K == 64) GLA_OUT(__nv_bfloat16, float, 64, float) else GLA_OUT(__nv_bfloat16, float, 128, float)
    } else if (pl.dtype == GLA_F16_GF32) {
        if (pl.K == 64) GLA_OUT(__half, float, 64, float) else GLA_OUT(__half, float, 128, float)
    } else {
        if (pl.K == 64) GLA_OUT(__nv_bfloat16, __nv_bfloat16, 64)
        else GLA_OUT(__nv_bfloat16, __nv_bfloat16, 128)
    }
#undef GLA_OUT
}

cudaError_t launch_chunk_cumsum(const void *g, float *G, const int32_t *cu, int N, int B, int T, int H,
                                int K, int chunk, int dtype, cudaStream_t s)
{
    const int rows = cu ? T : B * T;
    if (rows == 0)
        return cudaSuccess;
    dim3 grid((rows + chunk - 1) / chunk, H);
    const int threads = K < 128 ? K : 128;
    if (dtype == GLA_F32)
        chunk_cumsum_standalone<float><<<grid, threads, 0, s>>>(static_cast<const float *>(g), G, cu,
                                                                  N, T, rows, H, K, chunk);
    else if (dtype == GLA_F16)
        chunk_cumsum_standalone<__half><<<grid, threads, 0, s>>>(static_cast<const __half *>(g), G, cu, N, T,
                                                                   rows, H, K, chunk);
    else
        chunk_cumsum_standalone<__nv_bfloat16><<<grid, threads, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(g), G, cu, N, T, rows, H, K, chunk);
    return cudaGetLastError();
}

}  // namespace gla
