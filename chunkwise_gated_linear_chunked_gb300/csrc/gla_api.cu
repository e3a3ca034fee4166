// libgla C ABI: argument validation, the segment planner, the workspace layout and the launch sequence
// of the chunkwise GLA forward.  Declarations and contracts: include/gla.h.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "gla_internal.h"

namespace gla {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int sm_count()
{
    static std::mutex mu;
    static int cache[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128)
        return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

bool supported_k(int K) { return K == 64 || K == 128; }
// Accepted chunk lengths.  The kernels always tile at kChunk rows: the result of the method does not depend
// on the chunk length in exact arithmetic, so the argument only selects rounding, and one tiling serves all.
bool supported_chunk(int chunk) { return chunk == 16 || chunk == 32 || chunk == 64 || chunk == 128; }
bool supported_v(int V) { return V == 64 || V == 128 || V == 256; }

int check_shape(int B, int T, int H, int K, int V, int N, int chunk, int dtype, bool varlen)
{
    if (dtype != GLA_F32 && dtype != GLA_BF16 && dtype != GLA_BF16_OBF16 && dtype != GLA_F16 &&
        dtype != GLA_BF16_GF32 && dtype != GLA_F16_GF32)
        return GLA_ERR_UNSUPPORTED;
    if (B < 0 || T < 0 || H <= 0 || N < 0 || K <= 0 || V <= 0)
        return GLA_ERR_INVALID_ARG;
    if (varlen ? B != 1 : N != B)
        return GLA_ERR_INVALID_ARG;
    if (!supported_chunk(chunk) || !supported_k(K) || !supported_v(V))
        return GLA_ERR_UNSUPPORTED;
    const long long rows = varlen ? (long long)T : (long long)B * T;
    if (rows * H * (K > V ? K : V) >= (1LL << 31) || (long long)N * H * K * V >= (1LL << 31))
        return GLA_ERR_UNSUPPORTED;
    return GLA_OK;
}

// Segment plan.  One segment per sequence when sequences x heads x value tiles already give about two
// CTAs per SM; otherwise segments of L rows (a multiple of the chunk, at least 4 chunks) sized so the
// output pass has about that many CTAs.
void make_plan(Plan &pl, int B, int T, int H, int K, int V, int N, int chunk, int dtype, bool varlen)
{
    std::memset(&pl, 0, sizeof pl);
    pl.B = B; pl.T = T; pl.H = H; pl.K = K; pl.V = V; pl.N = N; pl.chunk = chunk; pl.dtype = dtype;
    pl.varlen = varlen;
    pl.tc = tc_supported(dtype, K, V);
    pl.BV = pl.tc ? 128 : 64;
    pl.NV = V / pl.BV;
    const long long rows = varlen ? (long long)T : (long long)B * T;
    const int nseq = varlen ? N : B;
    const long long target = 2LL * sm_count();
    const long long base = (long long)nseq * H * pl.NV;
    const int C = chunk;
    long long whole = varlen ? (long long)T : (long long)T;   // longest possible sequence
    whole = (whole + C - 1) / C * C;
    if (whole < C)
        whole = C;
    long long L = whole;
    if (pl.tc && rows > 0) {
        // Fused tensor-core kernel (one persistent CTA per SM; a segment that is not the last of its sequence
        // runs a state pass first and publishes its contribution for the segment scan).  Measured on GB300:
        //  * dense batches whose (sequence, head, value tile) items already fill the GPU are not split (a
        //    state pass costs more than the wave it would balance);
        //  * otherwise the fewest segments that fill one wave: every item runs at once, so the segment scan
        //    waits only for the state passes, never for a claimed but unstarted predecessor;
        //  * varlen packs: the device plan cuts no sequence when the longest is not much longer than a CTA's
        //    average load, else segments of about that load (never shorter than kSegRows rows, the bound the
        //    slot count is sized for), longest sequences first.
        const long long sms = sm_count();
        const long long nv = pl.NV;
        if (varlen) {
            L = std::min<long long>(kSegRows, whole);
        } else {
            const long long units1 = (long long)B * H * nv;
            long long P = 1;
            if (units1 < sms)
                P = std::max(1LL, sms / units1);
            L = ((T + P - 1) / P + C - 1) / C * C;
            if (L < 4 * C)
                L = 4 * C;
            if (L > whole)
                L = whole;
            // Balanced pieces: when the units do not divide the CTAs evenly, equal segments per unit leave
            // sms % units1 CTAs idle and every CTA waits as long as the longest segment.  Instead the B*H
            // units' chunks, taken in order, are cut into sms / NV near-equal pieces (one CTA each, per value
            // tile); a piece crossing from one unit into the next is two segments run by one CTA.  Worth it
            // for long pieces only (every extra segment of a unit adds a tile to the segment scan), and only
            // when the longest CTA's load drops by a tenth; a chunk of a state pass costs about 0.41 of an
            // output chunk (it reads k, g, v at the HBM rate).
            const long long units = (long long)B * H, nc = (T + C - 1) / C, np = sms / nv;
            const double seg_load = (L < T ? 1.41 : 1.0) * (double)(L / C);
            const double piece_load = 1.41 * (double)(units * nc) / (double)np;
            if (units1 < sms && units < np && np % units != 0 && units * nc >= kPieceChunks * np &&
                piece_load < 0.9 * seg_load) {
                pl.np = (int)np;
                pl.nc = (int)nc;
            }
        }
    } else if (base < target && rows > 0) {
        long long per = (rows * H * pl.NV + target - 1) / target;   // rows per CTA
        per = (per + C - 1) / C;
        if (per < 4)
            per = 4;
        L = per * C;
        if (L > whole)
            L = whole;
    }
    pl.L = (int)L;
    if (varlen) {
        pl.P = 0;
        pl.J = N + (int)((T + L - 1) / L);
        pl.multi = L < T;
    } else if (pl.np) {
        // most segments of one unit: the pieces it overlaps
        const long long tot = (long long)B * H * pl.nc;
        auto piece_of = [&](long long x) { return ((x + 1) * pl.np + tot - 1) / tot - 1; };
        long long most = 1;
        for (long long U = 0; U < (long long)B * H; ++U)
            most = std::max(most, piece_of((U + 1) * pl.nc - 1) - piece_of(U * pl.nc) + 1);
        pl.P = (int)most;
        pl.J = B * pl.P;
        pl.multi = pl.P > 1;
    } else {
        pl.P = T > 0 ? (int)((T + L - 1) / L) : 1;
        pl.J = B * pl.P;
        pl.multi = pl.P > 1;
    }
    size_t off = 0;
    pl.off_status = off;
    off += kAlign;
    pl.off_table = off;
    if (varlen)
        off += align_up(sizeof(int4) * (size_t)pl.J);
    pl.off_seq = off;
    if (varlen)
        off += align_up(sizeof(int2) * (size_t)N);
    pl.off_ss = off;
    if (pl.multi)
        off += align_up(sizeof(float) * (size_t)pl.J * H * K * V);
    pl.off_agg = off;
    if (pl.multi && pl.tc)
        off += align_up(sizeof(float) * (size_t)pl.J * H * K * V);
    pl.off_gtot = off;
    if (pl.multi)
        off += align_up(sizeof(float) * (size_t)pl.J * H * K * (pl.tc ? pl.NV : 1));
    // the fused kernel's work counters and launch epoch live in the fixed header (status word at byte 0,
    // counters at 16, epoch at 24), so they mean the same thing whatever the layout of the previous call
    // that used this workspace
    pl.off_ctr = 16;
    pl.off_flags = off;
    if (pl.tc && pl.multi)
        off += align_up(sizeof(int) * (size_t)pl.J * H * pl.NV);
    pl.total = off;
}

// Per-thread measurement hook state (gla_profile_events).
struct Profile {
    cudaEvent_t *events = nullptr;
    int n_events = 0;
    int *ids = nullptr;
    int launches = 0;
};
thread_local Profile g_prof;

enum KernelId {
    K_PLAN = 1, K_STATE_FFMA = 2, K_SCAN = 3, K_OUT_FFMA = 4, K_FUSED_TC = 7,
    K_BWD_SUMS = 8, K_BWD_SCAN = 9, K_BWD_GRADS = 10, K_BWD_DG = 11, K_TTT = 12, K_WY = 13,
    K_WY_TC = 14, K_BWD_SUMS_TC = 15, K_BWD_GRADS_TC = 16, K_TTT_TC = 17
};

// Launch one kernel through `fn`, bracketed by the profiling events when they are armed.
template <typename Fn>
cudaError_t profiled(int id, cudaStream_t s, Fn fn)
{
    Profile &p = g_prof;
    const int i = p.launches++;
    const bool rec = p.events && 2 * i + 1 < p.n_events;
    if (rec && cudaEventRecord(p.events[2 * i], s) != cudaSuccess)
        return cudaErrorUnknown;
    cudaError_t e = fn();
    if (e != cudaSuccess)
        return e;
    if (rec) {
        if (p.ids)
            p.ids[i] = id;
        return cudaEventRecord(p.events[2 * i + 1], s);
    }
    return cudaSuccess;
}

bool misaligned(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u); }

struct Range {
    uintptr_t lo, hi;
};
Range range_of(const void *p, size_t bytes)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return {a, a + bytes};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

}  // namespace
}  // namespace gla

using namespace gla;

extern "C" size_t gla_fwd_workspace_size(int B, int T, int H, int K, int V, int N, int chunk, int dtype)
{
    dtype &= ~GLA_HEAD_FIRST;   // the layout does not change the workspace
    // The workspace size does not depend on whether cu_seqlens is given except through N; size for the
    // larger of the two layouts so one query serves both.
    const bool varlen_ok = check_shape(B, T, H, K, V, N, chunk, dtype, B == 1) == GLA_OK;
    const bool dense_ok = check_shape(B, T, H, K, V, N, chunk, dtype, false) == GLA_OK;
    size_t best = 0;
    Plan pl;
    if (varlen_ok && B == 1) {
        make_plan(pl, B, T, H, K, V, N, kChunk, dtype, true);
        best = pl.total;
    }
    if (dense_ok) {
        make_plan(pl, B, T, H, K, V, N, kChunk, dtype, false);
        if (pl.total > best)
            best = pl.total;
    }
    return best;
}

extern "C" int gla_fwd(const void *q, const void *k, const void *v, const void *g, void *o, float scale,
                       const float *h0, float *ht, const int32_t *cu_seqlens, int N, int B, int T, int H,
                       int K, int V, int chunk, int dtype, void *workspace, size_t workspace_bytes,
                       void *stream)
{
    const bool varlen = cu_seqlens != nullptr;
    const bool hf = (dtype & GLA_HEAD_FIRST) != 0;
    dtype &= ~GLA_HEAD_FIRST;
    int rc = check_shape(B, T, H, K, V, N, chunk, dtype, varlen);
    if (rc != GLA_OK)
        return rc;
    if (!(scale > 0.f) || !std::isfinite(scale))
        return GLA_ERR_INVALID_ARG;
    const size_t rows = varlen ? (size_t)T : (size_t)B * T;
    const size_t esz = dtype == GLA_F32 ? 4 : 2, osz = dtype == GLA_BF16_OBF16 ? 2 : 4;
    const size_t gsz = (dtype == GLA_F32 || dtype == GLA_BF16_GF32 || dtype == GLA_F16_GF32) ? 4 : 2;
    if (rows > 0 && (!q || !k || !v || !g || !o))
        return GLA_ERR_INVALID_ARG;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(g) || misaligned(o) ||
        misaligned(h0) || misaligned(ht) || misaligned(cu_seqlens))
        return GLA_ERR_ALIGNMENT;
    Plan pl;
    make_plan(pl, B, T, H, K, V, N, kChunk, dtype, varlen);
    if (!workspace)
        return GLA_ERR_WORKSPACE;
    if (workspace_bytes < pl.total)
        return GLA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign)
        return GLA_ERR_ALIGNMENT;
    // aliasing: outputs overlap no input and no other output (h0 == ht exactly is allowed)
    const Range rq = range_of(q, rows * H * K * esz), rk = range_of(k, rows * H * K * esz);
    const Range rg = range_of(g, rows * H * K * gsz), rv = range_of(v, rows * H * V * esz);
    const Range ro = range_of(o, rows * H * V * osz);
    const size_t sbytes = (size_t)N * H * K * V * 4;
    const Range rh0 = range_of(h0, h0 ? sbytes : 0), rht = range_of(ht, ht ? sbytes : 0);
    const Range rws = range_of(workspace, pl.total);
    const Range rcu = range_of(cu_seqlens, varlen ? sizeof(int32_t) * (size_t)(N + 1) : 0);
    for (Range in : {rq, rk, rg, rv, rh0, rcu, rws})
        if (overlap(ro, in))
            return GLA_ERR_INVALID_ARG;
    for (Range in : {rq, rk, rg, rv, rcu, rws, ro})
        if (overlap(rht, in))
            return GLA_ERR_INVALID_ARG;
    if (h0 && ht && h0 != ht && overlap(rh0, rht))
        return GLA_ERR_INVALID_ARG;
    for (Range in : {rq, rk, rg, rv, rh0, rcu})
        if (overlap(rws, in))
            return GLA_ERR_INVALID_ARG;
    if (pl.J == 0) {
        g_prof.launches = 0;
        return GLA_OK;
    }

    char *ws = static_cast<char *>(workspace);
    Args a;
    std::memset(&a, 0, sizeof a);
    a.q = q; a.k = k; a.v = v; a.g = g; a.o = o; a.h0 = h0; a.ht = ht; a.cu = cu_seqlens;
    a.scale = scale;
    a.seg_cap = 0;
    a.hf = hf ? 1 : 0;
    a.B = B; a.T = T; a.H = H; a.K = K; a.V = V; a.N = N; a.L = pl.L; a.P = pl.P; a.J = pl.J;
    a.sms = pl.tc && varlen ? sm_count() : 0;   // the tensor-core kernel's varlen plan follows the pack
    a.np = pl.np;
    a.nc = pl.nc;
    a.status = reinterpret_cast<int *>(ws + pl.off_status);
    if (varlen) {
        a.table = reinterpret_cast<const int4 *>(ws + pl.off_table);
        a.seqinfo = reinterpret_cast<const int2 *>(ws + pl.off_seq);
    }
    if (pl.multi) {
        a.ss = reinterpret_cast<float *>(ws + pl.off_ss);
        a.gtot = reinterpret_cast<float *>(ws + pl.off_gtot);
        if (pl.tc)
            a.agg = reinterpret_cast<float *>(ws + pl.off_agg);
    }
    if (pl.tc) {
        a.ctr = reinterpret_cast<int *>(ws + pl.off_ctr);
        if (pl.multi)
            a.flags = reinterpret_cast<int *>(ws + pl.off_flags);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    g_prof.launches = 0;
    if (varlen && profiled(K_PLAN, s, [&] { return launch_plan_varlen(pl, a, s); }) != cudaSuccess)
        return GLA_ERR_CUDA;
    if (pl.tc) {
        // one persistent kernel: state pass, segment scan and output pass per work item (its publication
        // flags are tagged with a launch epoch kept in the workspace header, so they need no clearing)
        const int sms = sm_count();
        if (profiled(K_FUSED_TC, s, [&] { return launch_fused_tc(pl, a, s, sms); }) != cudaSuccess)
            return GLA_ERR_CUDA;
        return GLA_OK;
    }
    if (pl.multi) {
        if (profiled(K_STATE_FFMA, s, [&] { return launch_state_ffma(pl, a, s); }) != cudaSuccess)
            return GLA_ERR_CUDA;
        if (profiled(K_SCAN, s, [&] { return launch_scan(pl, a, s); }) != cudaSuccess)
            return GLA_ERR_CUDA;
    }
    if (profiled(K_OUT_FFMA, s, [&] { return launch_out_ffma(pl, a, s); }) != cudaSuccess)
        return GLA_ERR_CUDA;
    return GLA_OK;
}

extern "C" int gla_get_status(void *workspace, void *stream)
{
    if (!workspace)
        return GLA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return GLA_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return GLA_ERR_CUDA;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpy(workspace, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return GLA_ERR_CUDA;
    }
    return word;
}

extern "C" const char *gla_strerror(int code)
{
    switch (code) {
    case GLA_OK: return "ok";
    case GLA_ERR_INVALID_ARG: return "invalid argument";
    case GLA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case GLA_ERR_ALIGNMENT: return "device pointer not 16-byte aligned (workspace: 256-byte)";
    case GLA_ERR_WORKSPACE: return "workspace missing or too small";
    case GLA_ERR_CUDA: return "CUDA runtime or launch failure";
    case GLA_ERR_TIMEOUT: return "a bounded device wait ran out";
    case GLA_ERR_RANGE: return "a value left the fp16 operand range of the tensor-core path";
    default: return "unknown status code";
    }
}

extern "C" int gla_chunk_local_cumsum(const void *g, float *G, const int32_t *cu_seqlens, int N, int B,
                                      int T, int H, int K, int chunk, int dtype, void *stream)
{
    const bool varlen = cu_seqlens != nullptr;
    if (dtype != GLA_F32 && dtype != GLA_BF16 && dtype != GLA_F16)
        return GLA_ERR_UNSUPPORTED;
    if (B < 0 || T < 0 || H <= 0 || K <= 0 || N < 0 || (varlen ? B != 1 : false))
        return GLA_ERR_INVALID_ARG;
    if (chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128)
        return GLA_ERR_UNSUPPORTED;
    const size_t rows = varlen ? (size_t)T : (size_t)B * T;
    if (rows > 0 && (!g || !G))
        return GLA_ERR_INVALID_ARG;
    if (rows * H * K >= (1ull << 31))
        return GLA_ERR_UNSUPPORTED;
    if (misaligned(g) || misaligned(G) || misaligned(cu_seqlens))
        return GLA_ERR_ALIGNMENT;
    const size_t esz = dtype == GLA_F32 ? 4 : 2;
    if (overlap(range_of(g, rows * H * K * esz), range_of(G, rows * H * K * 4)))
        return GLA_ERR_INVALID_ARG;
    if (launch_chunk_cumsum(g, G, cu_seqlens, N, B, T, H, K, chunk, dtype,
                            static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GLA_ERR_CUDA;
    return GLA_OK;
}

extern "C" int gla_profile_events(void **events, int n_events, int *kernel_ids)
{
    if (n_events < 0)
        return GLA_ERR_INVALID_ARG;
    g_prof.events = events ? reinterpret_cast<cudaEvent_t *>(events) : nullptr;
    g_prof.n_events = events ? n_events : 0;
    g_prof.ids = events ? kernel_ids : nullptr;
    return GLA_OK;
}

extern "C" int gla_profile_launches(void) { return g_prof.launches; }

extern "C" const char *gla_kernel_name(int kernel_id)
{
    switch (kernel_id) {
    case K_PLAN: return "plan_varlen";
    case K_STATE_FFMA: return "state_ffma";
    case K_SCAN: return "scan_segments";
    case K_OUT_FFMA: return "out_ffma";
    case K_FUSED_TC: return "fused_tc";
    case K_BWD_SUMS: return "bwd_chunk_sums";
    case K_BWD_SCAN: return "bwd_scan";
    case K_BWD_GRADS: return "bwd_grads";
    case K_BWD_DG: return "bwd_dg";
    case K_TTT: return "ttt_linear_fwd";
    case K_WY: return "wy_fwd_ffma";
    case K_WY_TC: return "wy_fwd_tc";
    case K_BWD_SUMS_TC: return "bwd_chunk_sums_tc";
    case K_BWD_GRADS_TC: return "bwd_grads_tc";
    case K_TTT_TC: return "ttt_linear_tc";
    default: return "unknown";
    }
}

// ---------------------------------------------------------------------------------------------------
// Backward pass
// ---------------------------------------------------------------------------------------------------
namespace gla {
namespace {

struct BwdPlan {
    int J, NC;
    size_t off_table, off_seq, off_dS, off_dR, off_gl, off_ht, off_dgt, total;
};

void make_bwd_plan(BwdPlan &bp, int B, int T, int H, int K, int V, int N, bool varlen)
{
    std::memset(&bp, 0, sizeof bp);
    const int C = kChunk;
    bp.NC = varlen ? 0 : (T + C - 1) / C;
    bp.J = varlen ? N + (T + C - 1) / C : B * bp.NC;
    const int nseq = varlen ? N : B;
    size_t off = kAlign;   // status header
    bp.off_table = off;
    if (varlen)
        off += align_up(sizeof(int4) * (size_t)bp.J);
    bp.off_seq = off;
    if (varlen)
        off += align_up(sizeof(int2) * (size_t)N);
    const size_t tile = sizeof(float) * (size_t)bp.J * H * K * V;
    bp.off_dS = off;
    off += align_up(tile);
    bp.off_dR = off;
    off += align_up(tile);
    bp.off_gl = off;
    off += align_up(sizeof(float) * (size_t)bp.J * H * K);
    bp.off_ht = off;
    off += align_up(sizeof(float) * (size_t)nseq * H * K * V);
    bp.off_dgt = off;
    off += align_up(sizeof(float) * (size_t)bp.J * H * K);
    bp.total = off;
}

int check_bwd_shape(int B, int T, int H, int K, int V, int N, int chunk, int dtype, bool varlen)
{
    if (dtype != GLA_F32 && dtype != GLA_BF16 && dtype != GLA_F16 && dtype != GLA_BF16_GF32 &&
        dtype != GLA_F16_GF32)
        return GLA_ERR_UNSUPPORTED;
    if (B < 0 || T < 0 || H <= 0 || N < 0)
        return GLA_ERR_INVALID_ARG;
    if (varlen ? B != 1 : N != B)
        return GLA_ERR_INVALID_ARG;
    // V = 256 runs as two 128-wide value slices
    if (!supported_chunk(chunk) || !bwd_supported(dtype, K, V == 256 ? 128 : V))
        return GLA_ERR_UNSUPPORTED;
    const long long rows = varlen ? (long long)T : (long long)B * T;
    if (rows * H * (K > V ? K : V) >= (1LL << 31) || (long long)(N + T / kChunk + 1) * H * K * V >= (1LL << 31))
        return GLA_ERR_UNSUPPORTED;
    return GLA_OK;
}

// The value width one pass of the backward handles: V, or 128-wide slices of a wider V.
int bwd_slice(int V) { return V > 128 ? 128 : V; }

}  // namespace
}  // namespace gla

using namespace gla;

extern "C" size_t gla_bwd_workspace_size(int B, int T, int H, int K, int V, int N, int chunk, int dtype)
{
    dtype &= ~GLA_HEAD_FIRST;
    if (check_bwd_shape(B, T, H, K, V, N, chunk, dtype, false) != GLA_OK &&
        check_bwd_shape(1, T, H, K, V, N, chunk, dtype, true) != GLA_OK)
        return 0;
    BwdPlan a, b;
    make_bwd_plan(a, B, T, H, K, bwd_slice(V), B, false);
    make_bwd_plan(b, 1, T, H, K, bwd_slice(V), N, true);
    return a.total > b.total ? a.total : b.total;
}

extern "C" int gla_bwd(const void *q, const void *k, const void *v, const void *g, const void *dout, float scale,
                       const float *h0, const float *dht, float *dq, float *dk, float *dv, float *dg, float *dh0,
                       const int32_t *cu_seqlens, int N, int B, int T, int H, int K, int V, int chunk, int dtype,
                       void *workspace, size_t workspace_bytes, void *stream)
{
    const bool varlen = cu_seqlens != nullptr;
    const bool hf = (dtype & GLA_HEAD_FIRST) != 0;
    dtype &= ~GLA_HEAD_FIRST;
    int rc = check_bwd_shape(B, T, H, K, V, N, chunk, dtype, varlen);
    if (rc != GLA_OK)
        return rc;
    if (!(scale > 0.f) || !std::isfinite(scale))
        return GLA_ERR_INVALID_ARG;
    const size_t rows = varlen ? (size_t)T : (size_t)B * T;
    const size_t esz = dtype == GLA_F32 ? 4 : 2;
    const size_t gsz = (dtype == GLA_F32 || dtype == GLA_BF16_GF32 || dtype == GLA_F16_GF32) ? 4 : 2;
    if (rows > 0 && (!q || !k || !v || !g || !dout || !dq || !dk || !dv || !dg))
        return GLA_ERR_INVALID_ARG;
    for (const void *p : {q, k, v, g, dout, (const void *)h0, (const void *)dht, (const void *)dq,
                          (const void *)dk, (const void *)dv, (const void *)dg, (const void *)dh0,
                          (const void *)cu_seqlens})
        if (misaligned(p))
            return GLA_ERR_ALIGNMENT;
    const int VS = bwd_slice(V);   // value width of one pass
    BwdPlan bp;
    make_bwd_plan(bp, B, T, H, K, VS, N, varlen);
    if (!workspace || workspace_bytes < bp.total)
        return GLA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign)
        return GLA_ERR_ALIGNMENT;
    // aliasing: every output overlaps no input, no workspace and no other output
    const size_t sbytes = (size_t)(varlen ? N : B) * H * K * V * 4;
    const Range in[] = {range_of(q, rows * H * K * esz), range_of(k, rows * H * K * esz),
                        range_of(g, rows * H * K * gsz), range_of(v, rows * H * V * esz),
                        range_of(dout, rows * H * V * esz), range_of(h0, h0 ? sbytes : 0),
                        range_of(dht, dht ? sbytes : 0),
                        range_of(cu_seqlens, varlen ? sizeof(int32_t) * (size_t)(N + 1) : 0),
                        range_of(workspace, bp.total)};
    const Range out[] = {range_of(dq, rows * H * K * 4), range_of(dk, rows * H * K * 4),
                         range_of(dg, rows * H * K * 4), range_of(dv, rows * H * V * 4),
                         range_of(dh0, dh0 ? sbytes : 0)};
    for (size_t i = 0; i < sizeof out / sizeof out[0]; ++i) {
        for (const Range &r : in)
            if (overlap(out[i], r))
                return GLA_ERR_INVALID_ARG;
        for (size_t j2 = i + 1; j2 < sizeof out / sizeof out[0]; ++j2)
            if (overlap(out[i], out[j2]))
                return GLA_ERR_INVALID_ARG;
    }
    for (size_t i = 0; i + 1 < sizeof in / sizeof in[0]; ++i)
        if (overlap(in[i], in[8]))
            return GLA_ERR_INVALID_ARG;
    const int nseq = varlen ? N : B;
    g_prof.launches = 0;
    if (nseq == 0)
        return GLA_OK;

    char *ws = static_cast<char *>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    BwdArgs a;
    std::memset(&a, 0, sizeof a);
    a.q = q; a.k = k; a.v = v; a.g = g; a.dout = dout; a.h0 = h0; a.dht = dht;
    a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dh0 = dh0;
    a.scale = scale;
    a.B = B; a.T = T; a.H = H; a.K = K; a.V = VS; a.N = nseq; a.NC = bp.NC;
    a.ldv = V; a.lds = V; a.acc = 0;
    a.hf = hf ? 1 : 0;
    a.status = reinterpret_cast<int *>(ws);
    a.dS = reinterpret_cast<float *>(ws + bp.off_dS);
    a.dR = reinterpret_cast<float *>(ws + bp.off_dR);
    a.gl = reinterpret_cast<float *>(ws + bp.off_gl);
    a.ht = reinterpret_cast<float *>(ws + bp.off_ht);
    a.dgt = reinterpret_cast<float *>(ws + bp.off_dgt);
    if (varlen) {
        // the forward's slot planner with 64-row segments gives the chunk table
        Args pa;
        std::memset(&pa, 0, sizeof pa);
        pa.cu = cu_seqlens; pa.N = N; pa.T = T; pa.L = kChunk; pa.J = bp.J; pa.seg_cap = 0;
        pa.status = a.status;
        pa.table = reinterpret_cast<const int4 *>(ws + bp.off_table);
        pa.seqinfo = reinterpret_cast<const int2 *>(ws + bp.off_seq);
        a.table = pa.table;
        a.seqinfo = pa.seqinfo;
        Plan pl;
        std::memset(&pl, 0, sizeof pl);
        if (profiled(K_PLAN, s, [&] { return launch_plan_varlen(pl, pa, s); }) != cudaSuccess)
            return GLA_ERR_CUDA;
    }
    const int J = bp.J;
    // bf16 q, k, v, dout with K = 128: chunk sums on the tensor cores (and the gradients for 128-wide values);
    // everything else on CUDA cores.  A V wider than one pass runs as value slices: dv, dh0 and the states are
    // per slice, dq, dk and dg (linear in the slices) are accumulated by the later slices.
    const bool sums_tc = bwd_sums_tc_supported(dtype, K, VS);
    const bool grads_tc = bwd_grads_tc_supported(dtype, K, VS);
    const size_t vbytes = dtype == GLA_F32 ? 4 : 2;
    for (int v0 = 0; v0 < V; v0 += VS) {
        a.v = static_cast<const char *>(v) + (size_t)v0 * vbytes;
        a.dout = static_cast<const char *>(dout) + (size_t)v0 * vbytes;
        a.dv = dv + v0;
        a.h0 = h0 ? h0 + v0 : nullptr;
        a.dht = dht ? dht + v0 : nullptr;
        a.dh0 = dh0 ? dh0 + v0 : nullptr;
        a.acc = v0 > 0;
        if (J > 0 && profiled(sums_tc ? K_BWD_SUMS_TC : K_BWD_SUMS, s, [&] {
                return sums_tc ? launch_bwd_sums_tc(a, J, dtype, s) : launch_bwd_sums(a, J, dtype, s);
            }) != cudaSuccess)
            return GLA_ERR_CUDA;
        if (profiled(K_BWD_SCAN, s, [&] { return launch_bwd_scan(a, s); }) != cudaSuccess)
            return GLA_ERR_CUDA;
        if (J > 0 && profiled(grads_tc ? K_BWD_GRADS_TC : K_BWD_GRADS, s, [&] {
                return grads_tc ? launch_bwd_grads_tc(a, J, s) : launch_bwd_grads(a, J, dtype, s);
            }) != cudaSuccess)
            return GLA_ERR_CUDA;
        if (profiled(K_BWD_DG, s, [&] { return launch_bwd_dg(a, J, s); }) != cudaSuccess)
            return GLA_ERR_CUDA;
    }
    return GLA_OK;
}

// ---------------------------------------------------------------------------------------------------
// TTT-linear forward
// ---------------------------------------------------------------------------------------------------
extern "C" size_t gla_ttt_workspace_size(void) { return 256; }

extern "C" int gla_ttt_linear_fwd(const void *q, const void *k, const void *v, const float *w, const float *b,
                                  const float *eta, float scale, float eps, const float *h0, const float *hb0,
                                  float *o, float *ht, float *hbt, const int32_t *cu_seqlens, int N, int B, int T,
                                  int H, int D, int chunk, int dtype, void *workspace, size_t workspace_bytes,
                                  void *stream)
{
    const bool varlen = cu_seqlens != nullptr;
    if (dtype != GLA_F32 && dtype != GLA_BF16 && dtype != GLA_F16)
        return GLA_ERR_UNSUPPORTED;
    if ((D != 64 && D != 128) || (chunk != 16 && chunk != 32))
        return GLA_ERR_UNSUPPORTED;
    if (B < 0 || T < 0 || H <= 0 || N < 0 || (varlen ? B != 1 : N != B))
        return GLA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale) || !(eps > 0.f) || !std::isfinite(eps))
        return GLA_ERR_INVALID_ARG;
    const size_t rows = varlen ? (size_t)T : (size_t)B * T;
    if (rows * H * D >= (1ull << 31))
        return GLA_ERR_UNSUPPORTED;
    if (rows > 0 && (!q || !k || !v || !eta || !o))
        return GLA_ERR_INVALID_ARG;
    if (!w || !b)
        return GLA_ERR_INVALID_ARG;
    for (const void *p : {q, k, v, (const void *)w, (const void *)b, (const void *)eta, (const void *)h0,
                          (const void *)hb0, (const void *)o, (const void *)ht, (const void *)hbt,
                          (const void *)cu_seqlens})
        if (misaligned(p))
            return GLA_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < gla_ttt_workspace_size())
        return GLA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign)
        return GLA_ERR_ALIGNMENT;
    const size_t esz = dtype == GLA_F32 ? 4 : 2;
    const size_t sq = (size_t)N * H * D * D * 4, sb = (size_t)N * H * D * 4;
    const Range in[] = {range_of(q, rows * H * D * esz), range_of(k, rows * H * D * esz),
                        range_of(v, rows * H * D * esz), range_of(w, (size_t)H * D * 4),
                        range_of(b, (size_t)H * D * 4), range_of(eta, rows * H * 4),
                        range_of(h0, h0 ? sq : 0), range_of(hb0, hb0 ? sb : 0),
                        range_of(cu_seqlens, varlen ? sizeof(int32_t) * (size_t)(N + 1) : 0),
                        range_of(workspace, 256)};
    const Range out[] = {range_of(o, rows * H * D * 4), range_of(ht, ht ? sq : 0), range_of(hbt, hbt ? sb : 0)};
    for (size_t i = 0; i < 3; ++i) {
        for (const Range &r : in)
            if (overlap(out[i], r))
                return GLA_ERR_INVALID_ARG;
        for (size_t j2 = i + 1; j2 < 3; ++j2)
            if (overlap(out[i], out[j2]))
                return GLA_ERR_INVALID_ARG;
    }
    g_prof.launches = 0;
    const int nseq = varlen ? N : B;
    if (nseq == 0)
        return GLA_OK;
    TttArgs a;
    std::memset(&a, 0, sizeof a);
    a.q = q; a.k = k; a.v = v; a.w = w; a.b = b; a.eta = eta; a.scale = scale; a.eps = eps;
    a.h0 = h0; a.hb0 = hb0; a.o = o; a.ht = ht; a.hbt = hbt; a.cu = cu_seqlens;
    a.N = nseq; a.T = T; a.H = H; a.D = D; a.BT = chunk;
    a.status = static_cast<int *>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // bf16 q, k, v with D == 128 on the tensor cores; other shapes on the CUDA-core cluster kernel
    const bool tc = ttt_tc_supported(dtype, D, chunk);
    if (profiled(tc ? K_TTT_TC : K_TTT, s,
                 [&] { return tc ? launch_ttt_linear_tc(a, s) : launch_ttt_linear_fwd(a, dtype, s); }) != cudaSuccess)
        return GLA_ERR_CUDA;
    return GLA_OK;
}

// ---------------------------------------------------------------------------------------------------
// WY representation forward (gated delta rule)
// ---------------------------------------------------------------------------------------------------

namespace {

struct WyPlan {
    int J, NT;
    size_t off_table, off_seq, total;
};

WyPlan make_wy_plan(int B, int T, int N, int chunk, bool varlen)
{
    WyPlan wp;
    std::memset(&wp, 0, sizeof wp);
    wp.NT = varlen ? 0 : (T + chunk - 1) / chunk;
    wp.J = varlen ? N + (T + chunk - 1) / chunk : B * wp.NT;
    size_t off = kAlign;   // status header
    wp.off_table = off;
    if (varlen)
        off += align_up(sizeof(int4) * (size_t)wp.J);
    wp.off_seq = off;
    if (varlen)
        off += align_up(sizeof(int2) * (size_t)N);
    wp.total = off;
    return wp;
}

}  // namespace

extern "C" size_t gla_wy_workspace_size(int T, int N, int chunk, int varlen)
{
    if (T < 0 || N < 0 || (chunk != 16 && chunk != 32 && chunk != 64))
        return 0;
    return make_wy_plan(1, T, N, chunk, varlen != 0).total;
}

extern "C" int gla_wy_fwd(const void *k, const void *v, const void *beta, const void *A, const float *g, void *w,
                          void *u, const int32_t *cu_seqlens, int N, int B, int T, int H, int HV, int K, int V,
                          int chunk, int dtype, void *workspace, size_t workspace_bytes, void *stream)
{
    const bool varlen = cu_seqlens != nullptr;
    if (dtype != GLA_F32 && dtype != GLA_BF16 && dtype != GLA_BF16_OBF16 && dtype != GLA_F16)
        return GLA_ERR_UNSUPPORTED;
    if (B < 0 || T < 0 || H <= 0 || HV <= 0 || N < 0 || K <= 0 || V <= 0 || (varlen ? B != 1 : N != B))
        return GLA_ERR_INVALID_ARG;
    if (HV % H)
        return GLA_ERR_INVALID_ARG;
    if (!wy_supported(dtype, K, V, chunk))
        return GLA_ERR_UNSUPPORTED;
    const size_t rows = varlen ? (size_t)T : (size_t)B * T;
    if (rows * HV * (size_t)(K > V ? (K > chunk ? K : chunk) : (V > chunk ? V : chunk)) >= (1ull << 31) ||
        rows * H * K >= (1ull << 31))
        return GLA_ERR_UNSUPPORTED;
    if (rows > 0 && (!k || !v || !beta || !A || !w || !u))
        return GLA_ERR_INVALID_ARG;
    for (const void *p : {k, v, beta, A, (const void *)g, (const void *)w, (const void *)u, (const void *)cu_seqlens})
        if (misaligned(p))
            return GLA_ERR_ALIGNMENT;
    const WyPlan wp = make_wy_plan(B, T, N, chunk, varlen);
    if (!workspace || workspace_bytes < wp.total)
        return GLA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign)
        return GLA_ERR_ALIGNMENT;
    const size_t esz = dtype == GLA_F32 ? 4 : 2, osz = dtype == GLA_BF16_OBF16 ? 2 : 4;
    const Range in[] = {range_of(k, rows * H * K * esz), range_of(v, rows * HV * V * esz),
                        range_of(beta, rows * HV * esz), range_of(A, rows * HV * chunk * esz),
                        range_of(g, g ? rows * HV * 4 : 0),
                        range_of(cu_seqlens, varlen ? sizeof(int32_t) * (size_t)(N + 1) : 0),
                        range_of(workspace, wp.total)};
    const Range out[] = {range_of(w, rows * HV * K * osz), range_of(u, rows * HV * V * osz)};
    for (const Range &o : out)
        for (const Range &r : in)
            if (overlap(o, r))
                return GLA_ERR_INVALID_ARG;
    if (overlap(out[0], out[1]))
        return GLA_ERR_INVALID_ARG;
    for (size_t i = 0; i + 1 < sizeof in / sizeof in[0]; ++i)   // the workspace is written (chunk table)
        if (overlap(in[i], in[6]))
            return GLA_ERR_INVALID_ARG;
    g_prof.launches = 0;
    if ((varlen ? N : B) == 0 || rows == 0)
        return GLA_OK;
    char *ws = static_cast<char *>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WyArgs a;
    std::memset(&a, 0, sizeof a);
    a.k = k; a.v = v; a.beta = beta; a.A = A; a.g = g; a.w = w; a.u = u;
    a.B = B; a.T = T; a.H = H; a.HV = HV; a.K = K; a.V = V; a.BT = chunk; a.NT = wp.NT;
    a.status = reinterpret_cast<int *>(ws);
    if (varlen) {
        // the forward's slot planner with segments of one chunk gives the chunk table
        Args pa;
        std::memset(&pa, 0, sizeof pa);
        pa.cu = cu_seqlens; pa.N = N; pa.T = T; pa.L = chunk; pa.J = wp.J; pa.seg_cap = 0;
        pa.status = reinterpret_cast<int *>(ws);
        pa.table = reinterpret_cast<const int4 *>(ws + wp.off_table);
        pa.seqinfo = reinterpret_cast<const int2 *>(ws + wp.off_seq);
        a.table = pa.table;
        Plan pl;
        std::memset(&pl, 0, sizeof pl);
        if (profiled(K_PLAN, s, [&] { return launch_plan_varlen(pl, pa, s); }) != cudaSuccess)
            return GLA_ERR_CUDA;
    }
    // bf16 inputs with K == V in {64, 128}: tensor cores; every other case: fp32 CUDA cores
    const bool tc = wy_tc_supported(dtype, K, V);
    if (wp.J > 0 && profiled(tc ? K_WY_TC : K_WY, s, [&] {
            return tc ? launch_wy_fwd_tc(a, wp.J, dtype, s) : launch_wy_fwd(a, wp.J, dtype, s);
        }) != cudaSuccess)
        return GLA_ERR_CUDA;
    return GLA_OK;
}
