// gla_fwd_host: the forward on inputs and outputs in host memory, pipelined by head groups.
//
// Heads are independent problems, so a call is split into G groups of H / G heads.  A group's rows are a
// strided slice of the time-major host tensors ([rows][H][D], the group's heads contiguous inside each row),
// copied with one two-dimensional copy per tensor into compact [rows][H/G][D] device buffers, computed by
// gla_fwd with H / G heads, and its o (and ht) copied back the same way.  Three slots of device buffers let
// the host-to-device copy of group i + 1, the kernels of group i and the device-to-host copy of group i - 1
// run at the same time (the copy engines move both directions at once), so the call takes about the time of
// its larger copy direction instead of the sum of both copies and the kernels.
#include <cstdint>

#include <cuda_runtime.h>

#include "gla.h"

namespace {

constexpr int kSlots = 3;
constexpr size_t kAlign = 256;

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// The device layout of the workspace: gla_fwd's own workspace (shared by the groups, which run in order on
// the caller's stream), the device copy of cu_seqlens, then `slots` slots of one group's q, k, v, g, h0, o, ht
// (offsets inside a slot; slot s starts at `slot` + s * `per`).
struct HostLayout {
    size_t wsz, cu, slot, per, q, k, v, g, h0, o, ht, total;
    int Hg, slots;
};

bool host_layout(HostLayout &L, int B, int T, int H, int K, int V, int N, int chunk, int dtype, int groups)
{
    if (groups <= 0 || H <= 0 || H % groups != 0 || (dtype & GLA_HEAD_FIRST))
        return false;
    const int Hg = H / groups;
    const size_t w = gla_fwd_workspace_size(B, T, Hg, K, V, N, chunk, dtype);
    if (w == 0)
        return false;
    const bool f32 = dtype == GLA_F32;
    const size_t esz = f32 ? 4 : 2, osz = dtype == GLA_BF16_OBF16 ? 2 : 4;
    const size_t gsz = (f32 || dtype == GLA_BF16_GF32 || dtype == GLA_F16_GF32) ? 4 : 2;
    const size_t rows = (size_t)B * T;   // dense: B*T; varlen (B == 1): T
    const size_t state = (size_t)N * Hg * K * V * 4;
    L.Hg = Hg;
    L.slots = groups < kSlots ? groups : kSlots;
    L.wsz = up(w);
    L.cu = L.wsz;
    L.slot = L.cu + up(((size_t)N + 1) * 4);
    L.q = 0;
    L.k = L.q + up(rows * Hg * K * esz);
    L.v = L.k + up(rows * Hg * K * esz);
    L.g = L.v + up(rows * Hg * V * esz);
    L.h0 = L.g + up(rows * Hg * K * gsz);
    L.o = L.h0 + up(state);
    L.ht = L.o + up(rows * Hg * V * osz);
    L.per = L.ht + up(state);
    L.total = L.slot + L.per * L.slots;
    return true;
}

// Two side streams (host-to-device, device-to-host) and the pipeline's events, per host thread and device:
// made on the first call and kept, so a call creates nothing after that.
struct Pipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t fork = nullptr, in_ready[kSlots] = {}, comp_done[kSlots] = {}, out_done[kSlots] = {};
};
constexpr int kMaxDevices = 64;
thread_local Pipe t_pipes[kMaxDevices];

Pipe *pipe_for_current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    Pipe &p = t_pipes[dev];
    if (p.ready)
        return &p;
    bool ok = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.fork, cudaEventDisableTiming) == cudaSuccess;
    for (int s = 0; ok && s < kSlots; ++s)
        ok = cudaEventCreateWithFlags(&p.in_ready[s], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p.comp_done[s], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p.out_done[s], cudaEventDisableTiming) == cudaSuccess;
    if (!ok)
        return nullptr;
    p.ready = true;
    return &p;
}

}  // namespace

extern "C" size_t gla_fwd_host_workspace_size(int B, int T, int H, int K, int V, int N, int chunk, int dtype,
                                              int head_groups)
{
    HostLayout L;
    return host_layout(L, B, T, H, K, V, N, chunk, dtype, head_groups) ? L.total : 0;
}

extern "C" int gla_fwd_host(const void *q, const void *k, const void *v, const void *g, void *o, float scale,
                            const float *h0, float *ht, const int32_t *cu_seqlens, int N, int B, int T, int H,
                            int K, int V, int chunk, int dtype, int head_groups, void *workspace,
                            size_t workspace_bytes, void *stream)
{
    if (dtype & GLA_HEAD_FIRST)
        return GLA_ERR_UNSUPPORTED;
    const bool varlen = cu_seqlens != nullptr;
    if (head_groups <= 0 || H <= 0 || H % head_groups != 0 || B < 0 || T < 0 || N < 0 ||
        (varlen ? B != 1 : N != B) || !(scale > 0.f))
        return GLA_ERR_INVALID_ARG;
    HostLayout L;
    if (!host_layout(L, B, T, H, K, V, N, chunk, dtype, head_groups))
        return GLA_ERR_UNSUPPORTED;   // a dtype, K, V or chunk gla_fwd does not take
    const size_t rows = varlen ? (size_t)T : (size_t)B * T;
    if (rows > 0 && (!q || !k || !v || !g || !o))
        return GLA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < L.total)
        return GLA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1))
        return GLA_ERR_ALIGNMENT;
    Pipe *pp = pipe_for_current_device();
    if (!pp)
        return GLA_ERR_CUDA;
    Pipe &P = *pp;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool f32 = dtype == GLA_F32;
    const size_t esz = f32 ? 4 : 2, osz = dtype == GLA_BF16_OBF16 ? 2 : 4;
    const size_t gsz = (f32 || dtype == GLA_BF16_GF32 || dtype == GLA_F16_GF32) ? 4 : 2;
    const int Hg = L.Hg, G = head_groups, S = L.slots;
    const size_t stateg = (size_t)Hg * K * V * 4, statep = (size_t)H * K * V * 4;
    char *ws = static_cast<char *>(workspace);
    const size_t per = L.per;
    int32_t *dcu = varlen ? reinterpret_cast<int32_t *>(ws + L.cu) : nullptr;

    auto ck = [](cudaError_t e) { return e == cudaSuccess; };
    bool ok = ck(cudaEventRecord(P.fork, s)) && ck(cudaStreamWaitEvent(P.h2d, P.fork, 0)) &&
              ck(cudaStreamWaitEvent(P.d2h, P.fork, 0));
    if (ok && varlen)
        ok = ck(cudaMemcpyAsync(dcu, cu_seqlens, ((size_t)N + 1) * 4, cudaMemcpyHostToDevice, s));
    if (!ok)
        return GLA_ERR_CUDA;
    // a [rows][H][D] host tensor's group slice <-> a compact [rows][Hg][D] device buffer
    auto slice_in = [&](void *dst, const void *src, int D, size_t el, int grp) {
        if (rows == 0)
            return true;
        const size_t w = (size_t)Hg * D * el;
        return ck(cudaMemcpy2DAsync(dst, w, static_cast<const char *>(src) + (size_t)grp * w, (size_t)H * D * el, w,
                                    rows, cudaMemcpyHostToDevice, P.h2d));
    };
    for (int i = 0; i < G && ok; ++i) {
        const int sl = i % S;
        char *b = ws + L.slot + (size_t)sl * per;
        // the slot's previous group has been copied out (and with that, computed)
        if (i >= S)
            ok = ck(cudaStreamWaitEvent(P.h2d, P.out_done[sl], 0));
        ok = ok && slice_in(b + L.q, q, K, esz, i) && slice_in(b + L.k, k, K, esz, i) &&
             slice_in(b + L.v, v, V, esz, i) && slice_in(b + L.g, g, K, gsz, i);
        if (ok && h0 && N > 0)
            ok = ck(cudaMemcpy2DAsync(b + L.h0, stateg, reinterpret_cast<const char *>(h0) + (size_t)i * stateg,
                                      statep, stateg, N, cudaMemcpyHostToDevice, P.h2d));
        ok = ok && ck(cudaEventRecord(P.in_ready[sl], P.h2d)) && ck(cudaStreamWaitEvent(s, P.in_ready[sl], 0));
        if (!ok)
            break;
        const int rc = gla_fwd(b + L.q, b + L.k, b + L.v, b + L.g, b + L.o, scale,
                               h0 ? reinterpret_cast<const float *>(b + L.h0) : nullptr,
                               ht ? reinterpret_cast<float *>(b + L.ht) : nullptr, dcu, N, B, T, Hg, K, V, chunk,
                               dtype, ws, L.wsz, s);
        if (rc != GLA_OK)
            return rc;
        ok = ck(cudaEventRecord(P.comp_done[sl], s)) && ck(cudaStreamWaitEvent(P.d2h, P.comp_done[sl], 0));
        if (ok && rows > 0) {
            const size_t w = (size_t)Hg * V * osz;
            ok = ck(cudaMemcpy2DAsync(static_cast<char *>(o) + (size_t)i * w, (size_t)H * V * osz, b + L.o, w, w,
                                      rows, cudaMemcpyDeviceToHost, P.d2h));
        }
        if (ok && ht && N > 0)
            ok = ck(cudaMemcpy2DAsync(reinterpret_cast<char *>(ht) + (size_t)i * stateg, statep, b + L.ht, stateg,
                                      stateg, N, cudaMemcpyDeviceToHost, P.d2h));
        ok = ok && ck(cudaEventRecord(P.out_done[sl], P.d2h));
    }
    // the caller's stream resumes once the last group's outputs are in host memory (the copy streams run in
    // order, so that covers every group)
    ok = ok && ck(cudaStreamWaitEvent(s, P.out_done[(G - 1) % S], 0));
    return ok ? GLA_OK : GLA_ERR_CUDA;
}
