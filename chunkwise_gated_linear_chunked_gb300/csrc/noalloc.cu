// gla_fwd_noalloc: gla_fwd for callers that cannot allocate device memory.  The scratch that gla_fwd
// otherwise takes from the caller (the status word, the varlen slot table, the per-segment states of the
// segment scan) lives in one file-scope device array instead.
#include <cudaTypedefs.h>

#include <mutex>

#include "gla_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;   // 32 MiB, held on every device that loads this module

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// The array's device address is a property of the context the module was loaded into: a device reset (or
// the primary context being released and created again) reloads the module, possibly elsewhere.  The
// address is therefore cached together with the ID of the context it was looked up in, and looked up again
// when the current context's ID differs.  The two driver calls come through the runtime's entry-point query,
// so the library does not link the driver library itself.
struct Cached {
    unsigned long long ctx_id = 0;
    void *ptr = nullptr;
};
std::mutex g_mu;
Cached g_cache[256];   // per device ordinal

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

template <typename Fn>
Fn driver_fn(const char *name, int version)
{
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}

// ID of the current context (0 if it cannot be told, e.g. before the runtime has made one current).
unsigned long long current_context_id()
{
    static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 4000);
    static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

}  // namespace

extern "C" int gla_fwd_noalloc(const void *q, const void *k, const void *v, const void *g, void *o, float scale,
                               const float *h0, float *ht, const int32_t *cu_seqlens, int N, int B, int T,
                               int H, int K, int V, int chunk, int dtype, void *stream)
{
    const size_t need = gla_fwd_workspace_size(B, T, H, K, V, N, chunk, dtype);
    if (need > kScratchBytes)
        return GLA_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256)
        return GLA_ERR_CUDA;
    const unsigned long long id = current_context_id();   // 0 before the runtime has made a context current
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        Cached &c = g_cache[dev];
        if (!c.ptr || id == 0 || c.ctx_id != id) {
            // In host code g_scratch names a host-side stand-in; the kernels need its device address.
            // (the lookup makes the device's primary context current if none was)
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p)
                return GLA_ERR_CUDA;
            c.ptr = p;
            c.ctx_id = current_context_id();
        }
        scratch = c.ptr;
    }
    // gla_fwd checks every argument before it enqueues anything.  The array keeps the previous call's
    // contents: the work counters and the launch epoch in its header carry over between calls like in any
    // other workspace (they are left consistent by every launch), and the sticky status word keeps the first
    // device-side error of any call; it cannot be read back through this entry point.
    return gla_fwd(q, k, v, g, o, scale, h0, ht, cu_seqlens, N, B, T, H, K, V, chunk, dtype, scratch,
                   kScratchBytes, stream);
}
