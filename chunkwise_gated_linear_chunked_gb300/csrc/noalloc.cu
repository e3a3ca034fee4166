// gla_fwd_noalloc: gla_fwd for callers that cannot allocate device memory.  The scratch that gla_fwd
// otherwise takes from the caller (the status word, the varlen slot table, the per-segment states of the
// segment scan) lives in one file-scope device array instead.
#include <mutex>

#include "gla_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;   // 32 MiB, held on every device that loads this module

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[256];   // device address of g_scratch, per device ordinal

}  // namespace

extern "C" int gla_fwd_noalloc(const void *q, const void *k, const void *v, const void *g, void *o, float scale,
                               const float *h0, float *ht, const int32_t *cu_seqlens, int N, int B, int T,
                               int H, int K, int V, int chunk, int dtype, void *stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256)
        return GLA_ERR_CUDA;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_scratch_ptr[dev]) {
            // In host code g_scratch names a host-side stand-in; the kernels need its device address.
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p)
                return GLA_ERR_CUDA;
            g_scratch_ptr[dev] = p;
        }
        scratch = g_scratch_ptr[dev];
    }
    const size_t need = gla_fwd_workspace_size(B, T, H, K, V, N, chunk, dtype);
    if (need > kScratchBytes)
        return GLA_ERR_WORKSPACE;
    // The array keeps the previous call's contents; only the status word (the header's first 16 bytes) must
    // start at zero.  The work counters and the launch epoch behind it carry over between calls.
    if (need > 0 && cudaMemsetAsync(scratch, 0, 16, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GLA_ERR_CUDA;
    return gla_fwd(q, k, v, g, o, scale, h0, ht, cu_seqlens, N, B, T, H, K, V, chunk, dtype, scratch,
                   kScratchBytes, stream);
}
