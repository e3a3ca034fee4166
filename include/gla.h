/*
 * gla.h — C ABI of libgla: the chunkwise-parallel forward pass of gated linear attention (GLA) on one
 * NVIDIA GB300 (sm_103a).
 *
 * The method (page "fla/ops/gla/fused_chunk.py": fused_chunk_gla_fwd_kernel, fwd_inner_chunk,
 * prepare_qg_kg, FusedChunkGLAFunction.forward) is the recurrence, per sequence n and head h,
 *
 *     S_0 = h0[n,h] (or 0),   S_t = diag(exp(g_t)) S_{t-1} + k_t^T v_t,   o_t = scale * q_t S_t,
 *     ht[n,h] = S_{last}
 *
 * with a per-key-dimension log-decay g_t <= 0 and a K x V state.  The library computes it chunkwise: a
 * chunk-local cumsum of g, per-segment state contributions, a decayed scan over segments, and a fused
 * output kernel that adds the inter-chunk term q~ S to the causally masked intra-chunk term.
 *
 * Conventions shared by every entry point
 *   - Layout: time-major with interleaved heads, contiguous, no strides (page
 *     "fla/ops/ttt/fused_chunk.py", fused_chunk_ttt_linear: [B, T, H, K] inputs).
 *       q, k, g : [B, T, H, K]        v, o : [B, T, H, V]        h0, ht : [N, H, K, V] fp32, row-major
 *     (K rows, V columns: the state layout of fused_chunk_gla_fwd_kernel's h0/ht blocks).
 *   - Varlen packing: cu_seqlens != NULL is a DEVICE array of N+1 int32 offsets (page
 *     "fla/ops/ttt/fused_chunk.py", fused_chunk_ttt_linear_fwd_kernel: bos/eos from cu_seqlens); then
 *     B must be 1, T is the packed total and cu_seqlens must run non-decreasing from 0 to T.  Because the
 *     offsets live on the device they are checked there; a violation is reported through
 *     gla_get_status() as GLA_ERR_INVALID_ARG and no output is written.  Zero-length sequences are
 *     allowed (their ht is h0, or 0).  Without cu_seqlens, N must equal B.
 *   - Pointers: every device pointer must be 16-byte aligned (GLA_ERR_ALIGNMENT otherwise).  The
 *     caller owns every buffer, including o, ht and the workspace; the library allocates nothing.
 *     No input may alias an output, except h0 == ht (in-place state streaming), which is allowed.
 *   - Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call is
 *     stream-ordered and returns once its kernels are enqueued; nothing synchronises the host.
 *   - Errors: synchronous validation returns a gla_status code and enqueues nothing.  Device-side
 *     conditions (bad cu_seqlens, a bounded wait that ran out) are recorded in the workspace's status
 *     word, read with gla_get_status().
 */
#ifndef GLA_H
#define GLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gla_status {
    GLA_OK = 0,
    GLA_ERR_INVALID_ARG = 1,   /* NULL/negative/inconsistent argument, bad cu_seqlens, bad scale   */
    GLA_ERR_UNSUPPORTED = 2,   /* shape or dtype outside the supported set                          */
    GLA_ERR_ALIGNMENT = 3,     /* a device pointer is not 16-byte aligned                           */
    GLA_ERR_WORKSPACE = 4,     /* workspace NULL or smaller than gla_fwd_workspace_size()           */
    GLA_ERR_CUDA = 5,          /* a CUDA runtime call or kernel launch failed                       */
    GLA_ERR_TIMEOUT = 6,       /* (device) a bounded wait inside a kernel ran out; outputs invalid  */
    GLA_ERR_RANGE = 7          /* (device) a value left the fp16 operand range of the tensor-core
                                  path (see gla_fwd); outputs invalid, use GLA_F32 inputs instead  */
} gla_status;

typedef enum gla_dtype {
    GLA_F32 = 0,        /* q, k, v, g fp32; o fp32                                                  */
    GLA_BF16 = 1,       /* q, k, v, g bf16; o fp32 (default for bf16 inputs, see below)             */
    GLA_BF16_OBF16 = 2, /* q, k, v, g bf16; o bf16 (the pages' o.to(v) convention)                  */
    GLA_F16 = 3,        /* q, k, v, g fp16; o fp32 (same paths and bounds as GLA_BF16)                */
    GLA_BF16_GF32 = 4,  /* q, k, v bf16, g fp32; o fp32 (forward: the tensor-core path for K == 128)  */
    GLA_F16_GF32 = 5    /* q, k, v fp16, g fp32; o fp32 (as GLA_BF16_GF32)                             */
} gla_dtype;

/* OR-ed into the dtype argument of gla_fwd / gla_bwd (and their workspace queries): q, k, v, g, o (and the
 * gradients) are head-first [B, H, T, *] instead of [B, T, H, *]; with cu_seqlens (B == 1) that is [1, H, T, *]
 * over the packed rows.  h0 / ht keep [N, H, K, V].  Same paths, kernels and results otherwise. */
#define GLA_HEAD_FIRST 0x100
/* o is fp32 for bf16 inputs by default: at the benchmark magnitudes (|o| up to ~20) a bf16-rounded o
 * alone carries up to 0.06 of rounding error, above the 2e-2 max-abs parity bound.  State h0/ht is fp32
 * for every dtype (fused_chunk_gla_fwd_kernel keeps the state in fp32 and stores ht as fp32). */

/*
 * gla_fwd — GLA forward over a batch (or a varlen pack) of sequences.
 *
 *   q, k, g     [B,T,H,K] input dtype (device).  g is the per-step log-decay (expected <= 0).
 *   v           [B,T,H,V] input dtype (device).
 *   o           [B,T,H,V] output (device), fp32 for GLA_F32 / GLA_BF16, bf16 for GLA_BF16_OBF16.
 *   scale       multiplies q only (prepare_qg_kg); must be finite and > 0.  ht carries no scale.
 *   h0          [N,H,K,V] fp32 initial state (device) or NULL for zeros.  It is decayed by the first
 *               token's gate like any carried state (fused_chunk_gla_fwd_kernel).
 *   ht          [N,H,K,V] fp32 final state (device) or NULL to skip it.  May equal h0.
 *   cu_seqlens  int32 [N+1] device offsets or NULL (dense: N == B sequences of T rows).
 *   chunk       chunk length: 16, 32, 64 or 128.  The result does not depend on it in exact arithmetic;
 *               the kernels tile at 64 rows whatever the value (so it selects no different rounding here).
 *   K           64 or 128.          V  64, 128 or 256.          B, T, H, N >= 0 (T*H*max(K,V) < 2^31).
 *   workspace   device scratch of at least gla_fwd_workspace_size() bytes, 256-byte aligned, ZEROED
 *               BEFORE ITS FIRST USE and not written by the caller afterwards: its 256-byte header carries
 *               the sticky status word, work counters and a launch epoch between calls (the epoch tags
 *               the segment scan's publication flags, so they need no clearing per call).  One workspace
 *               must not be used by two calls that may run concurrently.
 *
 * Paths: 16-bit q, k, v (g 16-bit or fp32) with K == 128 and V in {128, 256} run on the tcgen05 tensor cores
 * with fp16 operands and fp32 accumulation; everything else runs on fp32 CUDA cores.  Valid domain of the tensor-core path
 * (its intra-chunk scores are factorised around an anchor row in the middle of each chunk): every
 * operand it forms must stay inside the fp16 range, i.e. |q|, |k| * exp(gate sum over up to half a chunk)
 * below 65000, |v| < 65000, |state| < 65000 and intra-chunk scores below 65000 in magnitude; the kernels
 * check this and report GLA_ERR_RANGE through gla_get_status() otherwise.  The fp32 path's domain is the
 * fp32 range of the same factorisation (gate sums over half a chunk above about -80).
 * Returns GLA_OK once enqueued, else a synchronous gla_status.
 */
int gla_fwd(const void *q, const void *k, const void *v, const void *g, void *o, float scale,
            const float *h0, float *ht, const int32_t *cu_seqlens, int N, int B, int T, int H,
            int K, int V, int chunk, int dtype, void *workspace, size_t workspace_bytes,
            void *stream);

/*
 * Bytes of device workspace gla_fwd needs for this problem on the CURRENT device (the segment plan
 * depends on its SM count).  Returns 0 for arguments gla_fwd would reject.  Never fails otherwise.
 */
size_t gla_fwd_workspace_size(int B, int T, int H, int K, int V, int N, int chunk, int dtype);

/*
 * Synchronises `stream`, then returns and clears the sticky device status word of `workspace`
 * (GLA_OK if no enqueued call since the last read reported a device-side error).  Returns
 * GLA_ERR_CUDA if the synchronisation itself failed, GLA_ERR_INVALID_ARG for a NULL workspace.
 */
int gla_get_status(void *workspace, void *stream);

/* Static description of a gla_status code (never NULL). */
const char *gla_strerror(int code);

/*
 * gla_chunk_local_cumsum — the chunk-local inclusive cumsum of the log-decay as a standalone pass
 * (FusedChunkGLAFunction.forward computes it in fp32 before everything else):
 *     G[t] = sum of g[u] for u from the first row of t's chunk to t,
 * chunks of `chunk` rows starting at every sequence start (cu_seqlens, or every T rows when NULL).
 * g [B,T,H,K] in the input dtype (GLA_F32 or GLA_BF16), G [B,T,H,K] fp32, both device.  gla_fwd does
 * not call this: its kernels form the same sums on chip.  Device-side cu_seqlens errors are not
 * checked here (pass valid offsets).  chunk in {16, 32, 64, 128}.
 */
int gla_chunk_local_cumsum(const void *g, float *G, const int32_t *cu_seqlens, int N, int B, int T,
                           int H, int K, int chunk, int dtype, void *stream);

/*
 * gla_fwd_noalloc — gla_fwd without a caller-provided workspace, for callers that cannot allocate device
 * memory: host runtimes that own every device byte through their own pool and forbid other allocations
 * once running, or call paths that must not risk an allocation failure or the device-wide
 * synchronisation a cudaMalloc can cause.  It has no counterpart on the pages.
 *
 * Arguments, layouts, results and synchronous errors are those of gla_fwd.  The scratch comes from one
 * 32 MiB device array inside the library (held by every device that loads it, until exit); problems whose
 * gla_fwd_workspace_size() exceeds 32 MiB are rejected with GLA_ERR_WORKSPACE before anything is enqueued.
 * The array's device address is looked up (cudaGetSymbolAddress) with the device current on the first call
 * in each context, i.e. on the first call on a device and again after a device reset; make such a call
 * before any stream capture.  Nothing is allocated: no cudaMalloc, cudaFree or allocating library routine
 * is called, and the call enqueues only the gla_fwd kernels.  All calls share the one array, which keeps
 * the previous call's contents, so calls that may overlap on the GPU (different streams without ordering)
 * race on it and must not be made.  Device-side conditions (bad cu_seqlens, GLA_ERR_RANGE,
 * GLA_ERR_TIMEOUT) go to a status word inside the array that cannot be read back; callers that need them
 * use gla_fwd with a workspace.
 */
int gla_fwd_noalloc(const void *q, const void *k, const void *v, const void *g, void *o, float scale,
                    const float *h0, float *ht, const int32_t *cu_seqlens, int N, int B, int T, int H,
                    int K, int V, int chunk, int dtype, void *stream);

/*
 * gla_fwd_host — gla_fwd on inputs and outputs in HOST memory (a serving path whose requests arrive in host
 * memory).  It has no counterpart on the pages: the result is gla_fwd's, computed head group by head group.
 *
 * q, k, g [rows, H, K], v [rows, H, V], o [rows, H, V], h0 / ht [N, H, K, V] (fp32, each may be NULL) and
 * cu_seqlens [N + 1] (int32 or NULL) are host pointers, time-major (GLA_HEAD_FIRST is rejected with
 * GLA_ERR_UNSUPPORTED); page-locked host memory lets the copies run asynchronously and at full speed, other
 * host memory works but is copied through staging.  The other arguments are gla_fwd's.  The H heads are
 * processed in head_groups groups of H / head_groups heads (H must be a multiple of it, else
 * GLA_ERR_INVALID_ARG): while one group's kernels run, the next group's inputs are copied to the device and
 * the previous group's o (and ht) copied back, so a call takes about the time of its larger copy direction.
 * Each group runs gla_fwd with H / head_groups heads; its segment plan can differ from that of one call with
 * all H heads, so the two results agree within the arithmetic's rounding, not bit for bit.
 *
 * workspace: device memory of at least gla_fwd_host_workspace_size() bytes, 256-byte aligned, zeroed before
 * its first use (it holds gla_fwd's workspace for one group, a copy of cu_seqlens and up to three groups'
 * device buffers); gla_get_status() reads its status word.  Calls that share a workspace must be ordered on
 * the GPU (for example on one stream).  The call enqueues everything on `stream` and on two side streams of
 * its own (created on the first call from each host thread on each device, with their events, and kept until
 * exit), joined back into `stream`: the host buffers may be read or reused once `stream` has reached that
 * point.  Returns GLA_OK once enqueued, else a synchronous gla_status (GLA_ERR_WORKSPACE for a missing or
 * small workspace, GLA_ERR_CUDA if an enqueue failed; work already enqueued then still runs).
 */
int gla_fwd_host(const void *q, const void *k, const void *v, const void *g, void *o, float scale,
                 const float *h0, float *ht, const int32_t *cu_seqlens, int N, int B, int T, int H, int K,
                 int V, int chunk, int dtype, int head_groups, void *workspace, size_t workspace_bytes,
                 void *stream);

/* Bytes of device workspace gla_fwd_host needs (0 for arguments it would reject). */
size_t gla_fwd_host_workspace_size(int B, int T, int H, int K, int V, int N, int chunk, int dtype,
                                   int head_groups);

/*
 * gla_bwd — gradients of the forward above (page "fla/ops/gla/fused_chunk.py": fused_chunk_gla_bwd_kernel,
 * bwd_inner_chunk, FusedChunkGLAFunction.backward) for the loss L = sum(o * dout) + sum(ht * dht):
 *
 *   dq = dL/dq, dk = dL/dk, dg = dL/dg   [rows, H, K] fp32 (device, written)
 *   dv = dL/dv                           [rows, H, V] fp32 (device, written)
 *   dh0 = dL/dh0                         [N, H, K, V] fp32 (device) or NULL to skip it
 *
 * q, k, v, g, scale, h0, cu_seqlens, N, B, T, H, chunk: as for gla_fwd (the forward is recomputed; pass the
 * same h0 the forward used, or NULL for a zero initial state).  dout [rows, H, V] in the input dtype (the
 * gradient of o); dht [N, H, K, V] fp32 or NULL (no loss on the final state).  dtype GLA_F32 (every input
 * fp32), GLA_BF16 (q, k, v, g, dout bf16), GLA_F16, GLA_BF16_GF32 or GLA_F16_GF32 (fp32 g), optionally OR-ed
 * with GLA_HEAD_FIRST.  Arithmetic is fp32: for bf16 inputs with K == 128 the per-chunk sums and the per-chunk
 * gradients run on the tcgen05 tensor cores (fp32 operands split exactly into three bf16 terms, fp32
 * accumulation), every other step on CUDA cores.  K in {64, 128}, V in {64, 128, 256} (V = 256 runs as two
 * 128-wide value slices: dq, dk and dg are accumulated over them); chunk 16, 32, 64 or 128 (tiled at 64 rows,
 * as for gla_fwd).  workspace: at least gla_bwd_workspace_size() bytes, 256-byte aligned, zeroed before its
 * first use (status word in its first bytes); it holds the chunk-start states and chunk-end adjoints of one
 * value slice (2 * chunks * H * K * min(V, 128) fp32).  Outputs must not overlap any input, the workspace or one another.  The
 * library allocates nothing and is stream-ordered.  Errors as for gla_fwd (GLA_ERR_UNSUPPORTED for other
 * dtypes or head sizes); valid domain: the fp32 range of the same mid-chunk factorisation as the fp32
 * forward path.  Returns GLA_OK once enqueued.
 */
int gla_bwd(const void *q, const void *k, const void *v, const void *g, const void *dout, float scale,
            const float *h0, const float *dht, float *dq, float *dk, float *dv, float *dg, float *dh0,
            const int32_t *cu_seqlens, int N, int B, int T, int H, int K, int V, int chunk, int dtype,
            void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of device workspace gla_bwd needs for this problem (0 for an unsupported shape). */
size_t gla_bwd_workspace_size(int B, int T, int H, int K, int V, int N, int chunk, int dtype);

/*
 * gla_ttt_linear_fwd — TTT-linear forward, the second workload of the same chunked-state machinery (page
 * "fla/ops/ttt/fused_chunk.py": fused_chunk_ttt_linear_fwd_kernel, then the norm_residual step of
 * fused_chunk_ttt_linear).  Per (sequence, head) an inner model h [D][D], hb [D] takes one gradient step of
 * 1/2 |LN(k h + hb) * w + b + k - v|^2 per mini-batch of `chunk` rows (the result depends on `chunk`), and
 * o_i = scale q_i h_i + hb_i (dual form, rows up to i of the mini-batch), followed by o += LN(o) * w + b.
 *
 *   q, k, v     [rows, H, D] device, fp32 / bf16 / fp16 by dtype (GLA_F32, GLA_BF16, GLA_F16); K == V == D
 *   w, b        [H, D] fp32 LayerNorm weight and bias;  eta [rows, H] fp32 per-token learning rate
 *   scale > 0, eps > 0;  h0 [N, H, D, D], hb0 [N, H, D] fp32 or NULL (zeros)
 *   o           [rows, H, D] fp32 (written);  ht [N, H, D, D], hbt [N, H, D] fp32 or NULL
 *   cu_seqlens  int32 [N+1] device offsets or NULL (as gla_fwd);  D in {64, 128};  chunk in {16, 32}
 *   workspace   gla_ttt_workspace_size() bytes, 256-byte aligned, zeroed before first use (status word:
 *               bad cu_seqlens are reported there, read it with gla_get_status; those sequences are skipped)
 *
 * Rows past the end of a sequence take no part in the last mini-batch (the page's kernel adds its zero-padded
 * rows to the hb update).  fp32 CUDA cores, one thread-block cluster of D / 16 CTAs per (sequence, head).
 * Errors as for gla_fwd; a bounded wait inside the kernel that ran out is reported as GLA_ERR_TIMEOUT in
 * the status word (the outputs of that call are then void).
 */
int gla_ttt_linear_fwd(const void *q, const void *k, const void *v, const float *w, const float *b,
                       const float *eta, float scale, float eps, const float *h0, const float *hb0, float *o,
                       float *ht, float *hbt, const int32_t *cu_seqlens, int N, int B, int T, int H, int D,
                       int chunk, int dtype, void *workspace, size_t workspace_bytes, void *stream);
size_t gla_ttt_workspace_size(void);

/*
 * Measurement hook (no counterpart on the pages; it exists so a benchmark can time each kernel of the
 * path with CUDA events on the stream the kernels run on).  While `events` is non-NULL, every later
 * gla_fwd / gla_bwd call made from this host thread records events[2i] right before and events[2i+1] right after
 * its i-th kernel launch (for i < n_events / 2), on the call's stream, and stores that launch's kernel id
 * in kernel_ids[i] (host array of n_events / 2 ints, may be NULL).  `events` are cudaEvent_t handles
 * created by the caller.  Pass events == NULL to stop.  Returns GLA_OK, or GLA_ERR_INVALID_ARG for
 * n_events < 0.  gla_profile_launches() returns how many kernels the last gla_fwd / gla_bwd call on this
 * thread launched, and gla_kernel_name() names a kernel id.
 */
int gla_profile_events(void **events, int n_events, int *kernel_ids);
int gla_profile_launches(void);
const char *gla_kernel_name(int kernel_id);

/*
 * gla_wy_fwd — WY representation forward of the gated delta rule, a third chunked workload (page
 * "fla/ops/gated_delta_rule/backends/triton_ascend/wy_fast.py": recompute_w_u_fwd_kernel_npu and its launcher
 * recompute_w_u_fwd_npu).  Each sequence is cut into chunks of `chunk` rows from its first row (the last one
 * may be partial).  For value head hv, whose key head is hv / (HV / H), and row t of chunk [c0, c1):
 *
 *   u_t = sum_{s in [c0, c1)} A_t[s - c0] beta_s v_s,   w_t = sum_{s in [c0, c1)} A_t[s - c0] beta_s 2^{g_s} k_s
 *
 *   k      [rows, H, K] device, input dtype          v     [rows, HV, V] device, input dtype
 *   beta   [rows, HV]   device, input dtype          A     [rows, HV, chunk] device, input dtype: row t holds
 *                                                           row t - c0 of its chunk's matrix (full square)
 *   g      [rows, HV] fp32 log2-domain gate (the factor is 2^g) or NULL (factor 1)
 *   w      [rows, HV, K], u [rows, HV, V] device, written: fp32, or bf16 for GLA_BF16_OBF16
 *   rows = B * T (dense) or the packed length T (varlen: cu_seqlens int32 [N+1] on the device, B == 1,
 *   cu_seqlens[N] == T; bad offsets are reported in the status word and no row is written)
 *   dtype  GLA_F32, GLA_BF16 (fp32 outputs), GLA_BF16_OBF16 or GLA_F16 (fp32 outputs);  K, V in {64, 128};
 *   HV a multiple of H;  chunk in {16, 32, 64}
 *   workspace  at least gla_wy_workspace_size(T, N, chunk) bytes, 256-byte aligned, zeroed before its first
 *              use (status word, then the varlen chunk table)
 *
 * Rows past the end of a sequence do not exist: the columns of A that would refer to them are not read.
 * bf16 inputs with K == V in {64, 128} run on the tcgen05 tensor cores (the fp32 operand k * beta * 2^g |
 * v * beta split into three bf16 terms, A as it is stored, fp32 accumulation; a bounded wait inside reports
 * GLA_ERR_TIMEOUT in the status word); everything else on fp32 CUDA cores.  Outputs must not overlap any
 * input, the workspace or each other.  Errors as for gla_fwd; returns GLA_OK once enqueued.
 */
int gla_wy_fwd(const void *k, const void *v, const void *beta, const void *A, const float *g, void *w, void *u,
               const int32_t *cu_seqlens, int N, int B, int T, int H, int HV, int K, int V, int chunk, int dtype,
               void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of device workspace gla_wy_fwd needs (dense batches: N is ignored). */
size_t gla_wy_workspace_size(int T, int N, int chunk, int varlen);

#ifdef __cplusplus
}
#endif
#endif /* GLA_H */
