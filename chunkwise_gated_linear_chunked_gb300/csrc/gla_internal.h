// Internal declarations shared by the translation units of libgla (host planner + kernels).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "gla.h"

namespace gla {

constexpr int kChunk = 64;          // chunk length C (rows per intra-chunk tile)
constexpr int kSegRows = 2048;      // varlen packs: most rows of one segment on the tensor-core path
constexpr int kPieceChunks = 16;    // dense balanced pieces: fewest chunks of a piece

// One forward call's launch plan.  Segments of L rows (L a multiple of the chunk) split each sequence
// so that long sequences with few heads still fill the GPU; a "slot" is one (sequence, segment) pair and
// carries all H heads.  Slots of one sequence are contiguous.
struct Plan {
    int B, T, H, K, V, N, chunk, dtype;
    bool varlen;
    int L;        // segment length in rows (multiple of chunk)
    int P;        // dense: segments per sequence (>= 1), or per (sequence, head) unit with pieces;
                  // varlen: 0 (per sequence, from the plan kernel)
    int J;        // slots: exact (dense) or an upper bound (varlen)
    int np;       // dense, tensor cores: the units' chunks cut into np balanced pieces (0: segments of L)
    int nc;       // chunks per sequence (pieces only)
    bool multi;   // some sequence may span more than one segment: state + scan passes are needed
    bool tc;      // tensor-core path (bf16 inputs, K == 128, V multiple of 128)
    int BV, NV;   // value-tile width and count (64 on CUDA cores, 128 on tensor cores)
    // workspace layout (byte offsets)
    size_t off_status, off_table, off_seq, off_ss, off_agg, off_gtot, off_ctr, off_flags, total;
};

// Kernel arguments (passed by value).
struct Args {
    const void *q, *k, *v, *g;
    void *o;
    const float *h0;
    float *ht;
    const int32_t *cu;     // device offsets or nullptr
    float scale;
    int B, T, H, K, V, N, L, P, J;
    int seg_cap;           // varlen: most segments per sequence (the segment length grows to respect it)
    int hf;                // head-first layout [B, H, T, *] of q, k, v, g, o (dense batches only)
    int lb;                // fused tensor kernel: segments per block of the start-state scan
    int sms;               // varlen plan for the tensor-core kernel: SM count (0: fixed segments of L rows)
    int np, nc;            // dense balanced pieces (tensor cores): piece count (0: off), chunks per sequence
    const int4 *table;     // varlen: per slot {n, p, bos, eos}; n < 0 marks an unused slot
    const int2 *seqinfo;   // varlen: per sequence {first slot, slot count}
    float *ss;             // CUDA cores: [J][H][K][V] segment contributions, then segment start states;
                           // tensor cores: [J][H][NV] tiles of the segment end states (key-interleaved)
    float *agg;            // tensor cores: [J][H][NV] tiles of the segment contributions (key-interleaved)
    float *gtot;           // CUDA cores: [J][H][K]; tensor cores: [J][H][NV][K]: total log-decay of a segment
    int *ctr;              // fused tensor kernel: [0] next work item, [1] finished CTAs (both zero between
                           // calls), [2] launch epoch (advanced by every launch)
    int *flags;            // fused tensor kernel: per work item (epoch << 2) | 1 once its segment contribution
                           // and decay are published, (epoch << 2) | 2 once its segment end state is
    int *status;           // sticky device status word
};

// Row-head index of packed row `row` (b*T + t for a dense batch) and head h: time-major [rows, H, *] or
// head-first [B, H, T, *] (dense batches only).  Multiply by the row width and add the column.
__device__ __forceinline__ size_t row_head(int row, int h, int H, int T, int hf)
{
    if (!hf)
        return (size_t)row * H + h;
    const int b = row / T;
    return ((size_t)b * H + h) * T + (row - b * T);
}

// Backward kernel arguments (passed by value).  Chunk slots: dense j = n * NC + c; varlen from the slot
// table (plan_varlen with 64-row segments).
struct BwdArgs {
    const void *q, *k, *v, *g, *dout;
    const float *h0, *dht;
    float *dq, *dk, *dv, *dg, *dh0;   // fp32 outputs; dh0 may be nullptr
    float scale;
    int B, T, H, K, V, N, NC;
    int hf;                           // head-first layout [B, H, T, *] of inputs and gradients (dense only)
    const int4 *table;                // varlen: per chunk slot {n, p, bos, eos}; n < 0 marks an unused slot
    const int2 *seqinfo;              // varlen: per sequence {first slot, slot count}
    float *dS;                        // [J][H][K][V]: chunk contributions, then chunk-start states
    float *dR;                        // [J][H][K][V]: adjoint contributions, then chunk-end adjoints
    float *gl;                        // [J][H][K]: chunk total log-decay (natural log)
    float *ht;                        // [N][H][K][V]: final states
    float *dgt;                       // [J][H][K]: chunk sums of q dq - k dk, then their carries
    int ldv;                          // row stride (elements) of v, dout and dv: V, or the full width when the
                                      // call runs as 128-wide value slices (v, dout, dv then point at the slice)
    int lds;                          // row stride of the rows of h0, dht and dh0 ([N][H][K][lds], likewise)
    int acc;                          // add into dq, dk and dg (a second value slice) instead of writing
    int *status;
};

// Map slot j to (sequence n, segment p, rows [bos, eos), sequence end).  False for an unused slot.
__device__ __forceinline__ bool resolve_slot(const Args &a, int j, int &n, int &p, int &bos, int &eos,
                                             int &send)
{
    if (a.table) {
        const int4 e = a.table[j];
        if (e.x < 0)
            return false;
        n = e.x;
        p = e.y;
        bos = e.z;
        eos = e.w;
        send = a.cu[n + 1];
        return true;
    }
    n = j / a.P;
    p = j - n * a.P;
    const int sb = n * a.T;
    bos = sb + p * a.L;
    send = sb + a.T;
    eos = min(bos + a.L, send);
    return true;
}

__device__ __forceinline__ void report(int *status, int code)
{
    if (status)
        atomicCAS(status, 0, code);
}

// Launchers (return cudaGetLastError() after the launch).
cudaError_t launch_plan_varlen(const Plan &pl, const Args &a, cudaStream_t s);
cudaError_t launch_state_ffma(const Plan &pl, const Args &a, cudaStream_t s);
cudaError_t launch_scan(const Plan &pl, const Args &a, cudaStream_t s);
cudaError_t launch_out_ffma(const Plan &pl, const Args &a, cudaStream_t s);
bool tc_supported(int dtype, int K, int V);
cudaError_t launch_fused_tc(const Plan &pl, const Args &a, cudaStream_t s, int sms);
// TTT-linear forward arguments (passed by value).
struct TttArgs {
    const void *q, *k, *v;            // [rows, H, D]
    const float *w, *b;               // [H, D] LayerNorm weight and bias
    const float *eta;                 // [rows, H] per-token learning rate
    float scale, eps;
    const float *h0, *hb0;            // [N, H, D, D], [N, H, D] or nullptr
    float *o, *ht, *hbt;              // [rows, H, D] fp32; final states or nullptr
    const int32_t *cu;                // varlen offsets or nullptr
    int N, T, H, D, BT;
    int *status;
};
cudaError_t launch_ttt_linear_fwd(const TttArgs &a, int dtype, cudaStream_t s);
bool ttt_tc_supported(int dtype, int D, int BT);
cudaError_t launch_ttt_linear_tc(const TttArgs &a, cudaStream_t s);

// WY representation forward arguments (passed by value).  Chunk slots: dense j = n * NT + p; varlen from
// the slot table (plan_varlen with segments of BT rows).
struct WyArgs {
    const void *k, *v, *beta, *A;     // [rows, H, K], [rows, HV, V], [rows, HV], [rows, HV, BT]
    const float *g;                   // [rows, HV] log2-domain gate or nullptr
    void *w, *u;                      // [rows, HV, K], [rows, HV, V]
    int B, T, H, HV, K, V, BT, NT;
    const int4 *table;                // varlen: per chunk slot {n, p, bos, eos}; n < 0 marks an unused slot
    int *status;                      // sticky device status word
};
bool wy_supported(int dtype, int K, int V, int BT);
cudaError_t launch_wy_fwd(const WyArgs &a, int J, int dtype, cudaStream_t s);
bool wy_tc_supported(int dtype, int K, int V);
cudaError_t launch_wy_fwd_tc(const WyArgs &a, int J, int dtype, cudaStream_t s);

bool bwd_supported(int dtype, int K, int V);
cudaError_t launch_bwd_sums(const BwdArgs &a, int J, int dtype, cudaStream_t s);
bool bwd_sums_tc_supported(int dtype, int K, int V);
cudaError_t launch_bwd_sums_tc(const BwdArgs &a, int J, int dtype, cudaStream_t s);
cudaError_t launch_bwd_scan(const BwdArgs &a, cudaStream_t s);
cudaError_t launch_bwd_grads(const BwdArgs &a, int J, int dtype, cudaStream_t s);
bool bwd_grads_tc_supported(int dtype, int K, int V);
cudaError_t launch_bwd_grads_tc(const BwdArgs &a, int J, cudaStream_t s);
cudaError_t launch_bwd_dg(const BwdArgs &a, int J, cudaStream_t s);
cudaError_t launch_chunk_cumsum(const void *g, float *G, const int32_t *cu, int N, int B, int T, int H,
                                int K, int chunk, int dtype, cudaStream_t s);

}  // namespace gla
