/*
 * Oracle for the gated linear attention (GLA) forward and backward passes — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, step-by-step fp64 CPU implementation.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library; the CUDA library never links or calls it and
 * shares no code with it.
 *
 * What it computes (the GLA recurrence; the chunked kernels of
 * "fla/ops/gla/fused_chunk.py" (fused_chunk_gla_fwd_kernel, fwd_inner_chunk) are an exact
 * re-association of it):
 *
 *     S_0     = h0[n,h]            (or 0)                          K x V state
 *     S_t     = diag(exp(g_t)) S_{t-1} + k_t^T v_t                 decay first, then the token's own term
 *     o_t     = scale * q_t S_t
 *     ht[n,h] = S_last
 *
 * Inputs are read in their stored type (fp32, fp16, or bf16 stored as raw 16-bit words) and widened exactly
 * to double element by element; nothing is rounded on the way.  Layouts are time-major with interleaved
 * heads: q, k, g are [rows, H, K] and v, o are [rows, H, V] where rows = B*T (dense) or the packed
 * total length (varlen, B == 1).  h0 / ht are [N, H, K, V] in double (an fp32 h0 widens exactly).
 *
 * Readings of the pages taken here (each one also listed in the design notes):
 *   - decay is applied before the token's own k^T v is added, and q_t sees S_t including token t
 *     (the inclusive diagonal of fwd_inner_chunk, and k*exp(G_last-G) being k at the last position in
 *     prepare_qg_kg);
 *   - scale multiplies q only, so ht carries no scale;
 *   - h0 is decayed by the first token's gate like any carried state (fused_chunk_gla_fwd_kernel);
 *   - varlen sequences are independent, a zero-length sequence gives ht = h0 (or 0).
 * The chunk size does not enter: the result is the same for every chunking in exact arithmetic.
 *
 * Also here: the chunk-local inclusive cumsum of g (chunk_local_cumsum as called by
 * FusedChunkGLAFunction.forward), with chunks aligned to each sequence's first token, and the backward
 * pass of the same recurrence by plain reverse-mode differentiation (oracle_gla_bwd, below).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2, ORACLE_F16 = 3 };

/* IEEE binary16 bit pattern to double, exactly: sign, 5-bit exponent (bias 15), 10-bit fraction. */
static double half_bits_to_double(uint16_t b)
{
    const int sign = b >> 15, e = (b >> 10) & 0x1f, f = b & 0x3ff;
    double x;
    if (e == 0)
        x = ldexp((double)f, -24);                       /* subnormal: f * 2^-24 */
    else if (e == 31)
        x = f ? NAN : INFINITY;
    else
        x = ldexp((double)(f | 0x400), e - 25);          /* (1 + f/1024) * 2^(e-15) */
    return sign ? -x : x;
}

/* Exact widening of one stored element to double. bf16 is the high half of an IEEE binary32; fp64 inputs
 * (used by the finite-difference checks of the backward) are read as they are. */
static double widen(const void *base, size_t idx, int dtype)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[idx];
    if (dtype == ORACLE_F64)
        return ((const double *)base)[idx];
    if (dtype == ORACLE_F16)
        return half_bits_to_double(((const uint16_t *)base)[idx]);
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

typedef struct {
    const void *q, *k, *v, *g;
    int dtype;
    const double *h0;         /* [N,H,K,V] or NULL */
    double *o;                /* [rows,H,V] */
    double *ht;               /* [N,H,K,V] or NULL */
    const int32_t *cu;        /* host [N+1] */
    int N, H, K, V;
    double scale;
    int next;                 /* shared work counter, guarded by mu */
    pthread_mutex_t mu;
} fwd_job;

static void run_one(fwd_job *J, int item, double *S)
{
    const int n = item / J->H, h = item % J->H;
    const int H = J->H, K = J->K, V = J->V;
    const long bos = J->cu[n], eos = J->cu[n + 1];

    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j)
            S[(size_t)i * V + j] = J->h0 ? J->h0[(((size_t)n * H + h) * K + i) * V + j] : 0.0;

    for (long t = bos; t < eos; ++t) {
        const size_t kb = ((size_t)t * H + h) * K, vb = ((size_t)t * H + h) * V;
        for (int i = 0; i < K; ++i) {
            const double decay = exp(widen(J->g, kb + i, J->dtype));
            const double ki = widen(J->k, kb + i, J->dtype);
            double *row = S + (size_t)i * V;
            for (int j = 0; j < V; ++j)
                row[j] = decay * row[j] + ki * widen(J->v, vb + j, J->dtype);
        }
        for (int j = 0; j < V; ++j) {
            double acc = 0.0;
            for (int i = 0; i < K; ++i)
                acc += widen(J->q, kb + i, J->dtype) * S[(size_t)i * V + j];
            J->o[vb + j] = J->scale * acc;
        }
    }
    if (J->ht)
        memcpy(J->ht + ((size_t)n * H + h) * K * V, S, sizeof(double) * (size_t)K * V);
}

static void *worker(void *arg)
{
    fwd_job *J = (fwd_job *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)J->K * J->V);
    if (!S)
        return (void *)1;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int item = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (item >= J->N * J->H)
            break;
        run_one(J, item, S);
    }
    free(S);
    return NULL;
}

static int resolve_threads(int nthreads, int items)
{
    if (nthreads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = c > 0 ? (int)c : 1;
    }
    if (nthreads > items)
        nthreads = items;
    return nthreads < 1 ? 1 : nthreads;
}

/*
 * Step-by-step fp64 recurrence.  cu_seqlens is a HOST array of N+1 offsets into the packed rows; pass
 * NULL for the dense batch (then N = B sequences of T rows each).  Returns the number of threads used,
 * or a negative value on bad arguments / allocation failure.
 */
int oracle_gla_fwd(const void *q, const void *k, const void *v, const void *g, int dtype,
                   const double *h0, double *o, double *ht, const int32_t *cu_seqlens, int N,
                   int B, int T, int H, int K, int V, double scale, int nthreads)
{
    if (!q || !k || !v || !g || !o || H <= 0 || K <= 0 || V <= 0 || B < 0 || T < 0)
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64 && dtype != ORACLE_F16)
        return -1;
    int32_t *dense = NULL;
    const int32_t *cu = cu_seqlens;
    if (!cu) {
        N = B;
        dense = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N + 1));
        if (!dense)
            return -2;
        for (int n = 0; n <= N; ++n)
            dense[n] = n * T;
        cu = dense;
    }
    if (N == 0) {
        free(dense);
        return 0;
    }
    fwd_job J = {q, k, v, g, dtype, h0, o, ht, cu, N, H, K, V, scale, 0, PTHREAD_MUTEX_INITIALIZER};
    const int nt = resolve_threads(nthreads, N * H);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    int rc = nt;
    if (!tid) {
        free(dense);
        return -2;
    }
    int started = 0;
    for (; started < nt; ++started)
        if (pthread_create(&tid[started], NULL, worker, &J) != 0)
            break;
    if (started == 0)
        worker(&J);
    for (int i = 0; i < started; ++i) {
        void *res = NULL;
        pthread_join(tid[i], &res);
        if (res)
            rc = -2;
    }
    free(tid);
    free(dense);
    return started ? rc : 1;
}

/*
 * Chunk-local inclusive cumsum of the log-decay: G[t] = sum of g[u] for u from the start of t's chunk
 * to t, where chunks of `chunk` rows start at each sequence's first row.  Single-threaded fp64.
 */
int oracle_chunk_local_cumsum(const void *g, int dtype, double *G, const int32_t *cu_seqlens, int N,
                              int B, int T, int H, int K, int chunk)
{
    if (!g || !G || H <= 0 || K <= 0 || chunk <= 0)
        return -1;
    const int nseq = cu_seqlens ? N : B;
    for (int n = 0; n < nseq; ++n) {
        const long bos = cu_seqlens ? cu_seqlens[n] : (long)n * T;
        const long eos = cu_seqlens ? cu_seqlens[n + 1] : (long)n * T + T;
        for (int h = 0; h < H; ++h)
            for (int i = 0; i < K; ++i) {
                double run = 0.0;
                for (long t = bos; t < eos; ++t) {
                    if ((t - bos) % chunk == 0)
                        run = 0.0;
                    const size_t idx = ((size_t)t * H + h) * K + i;
                    run += widen(g, idx, dtype);
                    G[idx] = run;
                }
            }
    }
    return 0;
}

/*
 * Backward pass of the recurrence above, by reverse-mode differentiation of its steps (the pages' chunked
 * backward, fused_chunk_gla_bwd_kernel and bwd_inner_chunk of "fla/ops/gla/fused_chunk.py", is a
 * re-association of the same gradients).  For the loss L = sum(o * do) + sum(ht * dht):
 *
 *     A_t      = dL/dS_t (everything after S_t included):   A_last = dht + scale q_last^T do_last,
 *                A_t = diag(exp(g_{t+1})) A_{t+1} + scale q_t^T do_t
 *     dq_t     = scale * S_t do_t^T              (contract over V)
 *     dk_t     = A_t v_t^T                       (contract over V)
 *     dv_t     = k_t A_t                         (contract over K)
 *     dg_t[k]  = exp(g_t[k]) * sum_v A_t[k,v] S_{t-1}[k,v]
 *     dh0      = diag(exp(g_first)) A_first
 *
 * S_{t-1} is needed on the way back: the forward sweep keeps the state at every 64th step and each block
 * of 64 steps is recomputed from its checkpoint before it is walked backwards.  do has the stored type of
 * q, k, v, g; h0 and dht are double [N,H,K,V] or NULL (zeros).  Outputs are double in the layouts of
 * q / v / h0; dh0 may be NULL.  Returns the threads used, or a negative value on bad arguments.
 */
enum { BWD_BLOCK = 64 };

typedef struct {
    const void *q, *k, *v, *g, *dout;
    int dtype;
    const double *h0, *dht;
    double *dq, *dk, *dv, *dg, *dh0;
    const int32_t *cu;
    int N, H, K, V;
    double scale;
    int next;
    pthread_mutex_t mu;
} bwd_job;

/* one step of the forward recurrence on a K x V state */
static void fwd_step(const bwd_job *J, long t, int h, double *S)
{
    const int H = J->H, K = J->K, V = J->V;
    const size_t kb = ((size_t)t * H + h) * K, vb = ((size_t)t * H + h) * V;
    for (int i = 0; i < K; ++i) {
        const double e = exp(widen(J->g, kb + i, J->dtype));
        const double kt = widen(J->k, kb + i, J->dtype);
        double *srow = S + (size_t)i * V;
        for (int j = 0; j < V; ++j)
            srow[j] = e * srow[j] + kt * widen(J->v, vb + j, J->dtype);
    }
}

static int bwd_one(bwd_job *J, int item)
{
    const int n = item / J->H, h = item % J->H;
    const int H = J->H, K = J->K, V = J->V;
    const long bos = J->cu[n], eos = J->cu[n + 1], len = eos - bos;
    const size_t KV = (size_t)K * V;
    const long nb = (len + BWD_BLOCK - 1) / BWD_BLOCK;
    /* ck[m] = state before block m (ck[0] = h0); blk[i] = state after the i-th step of the current block */
    double *ck = (double *)malloc(sizeof(double) * KV * (size_t)(nb > 0 ? nb : 1));
    double *blk = (double *)malloc(sizeof(double) * KV * BWD_BLOCK);
    double *S = (double *)malloc(sizeof(double) * KV);
    double *A = (double *)malloc(sizeof(double) * KV);
    if (!ck || !blk || !S || !A) {
        free(ck); free(blk); free(S); free(A);
        return -2;
    }
    const size_t st = ((size_t)n * H + h) * KV;
    for (size_t e = 0; e < KV; ++e) {
        S[e] = J->h0 ? J->h0[st + e] : 0.0;
        A[e] = J->dht ? J->dht[st + e] : 0.0;
    }
    for (long t = bos; t < eos; ++t) {
        if ((t - bos) % BWD_BLOCK == 0)
            memcpy(ck + (size_t)((t - bos) / BWD_BLOCK) * KV, S, sizeof(double) * KV);
        fwd_step(J, t, h, S);
    }
    for (long m = nb - 1; m >= 0; --m) {
        const long b0 = bos + m * BWD_BLOCK, b1 = b0 + BWD_BLOCK < eos ? b0 + BWD_BLOCK : eos;
        memcpy(S, ck + (size_t)m * KV, sizeof(double) * KV);
        for (long t = b0; t < b1; ++t) {
            fwd_step(J, t, h, S);
            memcpy(blk + (size_t)(t - b0) * KV, S, sizeof(double) * KV);
        }
        for (long t = b1 - 1; t >= b0; --t) {
            const size_t kb = ((size_t)t * H + h) * K, vb = ((size_t)t * H + h) * V;
            const double *St = blk + (size_t)(t - b0) * KV;                             /* S_t */
            const double *Sp = t > b0 ? blk + (size_t)(t - b0 - 1) * KV : ck + (size_t)m * KV;  /* S_{t-1} */
            /* A <- A + scale q_t^T do_t: now dL/dS_t */
            for (int i = 0; i < K; ++i) {
                const double qi = J->scale * widen(J->q, kb + i, J->dtype);
                for (int j = 0; j < V; ++j)
                    A[(size_t)i * V + j] += qi * widen(J->dout, vb + j, J->dtype);
            }
            for (int i = 0; i < K; ++i) {
                double aq = 0.0, ak = 0.0, ag = 0.0;
                for (int j = 0; j < V; ++j) {
                    const double dj = widen(J->dout, vb + j, J->dtype);
                    aq += St[(size_t)i * V + j] * dj;
                    ak += A[(size_t)i * V + j] * widen(J->v, vb + j, J->dtype);
                    ag += A[(size_t)i * V + j] * Sp[(size_t)i * V + j];
                }
                J->dq[kb + i] = J->scale * aq;
                J->dk[kb + i] = ak;
                J->dg[kb + i] = exp(widen(J->g, kb + i, J->dtype)) * ag;
            }
            for (int j = 0; j < V; ++j) {
                double av = 0.0;
                for (int i = 0; i < K; ++i)
                    av += widen(J->k, kb + i, J->dtype) * A[(size_t)i * V + j];
                J->dv[vb + j] = av;
            }
            /* A <- diag(exp(g_t)) A: dL/dS_{t-1} before the o_{t-1} term */
            for (int i = 0; i < K; ++i) {
                const double e = exp(widen(J->g, kb + i, J->dtype));
                for (int j = 0; j < V; ++j)
                    A[(size_t)i * V + j] *= e;
            }
        }
    }
    if (J->dh0)
        memcpy(J->dh0 + st, A, sizeof(double) * KV);
    free(ck); free(blk); free(S); free(A);
    return 0;
}

static void *bwd_worker(void *arg)
{
    bwd_job *J = (bwd_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int item = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (item >= J->N * J->H)
            break;
        if (bwd_one(J, item) != 0)
            return (void *)1;
    }
    return NULL;
}

int oracle_gla_bwd(const void *q, const void *k, const void *v, const void *g, const void *dout, int dtype,
                   const double *h0, const double *dht, double *dq, double *dk, double *dv, double *dg,
                   double *dh0, const int32_t *cu_seqlens, int N, int B, int T, int H, int K, int V,
                   double scale, int nthreads)
{
    if (!q || !k || !v || !g || !dout || !dq || !dk || !dv || !dg || H <= 0 || K <= 0 || V <= 0 || B < 0 ||
        T < 0)
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64 && dtype != ORACLE_F16)
        return -1;
    int32_t *dense = NULL;
    const int32_t *cu = cu_seqlens;
    if (!cu) {
        N = B;
        dense = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N + 1));
        if (!dense)
            return -2;
        for (int n = 0; n <= N; ++n)
            dense[n] = n * T;
        cu = dense;
    }
    if (N == 0) {
        free(dense);
        return 0;
    }
    if (dh0)
        memset(dh0, 0, sizeof(double) * (size_t)N * H * K * V);
    bwd_job J = {q, k, v, g, dout, dtype, h0, dht, dq, dk, dv, dg, dh0, cu, N, H, K, V, scale, 0,
                 PTHREAD_MUTEX_INITIALIZER};
    const int nt = resolve_threads(nthreads, N * H);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    int rc = nt;
    if (!tid) {
        free(dense);
        return -2;
    }
    int started = 0;
    for (; started < nt; ++started)
        if (pthread_create(&tid[started], NULL, bwd_worker, &J) != 0)
            break;
    if (started == 0 && bwd_worker(&J))
        rc = -2;
    for (int i = 0; i < started; ++i) {
        void *res = NULL;
        pthread_join(tid[i], &res);
        if (res)
            rc = -2;
    }
    free(tid);
    free(dense);
    return started ? rc : (rc < 0 ? rc : 1);
}

/*
 * TTT-linear forward by mini-batch gradient descent (page "fla/ops/ttt/fused_chunk.py":
 * fused_chunk_ttt_linear_fwd_kernel, then the norm_residual step of fused_chunk_ttt_linear), written in
 * the kernel's dual form, fp64.  Per (sequence, head), with state h [D][D] and bias hb [D] and chunks of
 * `chunk` rows (the mini-batch: the result depends on it):
 *
 *     kh_i  = k_i h + hb;  xhat_i = (kh_i - mean) / sqrt(var + eps) over D;  r_i = 1 / sqrt(var + eps)
 *     g_i   = (xhat_i * w + b + k_i - v_i) * w                     gradient of the inner loss wrt xhat
 *     v2_i  = r_i / D * (D g_i - sum(g_i) - xhat_i * sum(g_i * xhat_i))      ... and wrt kh_i
 *     o_i   = scale q_i h + hb - eta_i * sum_{j <= i} (scale q_i . k_j + 1) v2_j
 *     o_i  += LN(o_i) * w + b                                       (the residual norm of the wrapper)
 *     h    -= eta_last * sum_j k_j^T v2_j;   hb -= eta_last * sum_j v2_j
 *
 * Rows past the end of a sequence do not exist (a partial last chunk has only its valid rows).  q, k, v
 * are [rows, H, D] in the stored type `dtype`; w, b [H][D]; eta [rows][H]; h0 [N,H,D,D], hb0 [N,H,D] or
 * NULL; outputs o [rows, H, D], ht, hbt (or NULL) in double.  Returns threads used or a negative value.
 */
typedef struct {
    const void *q, *k, *v;
    int dtype;
    const double *w, *b, *eta, *h0, *hb0;
    double *o, *ht, *hbt;
    const int32_t *cu;
    int N, H, D, BT;
    double scale, eps;
    int next;
    pthread_mutex_t mu;
} ttt_job;

static void layer_norm(const double *x, int D, double eps, double *xhat, double *rstd)
{
    double mean = 0.0, var = 0.0;
    for (int d = 0; d < D; ++d)
        mean += x[d];
    mean /= D;
    for (int d = 0; d < D; ++d)
        var += (x[d] - mean) * (x[d] - mean);
    var /= D;
    const double r = 1.0 / sqrt(var + eps);
    for (int d = 0; d < D; ++d)
        xhat[d] = (x[d] - mean) * r;
    if (rstd)
        *rstd = r;
}

static int ttt_one(ttt_job *J, int item)
{
    const int n = item / J->H, h = item % J->H, H = J->H, D = J->D, BT = J->BT;
    const long bos = J->cu[n], eos = J->cu[n + 1];
    const double *w = J->w + (size_t)h * D, *b = J->b + (size_t)h * D;
    double *S = (double *)malloc(sizeof(double) * (size_t)D * D);
    double *hb = (double *)malloc(sizeof(double) * (size_t)D);
    double *V2 = (double *)malloc(sizeof(double) * (size_t)BT * D);
    double *kh = (double *)malloc(sizeof(double) * (size_t)D);
    double *xh = (double *)malloc(sizeof(double) * (size_t)D);
    double *gv = (double *)malloc(sizeof(double) * (size_t)D);
    if (!S || !hb || !V2 || !kh || !xh || !gv) {
        free(S); free(hb); free(V2); free(kh); free(xh); free(gv);
        return -2;
    }
    const size_t st = ((size_t)n * H + h);
    for (size_t e = 0; e < (size_t)D * D; ++e)
        S[e] = J->h0 ? J->h0[st * D * D + e] : 0.0;
    for (int d = 0; d < D; ++d)
        hb[d] = J->hb0 ? J->hb0[st * D + d] : 0.0;
    for (long r0 = bos; r0 < eos; r0 += BT) {
        const long r1 = r0 + BT < eos ? r0 + BT : eos;
        /* gradients of the inner loss at the chunk-start state */
        for (long t = r0; t < r1; ++t) {
            const size_t rb = ((size_t)t * H + h) * D;
            for (int c = 0; c < D; ++c) {
                double acc = hb[c];
                for (int kk = 0; kk < D; ++kk)
                    acc += widen(J->k, rb + kk, J->dtype) * S[(size_t)kk * D + c];
                kh[c] = acc;
            }
            double r;
            layer_norm(kh, D, J->eps, xh, &r);
            double sg = 0.0, sgx = 0.0;
            for (int c = 0; c < D; ++c) {
                gv[c] = (xh[c] * w[c] + b[c] + widen(J->k, rb + c, J->dtype) - widen(J->v, rb + c, J->dtype)) * w[c];
                sg += gv[c];
                sgx += gv[c] * xh[c];
            }
            for (int c = 0; c < D; ++c)
                V2[(size_t)(t - r0) * D + c] = r / D * (D * gv[c] - sg - xh[c] * sgx);
        }
        /* outputs, dual form, then the residual norm */
        for (long t = r0; t < r1; ++t) {
            const size_t rb = ((size_t)t * H + h) * D;
            const double et = J->eta[(size_t)t * H + h];
            for (int c = 0; c < D; ++c) {
                double acc = hb[c];
                for (int kk = 0; kk < D; ++kk)
                    acc += J->scale * widen(J->q, rb + kk, J->dtype) * S[(size_t)kk * D + c];
                kh[c] = acc;
            }
            for (long s = r0; s <= t; ++s) {
                const size_t sb = ((size_t)s * H + h) * D;
                double a = 0.0;
                for (int kk = 0; kk < D; ++kk)
                    a += J->scale * widen(J->q, rb + kk, J->dtype) * widen(J->k, sb + kk, J->dtype);
                for (int c = 0; c < D; ++c)
                    kh[c] -= et * (a + 1.0) * V2[(size_t)(s - r0) * D + c];
            }
            layer_norm(kh, D, J->eps, xh, NULL);
            for (int c = 0; c < D; ++c)
                J->o[rb + c] = kh[c] + xh[c] * w[c] + b[c];
        }
        /* state update with the learning rate of the chunk's last row */
        const double el = J->eta[(size_t)(r1 - 1) * H + h];
        for (long s = r0; s < r1; ++s) {
            const size_t sb = ((size_t)s * H + h) * D;
            for (int kk = 0; kk < D; ++kk) {
                const double kv = el * widen(J->k, sb + kk, J->dtype);
                for (int c = 0; c < D; ++c)
                    S[(size_t)kk * D + c] -= kv * V2[(size_t)(s - r0) * D + c];
            }
            for (int c = 0; c < D; ++c)
                hb[c] -= el * V2[(size_t)(s - r0) * D + c];
        }
    }
    if (J->ht)
        memcpy(J->ht + st * D * D, S, sizeof(double) * (size_t)D * D);
    if (J->hbt)
        memcpy(J->hbt + st * D, hb, sizeof(double) * (size_t)D);
    free(S); free(hb); free(V2); free(kh); free(xh); free(gv);
    return 0;
}

static void *ttt_worker(void *arg)
{
    ttt_job *J = (ttt_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int item = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (item >= J->N * J->H)
            break;
        if (ttt_one(J, item) != 0)
            return (void *)1;
    }
    return NULL;
}

int oracle_ttt_linear_fwd(const void *q, const void *k, const void *v, int dtype, const double *w,
                          const double *b, const double *eta, double scale, double eps, const double *h0,
                          const double *hb0, double *o, double *ht, double *hbt, const int32_t *cu_seqlens,
                          int N, int B, int T, int H, int D, int chunk, int nthreads)
{
    if (!q || !k || !v || !w || !b || !eta || !o || H <= 0 || D <= 0 || B < 0 || T < 0 || chunk <= 0)
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64 && dtype != ORACLE_F16)
        return -1;
    int32_t *dense = NULL;
    const int32_t *cu = cu_seqlens;
    if (!cu) {
        N = B;
        dense = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N + 1));
        if (!dense)
            return -2;
        for (int n = 0; n <= N; ++n)
            dense[n] = n * T;
        cu = dense;
    }
    if (N == 0) {
        free(dense);
        return 0;
    }
    ttt_job J = {q, k, v, dtype, w, b, eta, h0, hb0, o, ht, hbt, cu, N, H, D, chunk, scale, eps, 0,
                 PTHREAD_MUTEX_INITIALIZER};
    const int nt = resolve_threads(nthreads, N * H);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    int rc = nt;
    if (!tid) {
        free(dense);
        return -2;
    }
    int started = 0;
    for (; started < nt; ++started)
        if (pthread_create(&tid[started], NULL, ttt_worker, &J) != 0)
            break;
    if (started == 0 && ttt_worker(&J))
        rc = -2;
    for (int i = 0; i < started; ++i) {
        void *res = NULL;
        pthread_join(tid[i], &res);
        if (res)
            rc = -2;
    }
    free(tid);
    free(dense);
    return started ? rc : (rc < 0 ? rc : 1);
}

/*
 * WY representation forward of the gated delta rule (page
 * "fla/ops/gated_delta_rule/backends/triton_ascend/wy_fast.py": recompute_w_u_fwd_kernel_npu and its host
 * launcher recompute_w_u_fwd_npu), fp64.  Each sequence is cut into chunks of BT rows from its first row
 * (the last chunk may be partial).  For value head hv, whose key head is hv / (HV / H), and a row t of the
 * chunk [c0, c1):
 *
 *     u_t = sum_{s = c0}^{c1 - 1} A_t[s - c0] * beta_s * v_s
 *     w_t = sum_{s = c0}^{c1 - 1} A_t[s - c0] * beta_s * 2^{g_s} * k_s        (the factor 2^{g_s} is 1 without g)
 *
 * A_t is row t of A [rows, HV, BT]: the chunk's BT x BT matrix stored row by row, used as a full square.
 * Rows past the end of a sequence do not exist, and the columns of A that would refer to them are not read.
 * k [rows, H, K], v [rows, HV, V], A and beta [rows, HV] are in the stored type `dtype`; g [rows, HV] is in
 * double or NULL; the outputs w [rows, HV, K] and u [rows, HV, V] are double and start at zero.
 */
typedef struct {
    const void *k, *v, *A, *beta;
    int dtype;
    const double *g;
    double *w, *u;
    const int32_t *cu;
    int N, H, HV, K, V, BT;
    int next;
    pthread_mutex_t mu;
} wy_job;

static void wy_one(wy_job *J, int item)
{
    const int HV = J->HV, K = J->K, V = J->V, BT = J->BT;
    const int n = item / HV, hv = item % HV, hk = hv / (HV / J->H);
    const long first = J->cu[n], end = J->cu[n + 1];
    for (long c0 = first; c0 < end; c0 += BT) {
        const long c1 = c0 + BT < end ? c0 + BT : end;
        for (long t = c0; t < c1; ++t) {
            double *wrow = J->w + ((size_t)t * HV + hv) * K, *urow = J->u + ((size_t)t * HV + hv) * V;
            for (long s = c0; s < c1; ++s) {
                const double coef = widen(J->A, ((size_t)t * HV + hv) * BT + (size_t)(s - c0), J->dtype) *
                                    widen(J->beta, (size_t)s * HV + hv, J->dtype);
                const double decay = J->g ? exp2(J->g[(size_t)s * HV + hv]) : 1.0;
                for (int c = 0; c < V; ++c)
                    urow[c] += coef * widen(J->v, ((size_t)s * HV + hv) * V + c, J->dtype);
                for (int c = 0; c < K; ++c)
                    wrow[c] += coef * decay * widen(J->k, ((size_t)s * J->H + hk) * K + c, J->dtype);
            }
        }
    }
}

static void *wy_worker(void *arg)
{
    wy_job *J = (wy_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int item = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (item >= J->N * J->HV)
            break;
        wy_one(J, item);
    }
    return NULL;
}

int oracle_wy_fwd(const void *k, const void *v, const void *A, const void *beta, int dtype, const double *g,
                  double *w, double *u, const int32_t *cu_seqlens, int N, int B, int T, int H, int HV, int K,
                  int V, int BT, int nthreads)
{
    if (!k || !v || !A || !beta || !w || !u || H <= 0 || HV <= 0 || HV % H || K <= 0 || V <= 0 || BT <= 0 ||
        B < 0 || T < 0)
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64 && dtype != ORACLE_F16)
        return -1;
    int32_t *dense = NULL;
    const int32_t *cu = cu_seqlens;
    if (!cu) {
        N = B;
        dense = (int32_t *)malloc(sizeof(int32_t) * (size_t)(N + 1));
        if (!dense)
            return -2;
        for (int n = 0; n <= N; ++n)
            dense[n] = n * T;
        cu = dense;
    }
    if (N == 0) {
        free(dense);
        return 0;
    }
    wy_job J = {k, v, A, beta, dtype, g, w, u, cu, N, H, HV, K, V, BT, 0, PTHREAD_MUTEX_INITIALIZER};
    const int nt = resolve_threads(nthreads, N * HV);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!tid) {
        free(dense);
        return -2;
    }
    int started = 0;
    for (; started < nt; ++started)
        if (pthread_create(&tid[started], NULL, wy_worker, &J) != 0)
            break;
    if (started == 0)
        wy_worker(&J);
    for (int i = 0; i < started; ++i)
        pthread_join(tid[i], NULL);
    free(tid);
    free(dense);
    return started ? nt : 1;
}
