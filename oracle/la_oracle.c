/*
 * la_oracle.c -- fp64 CPU oracle for causal linear attention with a per-head
 * scalar exponential decay (the Lightning / g_gamma recurrence).
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  It shares
 * no code, header or constant with the CUDA library under
 * linear_attention_head_gb300/, and the product never calls it.
 *
 * What it computes (token by token, no chunking, no reordering):
 *
 *   ejkernel docs, kernels/_xla/recurrent/_interface, `recurrent` docstring,
 *   its state-update formula: the state h decays by decay_t and gains the
 *   outer product of k_t and v_t; the output reads the state with q_t.
 *   Read as (see the readings below)
 *        S_t = gamma * S_{t-1} + outer(k_t, v_t)          S is d x e
 *        o_t = scale * (q_t^T S_t)                        an e-vector
 *   with gamma = exp(g_gamma[h])   (g_gamma holds one log-decay per head, same
 *   docstring, Args; Lightning's layer-dependent g_gamma formula in the
 *   ejkernel lightning_attn page, module docstring, is negative, so the decay
 *   is exp of it),
 *   scale multiplying the query only (softmax_scale, same Args),
 *   S_0 = initial_state or zeros, final_state = S after the last processed
 *   token, `reverse` = the same recurrence over t = L-1 .. 0 of each sequence,
 *   and packed sequences delimited by cu_seqlens = [0, len1, len1+len2, ...]
 *   (lightning_attn docstring, Args: cu_seqlens), each with its own state.
 *
 * Backward (the custom VJP on the same page, `_recurrent_bwd`, upstream grads
 * (do, dfinal_state); g_gamma, scale, reverse and cu_seqlens are not
 * differentiated): for the scalar loss  sum(o * do) + sum(final * dfinal),
 *   sweep A, processing order:  recompute S_t, dq_t = scale * S_t do_t
 *   sweep B, opposite order:    G = dfinal (or 0);  for each t:
 *                                  G += scale * outer(q_t, do_t)
 *                                  dk_t = G v_t ;  dv_t = G^T k_t ;  G = gamma*G
 *                               d_initial_state = G
 *   (G before the decay is dL/dS_t; the last decay carries it back to S_0.)
 *
 * Gated form (ejkernel `recurrent` Args: the optional gate `g`, shaped like
 * the keys; the GLA page's `recurrent_gla` passes it on to
 * `recurrent`).  Read as a log-decay per key channel, added to the head's
 * g_gamma:
 *        S_t[a, :] = exp(g_gamma[h] + g_t[a]) * S_{t-1}[a, :] + k_t[a] v_t
 * (the gate of token t multiplies the state that token t is added to, in
 * either direction).  Backward as above with the row-wise decay, and
 *        dg_t[a] = exp(g_gamma[h] + g_t[a]) * sum_b G_t[a, b] S_{t-1}[a, b]
 * with G_t = dL/dS_t (after token t's term, before its decay) and S_{t-1}
 * the state token t decays.  Sweep B needs S_{t-1} in reverse order: the
 * forward states are kept every K = ceil(sqrt(L)) tokens and each block of K
 * is recomputed from its checkpoint when sweep B reaches it.
 *
 * Layout: every token tensor is a dense row-major fp64 array [B, T, H, X]
 * (X = d for q, k, dq, dk and e for v, o, do, dv); states are [N, H, d, e].
 * With cu_seqlens (B must be 1) sequence n covers tokens cu[n] .. cu[n+1]-1
 * and N = num_seqs; otherwise N = B and each batch row is one sequence of
 * length T.  Zero-length sequences are allowed: final = initial (or 0) and
 * d_initial = dfinal (or 0).
 *
 * Threads: one task per (sequence, head) on `threads` POSIX threads (0 = all
 * online cores).  Each task touches disjoint output rows, so the result does
 * not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    int B, T, H, d, e, N;
    const int32_t *cu;          /* [N+1] or NULL */
    const double *q, *k, *v, *g_gamma, *init;
    const double *gate;         /* [B,T,H,d] per-key log-decay, or NULL */
    double scale;
    int reverse;
    /* forward outputs */
    double *o, *final_state;
    /* backward inputs / outputs */
    const double *dout, *dfinal;
    double *dq, *dk, *dv, *dinit;
    double *dgate;              /* [B,T,H,d], written when gate is given */
    int mode;                   /* 0 = forward, 1 = backward */
    /* work distribution */
    int next;                   /* next (n, h) task, guarded by lock */
    pthread_mutex_t lock;
} job_t;

/* Token range of sequence n: [*bos, *bos + *len); the batch row used to
 * address the token tensors is *row. */
static void seq_range(const job_t *J, int n, int64_t *bos, int64_t *len, int64_t *row)
{
    if (J->cu) {
        *row = 0;
        *bos = J->cu[n];
        *len = (int64_t)J->cu[n + 1] - J->cu[n];
    } else {
        *row = n;
        *bos = 0;
        *len = J->T;
    }
}

static inline const double *tok(const double *base, const job_t *J, int64_t row,
                                int64_t t, int h, int width)
{
    return base + (((row * J->T + t) * J->H) + h) * (int64_t)width;
}

static inline double *tok_w(double *base, const job_t *J, int64_t row, int64_t t,
                            int h, int width)
{
    return base + (((row * J->T + t) * J->H) + h) * (int64_t)width;
}

/* decay of row a at token t of batch row `row` */
static inline double decay(const job_t *J, int64_t row, int64_t t, int h, int a, double gh)
{
    return J->gate ? exp(gh + tok(J->gate, J, row, t, h, J->d)[a]) : exp(gh);
}

/* S <- diag(decay_t) S + outer(k_t, v_t) */
static void step_state(const job_t *J, int64_t row, int64_t t, int h, double *S)
{
    const int d = J->d, e = J->e;
    const double gh = J->g_gamma[h];
    const double *kt = tok(J->k, J, row, t, h, d);
    const double *vt = tok(J->v, J, row, t, h, e);
    for (int a = 0; a < d; ++a) {
        const double da = decay(J, row, t, h, a, gh);
        for (int b = 0; b < e; ++b)
            S[a * e + b] = da * S[a * e + b] + kt[a] * vt[b];
    }
}

static void run_forward(const job_t *J, int n, int h, double *S)
{
    const int d = J->d, e = J->e;
    int64_t bos, len, row;
    seq_range(J, n, &bos, &len, &row);
    const int64_t sidx = ((int64_t)n * J->H + h) * d * e;
    if (J->init)
        memcpy(S, J->init + sidx, sizeof(double) * d * e);
    else
        memset(S, 0, sizeof(double) * d * e);
    for (int64_t step = 0; step < len; ++step) {
        const int64_t t = bos + (J->reverse ? len - 1 - step : step);
        const double *qt = tok(J->q, J, row, t, h, d);
        step_state(J, row, t, h, S);
        double *ot = tok_w(J->o, J, row, t, h, e);
        for (int b = 0; b < e; ++b) {
            double acc = 0.0;
            for (int a = 0; a < d; ++a)
                acc += qt[a] * S[a * e + b];
            ot[b] = J->scale * acc;
        }
    }
    if (J->final_state)
        memcpy(J->final_state + sidx, S, sizeof(double) * d * e);
}

static void run_backward(const job_t *J, int n, int h, double *S, double *ck)
{
    const int d = J->d, e = J->e;
    const int64_t de = (int64_t)d * e;
    const double gh = J->g_gamma[h];
    int64_t bos, len, row;
    seq_range(J, n, &bos, &len, &row);
    const int64_t sidx = ((int64_t)n * J->H + h) * de;
    /* gated: checkpoint every K tokens; ck holds the block-start states, then
     * the K + 1 states of the block being replayed */
    int64_t K = 1;
    while (K * K < len)
        ++K;
    double *blk = ck ? ck + ((len + K - 1) / K) * de : NULL;

    /* sweep A: recompute the forward states, dq_t = scale * S_t do_t */
    if (J->init)
        memcpy(S, J->init + sidx, sizeof(double) * de);
    else
        memset(S, 0, sizeof(double) * de);
    for (int64_t step = 0; step < len; ++step) {
        const int64_t t = bos + (J->reverse ? len - 1 - step : step);
        if (J->gate && step % K == 0)
            memcpy(ck + (step / K) * de, S, sizeof(double) * de);
        const double *dot = tok(J->dout, J, row, t, h, e);
        step_state(J, row, t, h, S);
        double *dqt = tok_w(J->dq, J, row, t, h, d);
        for (int a = 0; a < d; ++a) {
            double acc = 0.0;
            for (int b = 0; b < e; ++b)
                acc += S[a * e + b] * dot[b];
            dqt[a] = J->scale * acc;
        }
    }

    /* sweep B: carry G = dL/dS backwards through the processing order */
    double *G = S;
    if (J->dfinal)
        memcpy(G, J->dfinal + sidx, sizeof(double) * de);
    else
        memset(G, 0, sizeof(double) * de);
    for (int64_t step = len - 1; step >= 0; --step) {
        const int64_t t = bos + (J->reverse ? len - 1 - step : step);
        if (J->gate && (step == len - 1 || step % K == K - 1)) {
            /* replay the block holding `step`: blk[i] = state before step b0 + i */
            const int64_t b0 = (step / K) * K;
            memcpy(blk, ck + (step / K) * de, sizeof(double) * de);
            for (int64_t i = 0; b0 + i < step; ++i) {
                const int64_t ti = bos + (J->reverse ? len - 1 - (b0 + i) : b0 + i);
                memcpy(blk + (i + 1) * de, blk + i * de, sizeof(double) * de);
                step_state(J, row, ti, h, blk + (i + 1) * de);
            }
        }
        const double *qt = tok(J->q, J, row, t, h, d);
        const double *kt = tok(J->k, J, row, t, h, d);
        const double *vt = tok(J->v, J, row, t, h, e);
        const double *dot = tok(J->dout, J, row, t, h, e);
        for (int a = 0; a < d; ++a)
            for (int b = 0; b < e; ++b)
                G[a * e + b] += J->scale * qt[a] * dot[b];
        double *dkt = tok_w(J->dk, J, row, t, h, d);
        for (int a = 0; a < d; ++a) {
            double acc = 0.0;
            for (int b = 0; b < e; ++b)
                acc += G[a * e + b] * vt[b];
            dkt[a] = acc;
        }
        double *dvt = tok_w(J->dv, J, row, t, h, e);
        for (int b = 0; b < e; ++b) {
            double acc = 0.0;
            for (int a = 0; a < d; ++a)
                acc += G[a * e + b] * kt[a];
            dvt[b] = acc;
        }
        if (J->gate) {
            const double *prev = blk + (step % K) * de;   /* S_{t-1} */
            double *dgt = tok_w(J->dgate, J, row, t, h, d);
            for (int a = 0; a < d; ++a) {
                double acc = 0.0;
                for (int b = 0; b < e; ++b)
                    acc += G[a * e + b] * prev[a * e + b];
                dgt[a] = decay(J, row, t, h, a, gh) * acc;
            }
        }
        for (int a = 0; a < d; ++a) {
            const double da = decay(J, row, t, h, a, gh);
            for (int b = 0; b < e; ++b)
                G[a * e + b] *= da;
        }
    }
    if (J->dinit)
        memcpy(J->dinit + sidx, G, sizeof(double) * de);
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    const size_t de = (size_t)J->d * (size_t)J->e;
    double *S = (double *)malloc(sizeof(double) * de);
    /* gated backward: checkpoints of the longest sequence plus one block */
    size_t ck_states = 0;
    if (J->gate && J->mode == 1) {
        int64_t K = 1;
        while (K * K < J->T)
            ++K;
        ck_states = (size_t)(2 * K + 2);   /* >= ceil(L/K_L) + K_L for every L <= T */
    }
    double *ck = ck_states ? (double *)malloc(sizeof(double) * de * ck_states) : NULL;
    if (!S || (ck_states && !ck)) {
        free(S);
        free(ck);
        return (void *)1;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int task = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (task >= J->N * J->H)
            break;
        const int n = task / J->H, h = task % J->H;
        if (J->mode == 0)
            run_forward(J, n, h, S);
        else
            run_backward(J, n, h, S, ck);
    }
    free(S);
    free(ck);
    return NULL;
}

static int run_job(job_t *J, int threads)
{
    if (threads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        threads = c > 0 ? (int)c : 1;
    }
    if (threads > J->N * J->H)
        threads = J->N * J->H > 0 ? J->N * J->H : 1;
    J->next = 0;
    pthread_mutex_init(&J->lock, NULL);
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    int rc = tid ? 0 : 1, started = 0;
    for (int i = 0; i < threads && !rc; ++i) {
        if (pthread_create(&tid[i], NULL, worker, J) != 0)
            rc = 1;
        else
            ++started;
    }
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(tid[i], &ret);
        if (ret)
            rc = 1;
    }
    free(tid);
    pthread_mutex_destroy(&J->lock);
    return rc;
}

static int fill_common(job_t *J, int B, int T, int H, int d, int e, int num_seqs,
                       const int32_t *cu, const double *q, const double *k,
                       const double *v, const double *g_gamma, double scale,
                       const double *init, int reverse)
{
    memset(J, 0, sizeof(*J));
    if (B < 0 || T < 0 || H <= 0 || d <= 0 || e <= 0)
        return 2;
    if (cu && (B != 1 || num_seqs < 0))
        return 2;
    J->B = B; J->T = T; J->H = H; J->d = d; J->e = e;
    J->N = cu ? num_seqs : B;
    J->cu = cu;
    J->q = q; J->k = k; J->v = v; J->g_gamma = g_gamma; J->init = init;
    J->scale = scale;
    J->reverse = reverse ? 1 : 0;
    return 0;
}

/* Forward: writes o [B,T,H,e] and, if final_state is not NULL, [N,H,d,e].
 * gate: [B,T,H,d] per-key log-decay added to g_gamma, or NULL.
 * Returns 0 on success, 2 on bad sizes, 1 on a thread/allocation failure. */
int la_oracle_gla_fwd(int B, int T, int H, int d, int e, int num_seqs,
                      const int32_t *cu_seqlens, const double *q, const double *k,
                      const double *v, const double *g_gamma, const double *gate, double scale,
                      const double *initial_state, int reverse, double *o, double *final_state,
                      int threads)
{
    job_t J;
    int rc = fill_common(&J, B, T, H, d, e, num_seqs, cu_seqlens, q, k, v, g_gamma,
                         scale, initial_state, reverse);
    if (rc)
        return rc;
    J.gate = gate;
    J.mode = 0;
    J.o = o;
    J.final_state = final_state;
    return run_job(&J, threads);
}

int la_oracle_fwd(int B, int T, int H, int d, int e, int num_seqs, const int32_t *cu_seqlens,
                  const double *q, const double *k, const double *v,
                  const double *g_gamma, double scale, const double *initial_state,
                  int reverse, double *o, double *final_state, int threads)
{
    return la_oracle_gla_fwd(B, T, H, d, e, num_seqs, cu_seqlens, q, k, v, g_gamma, NULL, scale,
                             initial_state, reverse, o, final_state, threads);
}

/* Backward: writes dq, dk [B,T,H,d], dv [B,T,H,e], with a gate dgate
 * [B,T,H,d], and, if d_initial_state is not NULL, [N,H,d,e].  dout is dL/do;
 * d_final_state (or NULL = 0) is dL/dfinal_state. */
int la_oracle_gla_bwd(int B, int T, int H, int d, int e, int num_seqs,
                      const int32_t *cu_seqlens, const double *q, const double *k,
                      const double *v, const double *g_gamma, const double *gate, double scale,
                      const double *initial_state, int reverse, const double *dout,
                      const double *d_final_state, double *dq, double *dk, double *dv,
                      double *dgate, double *d_initial_state, int threads)
{
    job_t J;
    int rc = fill_common(&J, B, T, H, d, e, num_seqs, cu_seqlens, q, k, v, g_gamma,
                         scale, initial_state, reverse);
    if (rc)
        return rc;
    if (gate && !dgate)
        return 2;
    J.gate = gate;
    J.dgate = dgate;
    J.mode = 1;
    J.dout = dout;
    J.dfinal = d_final_state;
    J.dq = dq; J.dk = dk; J.dv = dv; J.dinit = d_initial_state;
    return run_job(&J, threads);
}

int la_oracle_bwd(int B, int T, int H, int d, int e, int num_seqs, const int32_t *cu_seqlens,
                  const double *q, const double *k, const double *v,
                  const double *g_gamma, double scale, const double *initial_state,
                  int reverse, const double *dout, const double *d_final_state,
                  double *dq, double *dk, double *dv, double *d_initial_state, int threads)
{
    return la_oracle_gla_bwd(B, T, H, d, e, num_seqs, cu_seqlens, q, k, v, g_gamma, NULL, scale,
                             initial_state, reverse, dout, d_final_state, dq, dk, dv, NULL,
                             d_initial_state, threads);
}
