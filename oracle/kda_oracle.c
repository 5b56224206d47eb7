/*
 * kda_oracle.c -- plain fp64 CPU oracle for the Kimi Delta Attention (KDA) recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this
 * file: only the test suite, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header or constant with the CUDA library.
 *
 * What it computes (source: "Kimi K3 im Detail" (flozi.net), section
 * "Sequenz-Mixing: KDA-Zustand und globale MLA", first and second paragraphs):
 *   per head a recurrent matrix S in R^{d_k x d_v}; for every token the old state is
 *   attenuated channel-wise by a retention vector alpha_t, then a scalar write gate
 *   beta_t applies a delta-rule correction, then the query reads S_t^T q_t.  The
 *   published log-decay is bounded below by g_min = -5 (second paragraph), so the
 *   retention of one step is >= e^-5.
 *
 * Readings fixed where the page is silent:
 *   - the channel-wise decay acts on the key axis:  S' = diag(exp(g_t)) S;
 *   - g is clamped to [-5, 0] before the exponential (natural base);
 *   - the delta rule reads the decayed state: r = S'^T k_t, S_t = S' + beta_t k_t (v_t - r)^T;
 *   - the read comes after the write of the same token: o_t = S_t^T q_t (the page's
 *     intra-chunk causal mask "contains the diagonal");
 *   - no 1/sqrt(d) query scaling;
 *   - sparse checkpoints: the state after token m*stride of a sequence, m = 1..floor(len/stride)
 *     (the page's prefix-reuse paragraph: only sparsely stored KDA states).
 *
 * Two independent evaluations are provided:
 *   kda_oracle_prefill   -- the per-token recurrence above, token by token;
 *   kda_oracle_chunked   -- the same result by the chunk algebra (a chunk of C tokens is
 *                           solved at once; the state is carried between chunks), following
 *                           the page's statement that prefill processes the tokens of a chunk
 *                           in parallel and passes the recurrent state between chunks.
 * and the one-token update used by decode:
 *   kda_oracle_decode    -- one step of the recurrence on each (sequence, head), in place.
 * Around the recurrence (readings at each function):
 *   kda_oracle_premix        -- short convolution of the projections, q/k normalisation, gates;
 *   kda_oracle_output_gate   -- the input-dependent output gate.
 *
 * Layouts (row-major, last index contiguous):
 *   q, k, g : [T_total, H, d_k]     v, out : [T_total, H, d_v]     beta : [T_total, H]
 *   states  : [N, H, d_k, d_v]  with S[i][j], i = key channel, j = value channel
 *   ckpts   : [n_ckpt, H, d_k, d_v], slots ordered by sequence, then by position
 *   cu_seqlens : [N + 1] host int64, cu_seqlens[0] = 0, non-decreasing
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KDA_ORACLE_OK 0
#define KDA_ORACLE_EINVAL 1
#define KDA_ORACLE_ENOMEM 2

/* clamp of the log-decay to the published range [-5, 0] */
static double clamp_logdecay(double g)
{
    if (g < -5.0) return -5.0;
    if (g > 0.0) return 0.0;
    return g;
}

/*
 * One token of the recurrence on one head's state S[dk][dv], in place.
 * r is caller scratch of length dv.  o receives S_t^T q (may be NULL).
 */
static void token_step(double *S, int64_t dk, int64_t dv, const double *q, const double *k,
                       const double *v, const double *g, double beta, double *o, double *r)
{
    /* decay: S'[i][j] = exp(g_i) * S[i][j]  (channel-wise over the key axis) */
    for (int64_t i = 0; i < dk; ++i) {
        double a = exp(clamp_logdecay(g[i]));
        for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= a;
    }
    /* prediction of the decayed state for key k: r = S'^T k */
    for (int64_t j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int64_t i = 0; i < dk; ++i) acc += S[i * dv + j] * k[i];
        r[j] = acc;
    }
    /* delta-rule write: S = S' + beta * k (v - r)^T */
    for (int64_t i = 0; i < dk; ++i)
        for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += beta * k[i] * (v[j] - r[j]);
    /* read after the write: o = S^T q */
    if (o) {
        for (int64_t j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int64_t i = 0; i < dk; ++i) acc += S[i * dv + j] * q[i];
            o[j] = acc;
        }
    }
}

/* ---------------------------------------------------------------------------------------- */
/* shared job description for the threaded drivers                                           */

typedef struct {
    const double *q, *k, *v, *g, *beta;
    const int64_t *cu_seqlens;
    int64_t n_seqs, n_heads, dk, dv;
    const double *init_state;
    double *out, *final_state;
    int64_t ckpt_stride;
    double *ckpts;
    const int64_t *ckpt_first; /* [N] first checkpoint slot of each sequence */
    int64_t chunk;             /* 0 = per-token recurrence, else chunk length */
    int64_t next_item;         /* work counter, (sequence, head) items */
    int failed;
} job_t;

/* state of one (sequence, head) at the start: init_state[n][h] or zeros */
static void load_initial(const job_t *jb, int64_t n, int64_t h, double *S)
{
    size_t nel = (size_t)(jb->dk * jb->dv);
    if (jb->init_state)
        memcpy(S, jb->init_state + ((size_t)(n * jb->n_heads + h)) * nel, nel * sizeof(double));
    else
        memset(S, 0, nel * sizeof(double));
}

static void store_state(const job_t *jb, double *dst_base, int64_t slot, int64_t h, const double *S)
{
    size_t nel = (size_t)(jb->dk * jb->dv);
    memcpy(dst_base + ((size_t)(slot * jb->n_heads + h)) * nel, S, nel * sizeof(double));
}

/* after token number `count` (1-based within the sequence) emit a checkpoint if due */
static void maybe_checkpoint(const job_t *jb, int64_t n, int64_t h, int64_t count, const double *S)
{
    if (jb->ckpt_stride > 0 && jb->ckpts && count % jb->ckpt_stride == 0) {
        int64_t slot = jb->ckpt_first[n] + count / jb->ckpt_stride - 1;
        store_state(jb, jb->ckpts, slot, h, S);
    }
}

/* per-token evaluation of one (sequence, head) */
static int run_item_recurrent(const job_t *jb, int64_t n, int64_t h)
{
    const int64_t H = jb->n_heads, dk = jb->dk, dv = jb->dv;
    double *S = malloc(sizeof(double) * (size_t)(dk * dv));
    double *r = malloc(sizeof(double) * (size_t)dv);
    if (!S || !r) { free(S); free(r); return KDA_ORACLE_ENOMEM; }
    load_initial(jb, n, h, S);
    int64_t start = jb->cu_seqlens[n], end = jb->cu_seqlens[n + 1];
    for (int64_t t = start; t < end; ++t) {
        size_t th = (size_t)(t * H + h);
        token_step(S, dk, dv, jb->q + th * dk, jb->k + th * dk, jb->v + th * dv,
                   jb->g + th * dk, jb->beta[th], jb->out ? jb->out + th * dv : NULL, r);
        maybe_checkpoint(jb, n, h, t - start + 1, S);
    }
    if (jb->final_state) store_state(jb, jb->final_state, n, h, S);
    free(S);
    free(r);
    return KDA_ORACLE_OK;
}

/*
 * Chunked evaluation of one (sequence, head).  Within a chunk of C tokens with state S0
 * at its start, let G_r = sum_{t<=r} clamp(g_t) (per key channel, cumulative inside the
 * chunk) and b_r = exp(G_r).  Unrolling the recurrence inside the chunk gives
 *   S_r = diag(b_r) [ S0 + sum_{s<=r} (k_s / b_s) u_s^T ],
 *   u_r = beta_r ( v_r - S0^T (k_r*b_r) - sum_{s<r} ((k_r*b_r).(k_s/b_s)) u_s ),
 *   o_r = S0^T (q_r*b_r) + sum_{s<=r} ((q_r*b_r).(k_s/b_s)) u_s,
 *   S_C = diag(b_C) S0 + sum_s (k_s * b_C / b_s) u_s^T,
 * i.e. the strictly lower system (I + A) U = diag(beta)(V - K~ S0) with
 * A[r][s] = beta_r (k~_r . k^_s), solved here by forward substitution.  In fp64 the factors
 * exp(+-G) stay finite for chunks up to 141 tokens at the -5 floor.
 */
static int run_item_chunked(const job_t *jb, int64_t n, int64_t h)
{
    const int64_t H = jb->n_heads, dk = jb->dk, dv = jb->dv, C = jb->chunk;
    double *S = malloc(sizeof(double) * (size_t)(dk * dv));
    double *G = malloc(sizeof(double) * (size_t)(C * dk));   /* cumulative log-decay */
    double *kt = malloc(sizeof(double) * (size_t)(C * dk));  /* k * b        */
    double *kh = malloc(sizeof(double) * (size_t)(C * dk));  /* k / b        */
    double *qt = malloc(sizeof(double) * (size_t)(C * dk));  /* q * b        */
    double *U = malloc(sizeof(double) * (size_t)(C * dv));   /* pseudo-values */
    if (!S || !G || !kt || !kh || !qt || !U) {
        free(S); free(G); free(kt); free(kh); free(qt); free(U);
        return KDA_ORACLE_ENOMEM;
    }
    load_initial(jb, n, h, S);
    int64_t start = jb->cu_seqlens[n], end = jb->cu_seqlens[n + 1];
    for (int64_t c0 = start; c0 < end; c0 += C) {
        int64_t L = (end - c0 < C) ? (end - c0) : C; /* a short last chunk is allowed */
        /* cumulative log-decay and the scaled keys / queries */
        for (int64_t r = 0; r < L; ++r) {
            size_t th = (size_t)((c0 + r) * H + h);
            for (int64_t i = 0; i < dk; ++i) {
                double gi = clamp_logdecay(jb->g[th * dk + i]);
                G[r * dk + i] = (r == 0 ? 0.0 : G[(r - 1) * dk + i]) + gi;
                double b = exp(G[r * dk + i]);
                kt[r * dk + i] = jb->k[th * dk + i] * b;
                kh[r * dk + i] = jb->k[th * dk + i] / b;
                qt[r * dk + i] = jb->q[th * dk + i] * b;
            }
        }
        /* forward substitution for U */
        for (int64_t r = 0; r < L; ++r) {
            size_t th = (size_t)((c0 + r) * H + h);
            double beta = jb->beta[th];
            for (int64_t j = 0; j < dv; ++j) {
                double pred = 0.0; /* (S0^T k~_r)_j */
                for (int64_t i = 0; i < dk; ++i) pred += S[i * dv + j] * kt[r * dk + i];
                U[r * dv + j] = beta * (jb->v[th * dv + j] - pred);
            }
            for (int64_t s = 0; s < r; ++s) {
                double dot = 0.0;
                for (int64_t i = 0; i < dk; ++i) dot += kt[r * dk + i] * kh[s * dk + i];
                double a_rs = beta * dot;
                for (int64_t j = 0; j < dv; ++j) U[r * dv + j] -= a_rs * U[s * dv + j];
            }
        }
        /* outputs, reading the state after each token's own write (diagonal included) */
        if (jb->out) {
            for (int64_t r = 0; r < L; ++r) {
                size_t th = (size_t)((c0 + r) * H + h);
                double *o = jb->out + th * dv;
                for (int64_t j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int64_t i = 0; i < dk; ++i) acc += S[i * dv + j] * qt[r * dk + i];
                    o[j] = acc;
                }
                for (int64_t s = 0; s <= r; ++s) {
                    double dot = 0.0;
                    for (int64_t i = 0; i < dk; ++i) dot += qt[r * dk + i] * kh[s * dk + i];
                    for (int64_t j = 0; j < dv; ++j) o[j] += dot * U[s * dv + j];
                }
            }
        }
        /* state carried to the next chunk */
        for (int64_t i = 0; i < dk; ++i) {
            double GC = G[(L - 1) * dk + i];
            double bC = exp(GC);
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= bC;
            for (int64_t s = 0; s < L; ++s) {
                double w = jb->k[((size_t)((c0 + s) * H + h)) * dk + i] * exp(GC - G[s * dk + i]);
                for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += w * U[s * dv + j];
            }
        }
        /* checkpoints fall on chunk ends when the stride is a multiple of C */
        maybe_checkpoint(jb, n, h, c0 + L - start, S);
    }
    if (jb->final_state) store_state(jb, jb->final_state, n, h, S);
    free(S); free(G); free(kt); free(kh); free(qt); free(U);
    return KDA_ORACLE_OK;
}

static void *worker(void *arg)
{
    job_t *jb = (job_t *)arg;
    const int64_t total = jb->n_seqs * jb->n_heads;
    for (;;) {
        int64_t item = __atomic_fetch_add(&jb->next_item, 1, __ATOMIC_RELAXED);
        if (item >= total) break;
        int64_t n = item / jb->n_heads, h = item % jb->n_heads;
        int rc = jb->chunk > 0 ? run_item_chunked(jb, n, h) : run_item_recurrent(jb, n, h);
        if (rc) __atomic_store_n(&jb->failed, rc, __ATOMIC_RELAXED);
    }
    return NULL;
}

static int run_job(job_t *jb, int n_threads)
{
    if (n_threads < 1) n_threads = 1;
    jb->next_item = 0;
    jb->failed = 0;
    if (n_threads == 1) {
        worker(jb);
        return jb->failed;
    }
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!th) return KDA_ORACLE_ENOMEM;
    int started = 0;
    for (int t = 0; t < n_threads; ++t) {
        if (pthread_create(&th[t], NULL, worker, jb) != 0) break;
        ++started;
    }
    if (started == 0) worker(jb);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    free(th);
    return jb->failed;
}

static int prefill_common(const double *q, const double *k, const double *v, const double *g,
                          const double *beta, const int64_t *cu_seqlens, int64_t n_seqs,
                          int64_t n_heads, int64_t dk, int64_t dv, const double *init_state,
                          double *out, double *final_state, int64_t ckpt_stride, double *ckpts,
                          int64_t chunk, int n_threads)
{
    if (n_seqs < 0 || n_heads < 1 || dk < 1 || dv < 1 || ckpt_stride < 0 || !cu_seqlens)
        return KDA_ORACLE_EINVAL;
    if (cu_seqlens[0] != 0) return KDA_ORACLE_EINVAL;
    for (int64_t n = 0; n < n_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return KDA_ORACLE_EINVAL;
    if (chunk > 0 && ckpt_stride > 0 && ckpt_stride % chunk != 0) return KDA_ORACLE_EINVAL;
    int64_t *first = calloc((size_t)(n_seqs + 1), sizeof(int64_t));
    if (!first) return KDA_ORACLE_ENOMEM;
    for (int64_t n = 0; n < n_seqs; ++n) {
        int64_t len = cu_seqlens[n + 1] - cu_seqlens[n];
        first[n + 1] = first[n] + (ckpt_stride > 0 ? len / ckpt_stride : 0);
    }
    job_t jb = {q, k, v, g, beta, cu_seqlens, n_seqs, n_heads, dk, dv, init_state, out,
                final_state, ckpt_stride, ckpts, first, chunk, 0, 0};
    int rc = run_job(&jb, n_threads);
    free(first);
    return rc;
}

/* number of checkpoint slots a prefill with this stride emits */
int64_t kda_oracle_num_ckpts(const int64_t *cu_seqlens, int64_t n_seqs, int64_t ckpt_stride)
{
    if (ckpt_stride <= 0) return 0;
    int64_t total = 0;
    for (int64_t n = 0; n < n_seqs; ++n) total += (cu_seqlens[n + 1] - cu_seqlens[n]) / ckpt_stride;
    return total;
}

int kda_oracle_prefill(const double *q, const double *k, const double *v, const double *g,
                       const double *beta, const int64_t *cu_seqlens, int64_t n_seqs,
                       int64_t n_heads, int64_t dk, int64_t dv, const double *init_state,
                       double *out, double *final_state, int64_t ckpt_stride, double *ckpts,
                       int n_threads)
{
    return prefill_common(q, k, v, g, beta, cu_seqlens, n_seqs, n_heads, dk, dv, init_state, out,
                          final_state, ckpt_stride, ckpts, 0, n_threads);
}

int kda_oracle_chunked(const double *q, const double *k, const double *v, const double *g,
                       const double *beta, const int64_t *cu_seqlens, int64_t n_seqs,
                       int64_t n_heads, int64_t dk, int64_t dv, const double *init_state,
                       double *out, double *final_state, int64_t ckpt_stride, double *ckpts,
                       int64_t chunk, int n_threads)
{
    if (chunk < 1 || chunk > 141) return KDA_ORACLE_EINVAL;
    return prefill_common(q, k, v, g, beta, cu_seqlens, n_seqs, n_heads, dk, dv, init_state, out,
                          final_state, ckpt_stride, ckpts, chunk, n_threads);
}

/*
 * Decode: one new token per sequence, state updated in place.
 * q, k, g : [N, H, dk]   v, out : [N, H, dv]   beta : [N, H]   state : [N, H, dk, dv]
 */
int kda_oracle_decode(const double *q, const double *k, const double *v, const double *g,
                      const double *beta, double *state, double *out, int64_t n_seqs,
                      int64_t n_heads, int64_t dk, int64_t dv)
{
    if (n_seqs < 0 || n_heads < 1 || dk < 1 || dv < 1) return KDA_ORACLE_EINVAL;
    double *r = malloc(sizeof(double) * (size_t)dv);
    if (!r) return KDA_ORACLE_ENOMEM;
    for (int64_t n = 0; n < n_seqs; ++n) {
        for (int64_t h = 0; h < n_heads; ++h) {
            size_t nh = (size_t)(n * n_heads + h);
            token_step(state + nh * (size_t)(dk * dv), dk, dv, q + nh * dk, k + nh * dk,
                       v + nh * dv, g + nh * dk, beta[nh], out ? out + nh * dv : NULL, r);
        }
    }
    free(r);
    return KDA_ORACLE_OK;
}

/*
 * Pre-mixer: what turns the KDA projections into the recurrence's inputs.  The page ("Kimi K3
 * im Detail", section "Sequenz-Mixing: KDA-Zustand und globale MLA", first paragraph) names a
 * short convolution of width 4 for the KDA projections and nothing else.  Readings fixed here:
 *   - the convolution is causal and depthwise (one 4-tap filter per channel of each of the q, k
 *     and v projections), with no activation after it;
 *   - inputs before a sequence's first token are its conv history: zeros, or the three rows
 *     given in hist (the last three projected tokens of a prefix this sequence continues);
 *   - q and k are L2-normalised per (token, head) after the convolution (the workloads feed the
 *     recurrence unit-norm q and k):  q = y / max(||y||_2, eps);
 *   - the decay and write gate come from pre-activations a and b as in the workloads' recipe:
 *     g = clamp(-softplus(a), -5, 0),  beta = 1 / (1 + exp(-b)).
 * Per channel c of head h (C = h*d + c) and tensor x in {q, k, v}, with taps w[x][C][0..3]:
 *     y_t[C] = w[x][C][0] x_{t-3}[C] + w[x][C][1] x_{t-2}[C] + w[x][C][2] x_{t-1}[C] + w[x][C][3] x_t[C]
 * Layouts: xq, xk, xv, a, q, k, v, g : [T, H, d];  b, beta : [T, H];  w : [3][H*d][4];
 *          hist : [N][3 (q, k, v)][3 (t-3, t-2, t-1)][H*d] or NULL.
 */
static double premix_input(const double *x, const double *hist, int64_t xi, int64_t n,
                           int64_t start, int64_t t, int64_t HD, int64_t col)
{
    if (t >= start) return x[t * HD + col];
    int64_t back = start - t;                      /* 1, 2 or 3 tokens before the start */
    if (!hist) return 0.0;
    return hist[((n * 3 + xi) * 3 + (3 - back)) * HD + col];
}

int kda_oracle_premix(const double *xq, const double *xk, const double *xv, const double *a,
                      const double *b, const double *w, const double *hist,
                      const int64_t *cu_seqlens, int64_t n_seqs, int64_t n_heads, int64_t d,
                      double eps, double *q, double *k, double *v, double *g, double *beta)
{
    if (n_seqs < 0 || n_heads < 1 || d < 1 || !(eps > 0.0)) return KDA_ORACLE_EINVAL;
    const int64_t HD = n_heads * d;
    const double *xs[3] = {xq, xk, xv};
    double *ys[3] = {q, k, v};
    for (int64_t n = 0; n < n_seqs; ++n) {
        const int64_t start = cu_seqlens[n], end = cu_seqlens[n + 1];
        if (end < start) return KDA_ORACLE_EINVAL;
        for (int64_t t = start; t < end; ++t) {
            for (int xi = 0; xi < 3; ++xi) {
                for (int64_t col = 0; col < HD; ++col) {
                    const double *tap = w + ((int64_t)xi * HD + col) * 4;
                    double acc = 0.0;
                    for (int i = 0; i < 4; ++i)
                        acc += tap[i] * premix_input(xs[xi], hist, xi, n, start, t - 3 + i, HD, col);
                    ys[xi][t * HD + col] = acc;
                }
            }
            for (int64_t h = 0; h < n_heads; ++h) {
                for (int xi = 0; xi < 2; ++xi) {           /* q and k: unit L2 norm per head */
                    double *y = ys[xi] + t * HD + h * d;
                    double ss = 0.0;
                    for (int64_t c = 0; c < d; ++c) ss += y[c] * y[c];
                    double nrm = sqrt(ss);
                    if (nrm < eps) nrm = eps;
                    for (int64_t c = 0; c < d; ++c) y[c] /= nrm;
                }
                for (int64_t c = 0; c < d; ++c) {
                    const double x = a[t * HD + h * d + c];
                    const double softplus = x > 30.0 ? x + log1p(exp(-x)) : log1p(exp(x));
                    g[t * HD + h * d + c] = clamp_logdecay(-softplus);
                }
                beta[t * n_heads + h] = 1.0 / (1.0 + exp(-b[t * n_heads + h]));
            }
        }
    }
    return KDA_ORACLE_OK;
}

/*
 * Output gate: the page (same section, third paragraph) gives KDA an input-dependent output gate
 * acting on the output of its attention path.  Reading fixed here: an elementwise sigmoid gate,
 * out = o * 1 / (1 + exp(-z)), with z the gate's pre-activation for the same (token, head,
 * channel); no normalisation in front of it.
 */
int kda_oracle_output_gate(const double *o, const double *z, int64_t n, double *out)
{
    if (n < 0) return KDA_ORACLE_EINVAL;
    for (int64_t i = 0; i < n; ++i) out[i] = o[i] / (1.0 + exp(-z[i]));
    return KDA_ORACLE_OK;
}
