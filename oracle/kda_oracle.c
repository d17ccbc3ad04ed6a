/*
 * kda_oracle.c -- FP64 CPU oracle of the KDA (Kimi Delta Attention) gated
 * delta-rule serving path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the CUDA library computes.  Only the tests, the smoke
 * check and the CPU-baseline leg of the benchmark may load it.  It shares no
 * code, header, table or helper with the CUDA path.
 *
 * What it computes (per head, token by token, in double precision from the
 * BF16-rounded inputs, which the caller passes already widened to float):
 *
 *   fold      q <- q / sqrt(sum q^2 + 1e-6), k likewise      (use_qk_l2norm)
 *             beta <- sigmoid(beta_raw)                        (beta_is_raw)
 *             g[c] <- lower_bound * sigmoid(exp(A_log[h]) * (a[c] + dt_bias[h,c]))
 *                                                  (bounded gate, A_log given)
 *             g[c] <- input as given                           (A_log absent)
 *   update    S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *   output    o_t = scale * S_t^T q_t
 *
 * S is a K x V matrix per head.  The pages ("[KDA] Support Helion MTP
 * verification and harden prefill, decode", sglang PR #42857, Motivation and
 * Modifications) name the three serving phases and their flags but do not
 * print the update rule; the rule above is the KDA gated delta rule as this
 * library defines it.
 *
 * State layout follows the pool contract of the packed-decode validator
 * ("PR #35197 report: fix(kernel) Fix Helion small-token prefill bug", key
 * source snippet of kda_decode.py: `HV, V, K = initial_state.shape[-3:]`):
 * pool[slot][head][j][c] holds S[c][j], key index fastest.
 *
 * Phases:
 *   kdao_prefill  chunk_kda contract (same report, snippet of kda_prefill.py):
 *                 an indexed initial-state pool is required, g/beta may carry
 *                 padding rows beyond the token count which are never read,
 *                 sequences are delimited by cu_seqlens (or equal lengths).
 *   kdao_decode   packed single-token decode: one row of mixed_qkv per request
 *                 holding [q (H*K) | k (H*K) | v (HV*V)], gate input a
 *                 [B, HV*K] (the validator checks a.shape[1] == HV*K).
 *   kdao_verify   chain / tree speculative verify writing the state after
 *                 every draft token as a per-candidate snapshot (PR #42857,
 *                 Modifications: "chain/tree verification with per-candidate
 *                 state snapshots").
 *   kdao_commit   copies the accepted snapshot into the pool (PR #42857 review
 *                 thread: verify, commit a partially accepted prefix, replay).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - L2-norm epsilon 1e-6 inside the square root; scale applied after the norm.
 *   - A_log [HV] and dt_bias [HV*K] in FP32; no unbounded gate formula.
 *   - state slot -1 marks a padding request: skipped, its o rows are zero,
 *     its pool slot and snapshots are not written.
 *   - intermediate states: the state at the start of every chunk of every
 *     sequence, [sum_n ceil(T_n/chunk), HV, V, K], sequence-major.
 *   - snapshot[b][i] is the state after consuming draft token i; a tree node's
 *     state is one step from its parent's state (parent -1 = pool state).
 *   - grouped value heads: HV may be a multiple of H, and value head h then
 *     takes its q and k from q/k head h / (HV / H) (all other per-head
 *     inputs, the gate parameters and the state are per value head).  The
 *     pages' packed-decode validator reads HV from the state shape and checks
 *     the gate input against HV*K, while the q and k widths of a packed row
 *     follow H; the grouping itself is not printed there, and this is the
 *     plainest reading.
 *
 * Build: gcc -O2 -std=c11 -Wall -Werror -ffp-contract=off -fPIC -shared -o libkda_oracle.so
 *        kda_oracle.c -lm -lpthread
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int H, HV, K, V;
  const float *A_log;   /* [HV] or NULL */
  const float *dt_bias; /* [HV*K] or NULL (zero bias) */
  double lower_bound;
  int beta_is_raw;
  int use_qk_l2norm;
  double scale;
} kdao_params;

enum {
  KDAO_OK = 0,
  KDAO_ERR_ARG = 1,
  KDAO_ERR_SLOT = 2,
  KDAO_ERR_PARENT = 3,
  KDAO_ERR_SEQLENS = 4,
  KDAO_ERR_NOMEM = 5
};

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* A0 fold of one token of one head: normalised q and k, the per-channel
 * log-decay g and the write strength beta. */
static void fold_token(const kdao_params *p, int h, const float *q_in,
                       const float *k_in, const float *g_in, float b_in,
                       double *q, double *k, double *g, double *beta) {
  const int K = p->K;
  double sq = 0.0, sk = 0.0;
  for (int c = 0; c < K; ++c) {
    q[c] = q_in[c];
    k[c] = k_in[c];
    sq += q[c] * q[c];
    sk += k[c] * k[c];
  }
  if (p->use_qk_l2norm) {
    const double rq = 1.0 / sqrt(sq + 1e-6), rk = 1.0 / sqrt(sk + 1e-6);
    for (int c = 0; c < K; ++c) {
      q[c] *= rq;
      k[c] *= rk;
    }
  }
  for (int c = 0; c < K; ++c) {
    if (p->A_log) {
      const double bias = p->dt_bias ? (double)p->dt_bias[h * K + c] : 0.0;
      g[c] = p->lower_bound *
             sigmoid(exp((double)p->A_log[h]) * ((double)g_in[c] + bias));
    } else {
      g[c] = g_in[c];
    }
  }
  *beta = p->beta_is_raw ? sigmoid((double)b_in) : (double)b_in;
}

/* One step of the gated delta rule on one head.
 * st: S^T in pool layout, st[j*K + c] = S[c][j].
 * work: scratch of V doubles.  g is overwritten with exp(g).
 *   X = Diag(exp(g)) S
 *   S = (I - beta k k^T) X + beta k v^T, applying (I - beta k k^T) to X as
 *       X - beta k (k^T X)
 *   o = scale * S^T q                                                     */
static void gated_delta_step(int K, int V, double *st, const double *q,
                             const double *k, const float *v, double *g,
                             double beta, double scale, double *o,
                             double *work) {
  for (int c = 0; c < K; ++c) g[c] = exp(g[c]); /* Diag(exp(g)), g consumed */
  for (int j = 0; j < V; ++j)
    for (int c = 0; c < K; ++c) st[j * K + c] *= g[c];
  for (int j = 0; j < V; ++j) { /* work = k^T X */
    double s = 0.0;
    for (int c = 0; c < K; ++c) s += k[c] * st[j * K + c];
    work[j] = s;
  }
  for (int j = 0; j < V; ++j)
    for (int c = 0; c < K; ++c) st[j * K + c] -= beta * k[c] * work[j];
  for (int j = 0; j < V; ++j)
    for (int c = 0; c < K; ++c) st[j * K + c] += beta * k[c] * (double)v[j];
  if (o) {
    for (int j = 0; j < V; ++j) {
      double s = 0.0;
      for (int c = 0; c < K; ++c) s += st[j * K + c] * q[c];
      o[j] = scale * s;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Minimal static work split over pthreads.                                  */

typedef void (*unit_fn)(void *ctx, long unit, double *scratch);

typedef struct {
  unit_fn fn;
  void *ctx;
  long units;
  int tid, nthreads;
  size_t scratch_doubles;
  int failed;
} worker_arg;

static void *worker_main(void *argp) {
  worker_arg *a = (worker_arg *)argp;
  double *scratch = (double *)malloc(a->scratch_doubles * sizeof(double));
  if (!scratch) {
    a->failed = 1;
    return NULL;
  }
  for (long u = a->tid; u < a->units; u += a->nthreads) a->fn(a->ctx, u, scratch);
  free(scratch);
  return NULL;
}

static int run_units(unit_fn fn, void *ctx, long units, int nthreads,
                     size_t scratch_doubles) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > units) nthreads = (int)(units > 0 ? units : 1);
  worker_arg *args = (worker_arg *)calloc((size_t)nthreads, sizeof(worker_arg));
  pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!args || !th) {
    free(args);
    free(th);
    return KDAO_ERR_NOMEM;
  }
  int rc = KDAO_OK;
  for (int i = 0; i < nthreads; ++i) {
    args[i] = (worker_arg){fn, ctx, units, i, nthreads, scratch_doubles, 0};
    if (nthreads == 1) {
      worker_main(&args[i]);
    } else if (pthread_create(&th[i], NULL, worker_main, &args[i]) != 0) {
      worker_main(&args[i]); /* run inline if a thread cannot be made */
      args[i].nthreads = -1;
    }
  }
  for (int i = 0; i < nthreads; ++i) {
    if (nthreads > 1 && args[i].nthreads != -1) pthread_join(th[i], NULL);
    if (args[i].failed) rc = KDAO_ERR_NOMEM;
  }
  free(args);
  free(th);
  return rc;
}

static size_t step_scratch(const kdao_params *p) {
  /* q, k, g (K each), work (V), state copy (K*V) */
  return (size_t)3 * p->K + (size_t)p->V + (size_t)p->K * p->V;
}

/* head counts: HV value heads in groups over H q/k heads */
static int heads_ok(const kdao_params *p) {
  return p->H >= 1 && p->HV >= p->H && p->HV % p->H == 0;
}

static int slots_distinct_and_valid(const int *idx, int n, int pool_slots) {
  for (int i = 0; i < n; ++i) {
    if (idx[i] < -1 || idx[i] >= pool_slots) return KDAO_ERR_SLOT;
    if (idx[i] < 0) continue;
    for (int j = 0; j < i; ++j)
      if (idx[j] == idx[i]) return KDAO_ERR_SLOT;
  }
  return KDAO_OK;
}

/* ------------------------------------------------------------------------ */
/* Prefill: chunk_kda contract.                                              */

typedef struct {
  const kdao_params *p;
  const float *q, *k, *v, *g, *beta;
  double *pool;
  const int *state_idx;
  const long *seq_start; /* [num_seqs+1] */
  const long *chunk_base; /* [num_seqs] first intermediate index per seq */
  int chunk;
  double *o;
  double *intermediate;
} prefill_ctx;

static void prefill_unit(void *vctx, long unit, double *scratch) {
  const prefill_ctx *cx = (const prefill_ctx *)vctx;
  const kdao_params *p = cx->p;
  const int H = p->H, HV = p->HV, K = p->K, V = p->V;
  const long n = unit / HV;
  const int h = (int)(unit % HV);
  const int slot = cx->state_idx[n];
  const long t0 = cx->seq_start[n], t1 = cx->seq_start[n + 1];
  double *q = scratch, *k = q + K, *g = k + K, *work = g + K, *st = work + V;
  if (slot < 0) { /* padding sequence: outputs are zero, pool untouched */
    for (long t = t0; t < t1; ++t)
      for (int j = 0; j < V; ++j) cx->o[(t * HV + h) * V + j] = 0.0;
    return;
  }
  double *src = cx->pool + ((long)slot * HV + h) * (long)V * K;
  memcpy(st, src, sizeof(double) * (size_t)K * V);
  for (long t = t0; t < t1; ++t) {
    if (cx->intermediate && (t - t0) % cx->chunk == 0) {
      const long ci = cx->chunk_base[n] + (t - t0) / cx->chunk;
      memcpy(cx->intermediate + (ci * HV + h) * (long)V * K, st,
             sizeof(double) * (size_t)K * V);
    }
    double beta;
    const int hk = h / (HV / H); /* q/k head of value head h */
    fold_token(p, h, cx->q + (t * H + hk) * K, cx->k + (t * H + hk) * K,
               cx->g + (t * HV + h) * K, cx->beta[t * HV + h], q, k, g, &beta);
    gated_delta_step(K, V, st, q, k, cx->v + (t * HV + h) * V, g, beta, p->scale,
                     cx->o + (t * HV + h) * V, work);
  }
  memcpy(src, st, sizeof(double) * (size_t)K * V);
}

/* q,k [T,H,K]; v [T,HV,V]; g [gb_rows,HV,K]; beta [gb_rows,HV] (rows >= T are
 * padding and never read); pool [slots,HV,V,K] updated in place; o [T,HV,V];
 * intermediate NULL or [sum ceil(T_n/chunk),HV,V,K]. */
int kdao_prefill(const kdao_params *p, const float *q, const float *k,
                 const float *v, const float *g, const float *beta,
                 long gb_rows, double *pool, int pool_slots,
                 const int *state_idx, const int *cu_seqlens, int num_seqs,
                 long total_tokens, int chunk, double *o, double *intermediate,
                 int nthreads) {
  if (!p || !pool || !state_idx || num_seqs < 1 || total_tokens < 0 ||
      chunk < 1 || !heads_ok(p))
    return KDAO_ERR_ARG;
  if (gb_rows < total_tokens) return KDAO_ERR_ARG; /* g/beta must cover q */
  int rc = slots_distinct_and_valid(state_idx, num_seqs, pool_slots);
  if (rc) return rc;
  long *seq_start = (long *)malloc(sizeof(long) * (size_t)(num_seqs + 1));
  long *chunk_base = (long *)malloc(sizeof(long) * (size_t)num_seqs);
  if (!seq_start || !chunk_base) {
    free(seq_start);
    free(chunk_base);
    return KDAO_ERR_NOMEM;
  }
  if (cu_seqlens) {
    for (int i = 0; i <= num_seqs; ++i) seq_start[i] = cu_seqlens[i];
  } else {
    if (total_tokens % num_seqs) {
      free(seq_start);
      free(chunk_base);
      return KDAO_ERR_SEQLENS;
    }
    for (int i = 0; i <= num_seqs; ++i)
      seq_start[i] = (total_tokens / num_seqs) * i;
  }
  rc = KDAO_OK;
  if (seq_start[0] != 0 || seq_start[num_seqs] != total_tokens) rc = KDAO_ERR_SEQLENS;
  long nchunks = 0;
  for (int i = 0; i < num_seqs && !rc; ++i) {
    if (seq_start[i + 1] < seq_start[i]) rc = KDAO_ERR_SEQLENS;
    chunk_base[i] = nchunks;
    nchunks += (seq_start[i + 1] - seq_start[i] + chunk - 1) / chunk;
  }
  if (!rc) {
    prefill_ctx cx = {p, q, k, v, g, beta, pool, state_idx, seq_start,
                      chunk_base, chunk, o, intermediate};
    rc = run_units(prefill_unit, &cx, (long)num_seqs * p->HV, nthreads,
                   step_scratch(p));
  }
  free(seq_start);
  free(chunk_base);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Packed decode.                                                            */

typedef struct {
  const kdao_params *p;
  const float *mixed_qkv;
  long row_stride;
  const float *a, *b;
  double *pool;
  const int *state_idx;
  double *o;
} decode_ctx;

static void decode_unit(void *vctx, long unit, double *scratch) {
  const decode_ctx *cx = (const decode_ctx *)vctx;
  const kdao_params *p = cx->p;
  const int H = p->H, HV = p->HV, K = p->K, V = p->V;
  const long r = unit / HV;
  const int h = (int)(unit % HV);
  const int slot = cx->state_idx[r];
  double *q = scratch, *k = q + K, *g = k + K, *work = g + K;
  double *o = cx->o + (r * HV + h) * V;
  if (slot < 0) {
    for (int j = 0; j < V; ++j) o[j] = 0.0;
    return;
  }
  const float *row = cx->mixed_qkv + r * cx->row_stride;
  double beta;
  const int hk = h / (HV / H); /* q/k head of value head h */
  fold_token(p, h, row + hk * K, row + (long)H * K + hk * K,
             cx->a + (r * HV + h) * K, cx->b[r * HV + h], q, k, g, &beta);
  gated_delta_step(K, V, cx->pool + ((long)slot * HV + h) * (long)V * K, q, k,
                   row + 2L * H * K + (long)h * V, g, beta, p->scale, o, work);
}

int kdao_decode(const kdao_params *p, const float *mixed_qkv, long row_stride,
                const float *a, const float *b, int B, double *pool,
                int pool_slots, const int *state_idx, double *o, int nthreads) {
  if (!p || !pool || !state_idx || B < 0 || !heads_ok(p) ||
      row_stride < 2L * p->H * p->K + (long)p->HV * p->V)
    return KDAO_ERR_ARG;
  int rc = slots_distinct_and_valid(state_idx, B, pool_slots);
  if (rc) return rc;
  decode_ctx cx = {p, mixed_qkv, row_stride, a, b, pool, state_idx, o};
  return run_units(decode_unit, &cx, (long)B * p->HV, nthreads, step_scratch(p));
}

/* ------------------------------------------------------------------------ */
/* Chain / tree verify with per-candidate snapshots.                         */

typedef struct {
  const kdao_params *p;
  const float *mixed_qkv;
  long row_stride;
  const float *a, *b;
  int T;
  const int *parent; /* NULL: chain */
  const double *pool;
  const int *state_idx;
  double *o;
  double *snapshots;
} verify_ctx;

static void verify_unit(void *vctx, long unit, double *scratch) {
  const verify_ctx *cx = (const verify_ctx *)vctx;
  const kdao_params *p = cx->p;
  const int H = p->H, HV = p->HV, K = p->K, V = p->V, T = cx->T;
  const long r = unit / HV;
  const int h = (int)(unit % HV);
  const int slot = cx->state_idx[r];
  const long hs = (long)V * K;
  double *q = scratch, *k = q + K, *g = k + K, *work = g + K, *st = work + V;
  if (slot < 0) {
    for (int i = 0; i < T; ++i)
      for (int j = 0; j < V; ++j) cx->o[((r * T + i) * HV + h) * V + j] = 0.0;
    return;
  }
  const double *root = cx->pool + ((long)slot * HV + h) * hs;
  for (int i = 0; i < T; ++i) {
    const int par = cx->parent ? cx->parent[r * T + i] : i - 1;
    const double *src =
        par < 0 ? root : cx->snapshots + ((r * T + par) * HV + h) * hs;
    memcpy(st, src, sizeof(double) * (size_t)hs);
    const long row = r * T + i;
    const float *x = cx->mixed_qkv + row * cx->row_stride;
    double beta;
    const int hk = h / (HV / H); /* q/k head of value head h */
    fold_token(p, h, x + hk * K, x + (long)H * K + hk * K,
               cx->a + (row * HV + h) * K, cx->b[row * HV + h], q, k, g, &beta);
    gated_delta_step(K, V, st, q, k, x + 2L * H * K + (long)h * V, g, beta,
                     p->scale, cx->o + (row * HV + h) * V, work);
    memcpy(cx->snapshots + (row * HV + h) * hs, st, sizeof(double) * (size_t)hs);
  }
}

/* mixed_qkv [B*T rows]; a [B*T, HV*K]; b [B*T, HV]; parent NULL (chain) or
 * [B, T] with -1 <= parent[i] < i; pool read only; o [B,T,HV,V];
 * snapshots [B,T,HV,V,K]. */
int kdao_verify(const kdao_params *p, const float *mixed_qkv, long row_stride,
                const float *a, const float *b, int B, int T,
                const int *parent, const double *pool, int pool_slots,
                const int *state_idx, double *o, double *snapshots,
                int nthreads) {
  if (!p || !pool || !state_idx || !snapshots || B < 0 || T < 1 ||
      !heads_ok(p) || row_stride < 2L * p->H * p->K + (long)p->HV * p->V)
    return KDAO_ERR_ARG;
  int rc = slots_distinct_and_valid(state_idx, B, pool_slots);
  if (rc) return rc;
  if (parent) {
    for (long r = 0; r < B; ++r)
      for (int i = 0; i < T; ++i) {
        const int par = parent[r * T + i];
        if (par < -1 || par >= i) return KDAO_ERR_PARENT;
      }
  }
  verify_ctx cx = {p, mixed_qkv, row_stride, a, b, T, parent, pool,
                   state_idx, o, snapshots};
  return run_units(verify_unit, &cx, (long)B * p->HV, nthreads, step_scratch(p));
}

/* pool[state_idx[b]] <- snapshots[b][accepted[b]] for accepted[b] >= 0. */
int kdao_commit(const double *snapshots, int B, int T, int HV, int V, int K,
                const int *accepted, double *pool, int pool_slots,
                const int *state_idx) {
  if (!snapshots || !accepted || !pool || !state_idx || B < 0 || T < 1)
    return KDAO_ERR_ARG;
  int rc = slots_distinct_and_valid(state_idx, B, pool_slots);
  if (rc) return rc;
  const long slot_elems = (long)HV * V * K;
  for (long r = 0; r < B; ++r) {
    if (accepted[r] >= T) return KDAO_ERR_ARG;
    if (accepted[r] < 0 || state_idx[r] < 0) continue;
    memcpy(pool + (long)state_idx[r] * slot_elems,
           snapshots + (r * T + accepted[r]) * slot_elems,
           sizeof(double) * (size_t)slot_elems);
  }
  return KDAO_OK;
}
