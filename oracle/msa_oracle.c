/*
 * msa_oracle.c -- float64 CPU oracle for the MSA (MiniMax Sparse Attention) training
 * hot path.  TEST INFRASTRUCTURE ONLY: the library never links, loads or calls this
 * file; only the tests, the package's smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header or table with the CUDA path.
 *
 * Every quantity is the plain definition, written out with loops in float64 on the
 * bf16-rounded inputs.  Sources (web pages describing the method):
 *   [MSA-7m]  "MiniMax Sparse Attention (MSA): una atención dispersa en bloques de dos
 *             ramas..." (7minutos.es), sections "¿Qué es MSA?", "Cómo funcionan las dos
 *             ramas", "Cómo se entrena MSA", "El codiseño del kernel".
 *   [FMSA-k]  Flash-MSA article (tech.kuratif.com), paragraphs 3, 6, 7.
 *   [FMSA-d]  "Accelerating Million-Token Training with Sparse Attention Kernels"
 *             (deephorus.pages.dev), paragraphs 3-4.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - index logits are plain dot products q_idx . k_idx; the softmax scale of the
 *     index branch (scale_idx) only enters lse_idx, the KL and its gradients;
 *   - the local block counts inside the k-block budget (local + k-1 others);
 *   - equal pooled scores rank the lower block id first;
 *   - fewer than k visible blocks: all are taken, unused slots are -1;
 *   - the KL is KL(p_T || p_I) summed over rows and multiplied by kl_weight;
 *   - the teacher p_T is detached, so dq/dk/dv carry no KL term and only
 *     q_idx/k_idx receive the KL gradient.
 *
 * Layouts (row-major): q,dO [B][N][H_q][d]; k,v [B][N][H_kv][d];
 * q_idx [B][N][H_kv][d_idx]; k_idx [B][N][d_idx].  Head h belongs to group h / G.
 * Inputs are bf16 bit patterns (uint16).  Rows are flat ids b*N + i.
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
  int32_t B, N, H_q, H_kv, d, d_idx, Bk, topk, causal;
  double scale;     /* main softmax scale */
  double scale_idx; /* index-logit scale sigma_I */
} oracle_problem_t;

#define OR_OK 0
#define OR_EARG (-1)
#define OR_ENOMEM (-2)

static inline double bf(uint16_t x) {
  uint32_t u = (uint32_t)x << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static int check_problem(const oracle_problem_t* p) {
  if (!p || p->B < 0 || p->N < 0 || p->H_q <= 0 || p->H_kv <= 0 || p->d <= 0 ||
      p->d_idx <= 0 || p->Bk <= 0 || p->topk <= 0 || p->H_q % p->H_kv != 0)
    return OR_EARG;
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* tiny parallel-for over [0, n) tasks                                         */
/* ------------------------------------------------------------------------- */
typedef void (*task_fn)(void* ctx, int64_t task, void* scratch);
typedef struct {
  task_fn fn;
  void* ctx;
  int64_t n;
  size_t scratch_bytes;
  atomic_llong next;
  atomic_int failed;
} pool_t;

static void* pool_worker(void* arg) {
  pool_t* pl = (pool_t*)arg;
  void* scratch = pl->scratch_bytes ? malloc(pl->scratch_bytes) : NULL;
  if (pl->scratch_bytes && !scratch) {
    atomic_store(&pl->failed, 1);
    return NULL;
  }
  for (;;) {
    int64_t t = atomic_fetch_add(&pl->next, 1);
    if (t >= pl->n) break;
    pl->fn(pl->ctx, t, scratch);
  }
  free(scratch);
  return NULL;
}

static int parallel_for(task_fn fn, void* ctx, int64_t n, size_t scratch_bytes, int n_threads) {
  pool_t pl;
  pl.fn = fn;
  pl.ctx = ctx;
  pl.n = n;
  pl.scratch_bytes = scratch_bytes;
  atomic_init(&pl.next, 0);
  atomic_init(&pl.failed, 0);
  if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if ((int64_t)n_threads > n) n_threads = (int)(n > 0 ? n : 1);
  pthread_t th[256];
  int started = 0;
  for (int t = 1; t < n_threads; ++t) {
    if (pthread_create(&th[started], NULL, pool_worker, &pl) == 0) started++;
  }
  pool_worker(&pl);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  return atomic_load(&pl.failed) ? OR_ENOMEM : OR_OK;
}

/* ------------------------------------------------------------------------- */
/* element access                                                              */
/* ------------------------------------------------------------------------- */
typedef struct {
  const oracle_problem_t* p;
  const uint16_t *q, *k, *v, *q_idx, *k_idx, *dO;
} inputs_t;

static inline const uint16_t* q_row(const inputs_t* in, int64_t b, int64_t i, int h) {
  const oracle_problem_t* p = in->p;
  return in->q + (((b * p->N + i) * p->H_q + h) * (int64_t)p->d);
}
static inline const uint16_t* dO_row(const inputs_t* in, int64_t b, int64_t i, int h) {
  const oracle_problem_t* p = in->p;
  return in->dO + (((b * p->N + i) * p->H_q + h) * (int64_t)p->d);
}
static inline const uint16_t* k_row(const inputs_t* in, int64_t b, int64_t j, int g) {
  const oracle_problem_t* p = in->p;
  return in->k + (((b * p->N + j) * p->H_kv + g) * (int64_t)p->d);
}
static inline const uint16_t* v_row(const inputs_t* in, int64_t b, int64_t j, int g) {
  const oracle_problem_t* p = in->p;
  return in->v + (((b * p->N + j) * p->H_kv + g) * (int64_t)p->d);
}
static inline const uint16_t* qi_row(const inputs_t* in, int64_t b, int64_t i, int g) {
  const oracle_problem_t* p = in->p;
  return in->q_idx + (((b * p->N + i) * p->H_kv + g) * (int64_t)p->d_idx);
}
static inline const uint16_t* ki_row(const inputs_t* in, int64_t b, int64_t j) {
  const oracle_problem_t* p = in->p;
  return in->k_idx + ((b * p->N + j) * (int64_t)p->d_idx);
}

static inline double dot_bb(const uint16_t* a, const uint16_t* b, int n) {
  double s = 0.0;
  for (int t = 0; t < n; ++t) s += bf(a[t]) * bf(b[t]);
  return s;
}
static inline double dot_db(const double* a, const uint16_t* b, int n) {
  double s = 0.0;
  for (int t = 0; t < n; ++t) s += a[t] * bf(b[t]);
  return s;
}

static inline int nblocks(const oracle_problem_t* p) { return (p->N + p->Bk - 1) / p->Bk; }

/* ------------------------------------------------------------------------- */
/* index branch: scoring, block max-pooling, top-k with forced local block      */
/* [MSA-7m] "Cómo funcionan las dos ramas" paragraphs 1-2; "¿Qué es MSA?" ¶2;     */
/* [FMSA-k] ¶3 (128-token blocks by max-pooling), ¶6 (local score set to inf).   */
/* ------------------------------------------------------------------------- */

/* Pooled index score of block c for query (b, i) of group g: the maximum over the
 * block's tokens of the raw index logit q_idx[b,i,g] . k_idx[b,j]. */
static double pooled_score(const inputs_t* in, int64_t b, int64_t i, int g, int c) {
  const oracle_problem_t* p = in->p;
  const uint16_t* qi = qi_row(in, b, i, g);
  int64_t j0 = (int64_t)c * p->Bk, j1 = j0 + p->Bk;
  if (j1 > p->N) j1 = p->N;
  double m = -INFINITY;
  for (int64_t j = j0; j < j1; ++j) {
    double s = dot_bb(qi, ki_row(in, b, j), p->d_idx);
    if (s > m) m = s;
  }
  return m;
}

/* Candidate (non-local, visible) blocks of query i: causal -> every block wholly
 * before the query's own block; non-causal -> every block except the own one. */
static int is_candidate(const oracle_problem_t* p, int64_t i, int c) {
  int ci = (int)(i / p->Bk);
  if (c == ci) return 0;
  if (p->causal) return c < ci;
  return 1;
}

/* Selects the block set of (b, i, g).  sel[topk] receives the ascending block ids,
 * padded with -1.  kth[0] = pooled score of the last non-local block taken (the
 * (k-1)-th best, +inf when none is taken), kth[1] = best score left out (-inf when
 * every candidate was taken).  pooled[nb] (optional) receives candidate scores,
 * NAN for non-candidates.  scratch holds nb doubles + nb ints. */
static void select_row(const inputs_t* in, int64_t b, int64_t i, int g, int32_t* sel,
                       double* kth, double* pooled_out, void* scratch) {
  const oracle_problem_t* p = in->p;
  int nb = nblocks(p);
  double* sc = (double*)scratch;
  char* taken = (char*)(sc + nb);
  int ci = (int)(i / p->Bk);
  int ncand = 0;
  for (int c = 0; c < nb; ++c) {
    taken[c] = 0;
    if (is_candidate(p, i, c)) {
      sc[c] = pooled_score(in, b, i, g, c);
      ncand++;
    } else {
      sc[c] = NAN;
    }
    if (pooled_out) pooled_out[c] = sc[c];
  }
  /* the local block always takes one of the k slots ([MSA-7m] two branches ¶2) */
  taken[ci] = 1;
  int want = p->topk - 1;
  double last = INFINITY;
  for (int n = 0; n < want && n < ncand; ++n) {
    int best = -1;
    for (int c = 0; c < nb; ++c) {
      if (taken[c] || isnan(sc[c])) continue;
      if (best < 0 || sc[c] > sc[best]) best = c; /* strict: ties keep the lower id */
    }
    taken[best] = 1;
    last = sc[best];
  }
  double runner = -INFINITY;
  for (int c = 0; c < nb; ++c)
    if (!taken[c] && !isnan(sc[c]) && sc[c] > runner) runner = sc[c];
  int n = 0;
  for (int c = 0; c < nb && n < p->topk; ++c)
    if (taken[c]) sel[n++] = c;
  for (; n < p->topk; ++n) sel[n] = -1;
  if (kth) {
    kth[0] = last;
    kth[1] = runner;
  }
}

/* Token set T of a row: the tokens of the selected blocks that the query may see
 * ([MSA-7m] two branches ¶3: causally visible tokens of the selected blocks).
 * Returns |T|; toks receives them in ascending order. */
static int token_set(const oracle_problem_t* p, int64_t i, const int32_t* sel, int64_t* toks) {
  int n = 0;
  for (int s = 0; s < p->topk; ++s) {
    int c = sel[s];
    if (c < 0) continue;
    int64_t j0 = (int64_t)c * p->Bk, j1 = j0 + p->Bk;
    if (j1 > p->N) j1 = p->N;
    for (int64_t j = j0; j < j1; ++j) {
      if (p->causal && j > i) break;
      toks[n++] = j;
    }
  }
  return n;
}

/* ------------------------------------------------------------------------- */
/* public: selection                                                           */
/* ------------------------------------------------------------------------- */
typedef struct {
  inputs_t in;
  const int64_t* rows;
  int64_t n_rows;
  int32_t* block_idx;
  double* kth;
  double* pooled;
} sel_ctx_t;

static inline int64_t row_id(const int64_t* rows, int64_t r) { return rows ? rows[r] : r; }

static void sel_task(void* vctx, int64_t t, void* scratch) {
  sel_ctx_t* cx = (sel_ctx_t*)vctx;
  const oracle_problem_t* p = cx->in.p;
  int64_t r = t / p->H_kv;
  int g = (int)(t % p->H_kv);
  int64_t flat = row_id(cx->rows, r);
  int64_t b = flat / p->N, i = flat % p->N;
  int nb = nblocks(p);
  select_row(&cx->in, b, i, g, cx->block_idx + t * p->topk, cx->kth ? cx->kth + 2 * t : NULL,
             cx->pooled ? cx->pooled + t * (int64_t)nb : NULL, scratch);
}

/* block_idx [n_rows][H_kv][topk]; kth [n_rows][H_kv][2] (nullable);
 * pooled [n_rows][H_kv][nb] (nullable). rows NULL = every row b*N+i in order. */
int oracle_select(const oracle_problem_t* p, const uint16_t* q_idx, const uint16_t* k_idx,
                  const int64_t* rows, int64_t n_rows, int32_t* block_idx, double* kth,
                  double* pooled, int n_threads) {
  if (check_problem(p) || !q_idx || !k_idx || !block_idx) return OR_EARG;
  if (!rows) n_rows = (int64_t)p->B * p->N;
  sel_ctx_t cx = {{p, NULL, NULL, NULL, q_idx, k_idx, NULL}, rows, n_rows, block_idx, kth, pooled};
  int nb = nblocks(p);
  return parallel_for(sel_task, &cx, n_rows * p->H_kv, (size_t)nb * (sizeof(double) + 1) + 64,
                      n_threads);
}

/* ------------------------------------------------------------------------- */
/* main branch forward + index LSE                                             */
/* [MSA-7m] two branches ¶3 (exact scaled-dot-product softmax over the token set, */
/* every head of the group shares the set); [FMSA-k] ¶6 (LSE kept for backward);  */
/* [FMSA-d] ¶4 (index LSE recomputed over the selected tokens).                 */
/* ------------------------------------------------------------------------- */
typedef struct {
  inputs_t in;
  const int64_t* rows;
  int64_t n_rows;
  const int32_t* block_idx;
  double *o, *lse, *lse_idx;
} fwd_ctx_t;

/* log of the sum of exp(x[t]) */
static double logsumexp(const double* x, int n) {
  double m = -INFINITY;
  for (int t = 0; t < n; ++t)
    if (x[t] > m) m = x[t];
  if (m == -INFINITY) return -INFINITY;
  double s = 0.0;
  for (int t = 0; t < n; ++t) s += exp(x[t] - m);
  return m + log(s);
}

static void fwd_task(void* vctx, int64_t t, void* scratch) {
  fwd_ctx_t* cx = (fwd_ctx_t*)vctx;
  const inputs_t* in = &cx->in;
  const oracle_problem_t* p = in->p;
  int G = p->H_q / p->H_kv;
  int64_t r = t / p->H_kv;
  int g = (int)(t % p->H_kv);
  int64_t flat = row_id(cx->rows, r);
  int64_t b = flat / p->N, i = flat % p->N;
  int64_t* toks = (int64_t*)scratch;
  double* s = (double*)(toks + (int64_t)p->topk * p->Bk);
  int nT = token_set(p, i, cx->block_idx + t * p->topk, toks);
  for (int hh = 0; hh < G && (cx->o || cx->lse); ++hh) {
    int h = g * G + hh;
    const uint16_t* qh = q_row(in, b, i, h);
    for (int n = 0; n < nT; ++n) s[n] = p->scale * dot_bb(qh, k_row(in, b, toks[n], g), p->d);
    double lse = logsumexp(s, nT);
    double* o = cx->o ? cx->o + (r * p->H_q + h) * (int64_t)p->d : NULL;
    if (o) {
      for (int e = 0; e < p->d; ++e) o[e] = 0.0;
      for (int n = 0; n < nT; ++n) {
        double P = exp(s[n] - lse);
        const uint16_t* vr = v_row(in, b, toks[n], g);
        for (int e = 0; e < p->d; ++e) o[e] += P * bf(vr[e]);
      }
    }
    if (cx->lse) cx->lse[r * p->H_q + h] = lse;
  }
  if (cx->lse_idx) {
    const uint16_t* qi = qi_row(in, b, i, g);
    for (int n = 0; n < nT; ++n) s[n] = p->scale_idx * dot_bb(qi, ki_row(in, b, toks[n]), p->d_idx);
    cx->lse_idx[r * p->H_kv + g] = logsumexp(s, nT);
  }
}

/* o [n_rows][H_q][d], lse [n_rows][H_q], lse_idx [n_rows][H_kv]; each nullable.
 * block_idx [n_rows][H_kv][topk] gives the block sets of the rows (from
 * oracle_select, or any other valid selection). */
int oracle_forward(const oracle_problem_t* p, const uint16_t* q, const uint16_t* k,
                   const uint16_t* v, const uint16_t* q_idx, const uint16_t* k_idx,
                   const int64_t* rows, int64_t n_rows, const int32_t* block_idx, double* o,
                   double* lse, double* lse_idx, int n_threads) {
  if (check_problem(p) || !block_idx) return OR_EARG;
  if ((o || lse) && (!q || !k || !v)) return OR_EARG;
  if (lse_idx && (!q_idx || !k_idx)) return OR_EARG;
  if (!rows) n_rows = (int64_t)p->B * p->N;
  fwd_ctx_t cx = {{p, q, k, v, q_idx, k_idx, NULL}, rows, n_rows, block_idx, o, lse, lse_idx};
  size_t scratch = (size_t)p->topk * p->Bk * (sizeof(int64_t) + sizeof(double)) + 64;
  return parallel_for(fwd_task, &cx, n_rows * p->H_kv, scratch, n_threads);
}

/* ------------------------------------------------------------------------- */
/* backward: main-branch gradients and the KL alignment gradient                */
/* [FMSA-k] ¶7 (proxy and main gradients together, reusing cached block ids);    */
/* [MSA-7m] "Cómo se entrena MSA" ¶1-2 (KL toward the group-averaged main         */
/* distribution over the selected tokens; stop-gradient so only the index        */
/* projections receive it).                                                     */
/*                                                                             */
/* Pass A, one task per (row, group): everything that belongs to the row:        */
/*   P_h = softmax(scale q_h . k_j) over T, o_h, D_h = dO_h . o_h,                */
/*   dS_h[j] = P_h[j] (dO_h . v_j - D_h),  dq_h = scale sum_j dS_h[j] k_j,        */
/*   z_j = q_idx . k_idx_j,  lse_idx = log sum_j exp(scale_idx z_j),              */
/*   p_I = exp(scale_idx z - lse_idx),  p_T = mean_h P_h,                         */
/*   dz = w (p_I - p_T),  dq_idx = scale_idx sum_j dz_j k_idx_j,                  */
/*   KL_row = sum_j p_T (log p_T - log p_I).                                      */
/* Pass B, one task per (batch, key block): the sums over rows for each key:      */
/*   dk_j = scale sum dS_h[j] q_h,  dv_j = sum P_h[j] dO_h,                       */
/*   dk_idx_j = scale_idx sum dz_j q_idx   (over every row, head and group that   */
/*   attends to j).                                                             */
/* ------------------------------------------------------------------------- */
typedef struct {
  inputs_t in;
  const int64_t* rows;
  int64_t n_rows;
  const int32_t* block_idx;
  double w;
  double *dq, *dk, *dv, *dq_idx, *dk_idx;
  double* row_lse;     /* [n_rows][H_q] */
  double* row_D;       /* [n_rows][H_q] */
  double* row_lse_idx; /* [n_rows][H_kv] */
  double* row_kl;      /* [n_rows][H_kv] */
  int64_t* batch_start; /* [B+1]: rows of batch b are [batch_start[b], batch_start[b+1]) */
} bwd_ctx_t;

static void bwd_row_task(void* vctx, int64_t t, void* scratch) {
  bwd_ctx_t* cx = (bwd_ctx_t*)vctx;
  const inputs_t* in = &cx->in;
  const oracle_problem_t* p = in->p;
  int G = p->H_q / p->H_kv;
  int64_t r = t / p->H_kv;
  int g = (int)(t % p->H_kv);
  int64_t flat = row_id(cx->rows, r);
  int64_t b = flat / p->N, i = flat % p->N;
  int64_t TK = (int64_t)p->topk * p->Bk;
  int64_t* toks = (int64_t*)scratch;
  double* s = (double*)(toks + TK);
  double* pT = s + TK;
  double* o = pT + TK;
  int nT = token_set(p, i, cx->block_idx + t * p->topk, toks);
  for (int n = 0; n < nT; ++n) pT[n] = 0.0;

  for (int hh = 0; hh < G; ++hh) {
    int h = g * G + hh;
    const uint16_t* qh = q_row(in, b, i, h);
    const uint16_t* dOh = dO_row(in, b, i, h);
    for (int n = 0; n < nT; ++n) s[n] = p->scale * dot_bb(qh, k_row(in, b, toks[n], g), p->d);
    double lse = logsumexp(s, nT);
    for (int e = 0; e < p->d; ++e) o[e] = 0.0;
    for (int n = 0; n < nT; ++n) {
      s[n] = exp(s[n] - lse); /* s now holds P_h */
      const uint16_t* vr = v_row(in, b, toks[n], g);
      for (int e = 0; e < p->d; ++e) o[e] += s[n] * bf(vr[e]);
    }
    double D = dot_db(o, dOh, p->d);
    double* dq = cx->dq + (r * p->H_q + h) * (int64_t)p->d;
    for (int e = 0; e < p->d; ++e) dq[e] = 0.0;
    for (int n = 0; n < nT; ++n) {
      double dP = dot_bb(dOh, v_row(in, b, toks[n], g), p->d);
      double dS = s[n] * (dP - D);
      const uint16_t* kr = k_row(in, b, toks[n], g);
      for (int e = 0; e < p->d; ++e) dq[e] += p->scale * dS * bf(kr[e]);
      pT[n] += s[n] / (double)G;
    }
    cx->row_lse[r * p->H_q + h] = lse;
    cx->row_D[r * p->H_q + h] = D;
  }

  const uint16_t* qi = qi_row(in, b, i, g);
  for (int n = 0; n < nT; ++n) s[n] = p->scale_idx * dot_bb(qi, ki_row(in, b, toks[n]), p->d_idx);
  double lse_idx = logsumexp(s, nT);
  double* dqi = cx->dq_idx + (r * p->H_kv + g) * (int64_t)p->d_idx;
  for (int e = 0; e < p->d_idx; ++e) dqi[e] = 0.0;
  double kl = 0.0;
  for (int n = 0; n < nT; ++n) {
    double logpI = s[n] - lse_idx;
    double pI = exp(logpI);
    double dz = cx->w * (pI - pT[n]);
    const uint16_t* kr = ki_row(in, b, toks[n]);
    for (int e = 0; e < p->d_idx; ++e) dqi[e] += p->scale_idx * dz * bf(kr[e]);
    if (pT[n] > 0.0) kl += pT[n] * (log(pT[n]) - logpI);
  }
  cx->row_lse_idx[r * p->H_kv + g] = lse_idx;
  cx->row_kl[r * p->H_kv + g] = kl;
}

static int sel_has(const int32_t* sel, int topk, int c) {
  for (int s = 0; s < topk; ++s)
    if (sel[s] == c) return 1;
  return 0;
}

static void bwd_key_task(void* vctx, int64_t t, void* scratch) {
  bwd_ctx_t* cx = (bwd_ctx_t*)vctx;
  const inputs_t* in = &cx->in;
  const oracle_problem_t* p = in->p;
  (void)scratch;
  int G = p->H_q / p->H_kv;
  int nb = nblocks(p);
  int64_t b = t / nb;
  int c = (int)(t % nb);
  int64_t j0 = (int64_t)c * p->Bk, j1 = j0 + p->Bk;
  if (j1 > p->N) j1 = p->N;
  for (int64_t r = cx->batch_start[b]; r < cx->batch_start[b + 1]; ++r) {
    int64_t i = row_id(cx->rows, r) % p->N;
    for (int g = 0; g < p->H_kv; ++g) {
      const int32_t* sel = cx->block_idx + (r * p->H_kv + g) * p->topk;
      if (!sel_has(sel, p->topk, c)) continue;
      const uint16_t* qi = qi_row(in, b, i, g);
      double lse_idx = cx->row_lse_idx[r * p->H_kv + g];
      for (int64_t j = j0; j < j1; ++j) {
        if (p->causal && j > i) break;
        const uint16_t* kr = k_row(in, b, j, g);
        const uint16_t* vr = v_row(in, b, j, g);
        double* dk = cx->dk + ((b * p->N + j) * p->H_kv + g) * (int64_t)p->d;
        double* dv = cx->dv + ((b * p->N + j) * p->H_kv + g) * (int64_t)p->d;
        double pT = 0.0;
        for (int hh = 0; hh < G; ++hh) {
          int h = g * G + hh;
          const uint16_t* qh = q_row(in, b, i, h);
          const uint16_t* dOh = dO_row(in, b, i, h);
          double P = exp(p->scale * dot_bb(qh, kr, p->d) - cx->row_lse[r * p->H_q + h]);
          double dS = P * (dot_bb(dOh, vr, p->d) - cx->row_D[r * p->H_q + h]);
          for (int e = 0; e < p->d; ++e) {
            dk[e] += p->scale * dS * bf(qh[e]);
            dv[e] += P * bf(dOh[e]);
          }
          pT += P / (double)G;
        }
        double pI = exp(p->scale_idx * dot_bb(qi, ki_row(in, b, j), p->d_idx) - lse_idx);
        double dz = cx->w * (pI - pT);
        double* dki = cx->dk_idx + (b * p->N + j) * (int64_t)p->d_idx;
        for (int e = 0; e < p->d_idx; ++e) dki[e] += p->scale_idx * dz * bf(qi[e]);
      }
    }
  }
}

/* Gradients of the rows listed (all rows when rows is NULL; rows must be sorted).
 *   dq [n_rows][H_q][d], dq_idx [n_rows][H_kv][d_idx]        (per listed row)
 *   dk, dv [B][N][H_kv][d], dk_idx [B][N][d_idx]              (full size; the sum of
 *       the listed rows' contributions; zeroed here)
 *   kl_rows [n_rows][H_kv] (nullable): KL_row, without the weight
 *   kl: kl_weight * sum of KL_row over the listed rows and groups.
 * kl_weight is the per-row weight w of the KL term (e.g. coef / (B*H_kv*N)). */
int oracle_backward(const oracle_problem_t* p, const uint16_t* q, const uint16_t* k,
                    const uint16_t* v, const uint16_t* q_idx, const uint16_t* k_idx,
                    const uint16_t* dO, const int64_t* rows, int64_t n_rows,
                    const int32_t* block_idx, double kl_weight, double* dq, double* dk,
                    double* dv, double* dq_idx, double* dk_idx, double* kl_rows, double* kl,
                    int n_threads) {
  if (check_problem(p) || !q || !k || !v || !q_idx || !k_idx || !dO || !block_idx || !dq ||
      !dk || !dv || !dq_idx || !dk_idx || !kl)
    return OR_EARG;
  if (!rows) n_rows = (int64_t)p->B * p->N;
  for (int64_t r = 1; rows && r < n_rows; ++r)
    if (rows[r] <= rows[r - 1]) return OR_EARG;
  bwd_ctx_t cx;
  memset(&cx, 0, sizeof cx);
  cx.in = (inputs_t){p, q, k, v, q_idx, k_idx, dO};
  cx.rows = rows;
  cx.n_rows = n_rows;
  cx.block_idx = block_idx;
  cx.w = kl_weight;
  cx.dq = dq;
  cx.dk = dk;
  cx.dv = dv;
  cx.dq_idx = dq_idx;
  cx.dk_idx = dk_idx;
  int rc = OR_ENOMEM;
  cx.row_lse = (double*)malloc(sizeof(double) * (size_t)(n_rows * p->H_q + 1));
  cx.row_D = (double*)malloc(sizeof(double) * (size_t)(n_rows * p->H_q + 1));
  cx.row_lse_idx = (double*)malloc(sizeof(double) * (size_t)(n_rows * p->H_kv + 1));
  cx.row_kl = (double*)malloc(sizeof(double) * (size_t)(n_rows * p->H_kv + 1));
  cx.batch_start = (int64_t*)malloc(sizeof(int64_t) * (size_t)(p->B + 1));
  if (!cx.row_lse || !cx.row_D || !cx.row_lse_idx || !cx.row_kl || !cx.batch_start) goto done;
  {
    int64_t r = 0;
    for (int64_t b = 0; b <= p->B; ++b) {
      while (r < n_rows && row_id(rows, r) / p->N < b) ++r;
      cx.batch_start[b] = r;
    }
  }
  memset(dk, 0, sizeof(double) * (size_t)p->B * p->N * p->H_kv * p->d);
  memset(dv, 0, sizeof(double) * (size_t)p->B * p->N * p->H_kv * p->d);
  memset(dk_idx, 0, sizeof(double) * (size_t)p->B * p->N * p->d_idx);
  {
    int64_t TK = (int64_t)p->topk * p->Bk;
    size_t scratch = (size_t)TK * (sizeof(int64_t) + 2 * sizeof(double)) +
                     (size_t)p->d * sizeof(double) + 64;
    rc = parallel_for(bwd_row_task, &cx, n_rows * p->H_kv, scratch, n_threads);
    if (rc) goto done;
    rc = parallel_for(bwd_key_task, &cx, (int64_t)p->B * nblocks(p), 0, n_threads);
    if (rc) goto done;
  }
  {
    double total = 0.0;
    for (int64_t t = 0; t < n_rows * p->H_kv; ++t) total += cx.row_kl[t];
    *kl = kl_weight * total;
    if (kl_rows) memcpy(kl_rows, cx.row_kl, sizeof(double) * (size_t)(n_rows * p->H_kv));
  }
  rc = OR_OK;
done:
  free(cx.row_lse);
  free(cx.row_D);
  free(cx.row_lse_idx);
  free(cx.row_kl);
  free(cx.batch_start);
  return rc;
}
