/*
 * fa_oracle.c -- plain, slow CPU oracle for exact training attention (forward O, L and
 * backward dQ, dK, dV).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call, link or load this file;
 * only the tests, the smoke check and the benchmark's CPU-baseline leg use it. It shares no
 * code, header or constant with the CUDA path.
 *
 * What it computes (the plain definition, in f64 over inputs that hold exact bf16 values):
 * for batch b, query head h, query row i, with G = n_heads / n_kv_heads and kv head
 * kh = h / G (page "mlx-native tests/test_flash_attn_train.rs", `sdpa_reference_with_logsumexp`,
 * the `kv_h = h / heads_per_kv` head map):
 *
 *   visible(i, j) = !causal || j <= kl - ql + i            (bottom-right causal alignment)
 *   s_ij  = scale * <q_i, k_j> + mask_ij   if visible, else -inf
 *   L_i   = log sum_j exp(s_ij)            (-inf when no s_ij is finite)
 *   O_i   = sum_j exp(s_ij - L_i) v_j      (0 when L_i = -inf)
 *
 * Backward (same page, `sdpa_backward_reference_f32`, the FlashAttention-2 backward
 * equations), with dO the upstream gradient of O:
 *
 *   P_ij  = exp(s_ij - L_i)     (0 where s_ij = -inf or L_i = -inf)
 *   D_i   = <dO_i, O_i>         (O the oracle's own f64 output)
 *   dP_ij = <dO_i, v_j>,   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j  = scale * sum_{h in group(kh)} sum_i dS_ij q_i
 *   dV_j  =         sum_{h in group(kh)} sum_i P_ij dO_i
 *
 * Readings where the pages are silent or disagree:
 *   - causal alignment is bottom-right in BOTH passes (the backward oracle on the mlx-native
 *     page uses top-left `k_j > q_i`, which agrees only when ql == kl; the forward oracle on
 *     that page and the nuvec-core direct formula `visible = i + lk - lq + 1` are bottom-right);
 *   - kl - ql + i is signed: with causal and ql > kl the first ql - kl rows see no key and are
 *     fully masked (the mlx-native forward clamps with saturating_sub instead; parity of that
 *     corner is unpinned by the pages because the two disagree);
 *   - the mask is natural-log additive, shape [B, H, ql, kl], an entry -inf hides the key.
 *
 * Attention sinks (page "nuvec-core tests/fast.rs", `attention_kernels_match_the_fallback`,
 * where the fused attention takes an optional `sinks` array of shape [n_heads]): the page
 * shows only the shape, so the plainest reading is taken: sink_h is one extra natural-log
 * logit of every row of query head h that enters the softmax normaliser but carries no
 * value and is not scaled, i.e.
 *
 *   L_i = log( exp(sink_h) + sum_j exp(s_ij) ),   O_i = sum_j exp(s_ij - L_i) v_j
 *
 * so a row that sees no key has O = 0 and L = sink_h. The backward formulas above hold as
 * written (L carries the sink), and the sink's own gradient follows from the definition
 * (its score has no value, so its dP is 0 and dS_sink = P_sink (0 - D_i)):
 *
 *   dsink_h = - sum_b sum_i exp(sink_h - L_i) D_i
 *
 * Value head dimension (same page: its shapes list (D, Dv) pairs with Dv != D): q and k have
 * d columns, v, O, dO, dV have dv columns; every formula above is unchanged, the QK dot
 * products run over d and the dO.v, dO.O dot products over dv.
 *
 * Local (sliding-window) attention, the windowed form of the mlx-native SWA tests (sections 7
 * and 15, which build it as an additive mask): with window_left = wl >= 0 a key j is hidden
 * when j < q_abs - wl, with window_right = wr >= 0 when j > q_abs + wr; -1 leaves that side
 * unbounded. It composes with causal (which hides j > q_abs) and with the mask.
 *
 * A second forward mode (base2 = 1) takes the mlx-native forward oracle's own steps: the score
 * is multiplied by scale*log2(e), the mask by log2(e), the row max starts at the finite
 * sentinel -FLT_MAX/2, p = exp2(s - max), L = max*ln(2) + ln(sum p), O = sum (p / safe_sum) v
 * with safe_sum = 1 when the sum is 0. Both modes must agree to rounding on any input.
 *
 * Attention over a paged key/value cache (page "nuvec-core tests/fast.rs",
 * `paged_attention_equals_contiguous_attention` and its `paged` helper; page "tang
 * src/compute/cuda.rs", `kv_attention`, for single-query decode and the cached prefill with
 * `cache_start`): the keys of sequence b are its first len_b cache positions; logical key j
 * lives in physical page table[b][j / bs], slot j % bs, of caches shaped
 * [num_pages, Hk, bs, d]. The lq queries of a sequence are its last lq positions, so with the
 * causal mask query i sees key j iff j <= len_b - lq + i (the bottom-right alignment above,
 * per sequence; tang's cached prefill is the case len_b = cache_start + lq). Then the same
 * definition: s = scale <q, k_j>, L = log sum exp s, O = sum exp(s - L) v_j.
 *
 * Layouts (all contiguous, row-major): q, dQ [B, H, ql, d]; O, dO [B, H, ql, dv];
 * k, dK [B, Hk, kl, d]; v, dV [B, Hk, kl, dv]; L [B, H, ql]; mask [B, H, ql, kl] or NULL;
 * sinks [H] or NULL (set with fa_oracle_set_sinks).
 *
 * A mutation switch (fa_oracle_set_mutation) plants one known mistake at a time. It is off (0)
 * by default and exists only so that the tests can show that each planted mistake fails one
 * of the oracle's pins.
 */
#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int B, H, Hk, ql, kl, d, dv; /* d: q/k head dim; dv: v/O/dO head dim */
  double scale;
  int causal;
  int wl, wr; /* local window around q_abs = kl - ql + i: -1 = unbounded on that side */
  const float *q, *k, *v, *mask, *dO;
  const float *sinks; /* [H] natural-log sink logits, or NULL */
} prob_t;

/* Planted mistakes (tests only). 0 = none. */
enum {
  MUT_NONE = 0,
  MUT_NO_SCALE = 1,        /* score without the scale factor */
  MUT_TOP_LEFT = 2,        /* causal aligned top-left instead of bottom-right */
  MUT_GQA_MODULO = 3,      /* kv head = h % Hk instead of h / G */
  MUT_NO_NORMALISE = 4,    /* O not divided by the row sum */
  MUT_MASK_SIGN = 5,       /* mask subtracted instead of added */
  MUT_L_NO_MAX = 6,        /* L = log(sum exp(s - m)), max dropped */
  MUT_DS_NO_D = 7,         /* dS = P * dP (the -D term dropped) */
  MUT_DK_USES_K = 8,       /* dK accumulates dS * k_j instead of dS * q_i */
  MUT_DV_USES_DS = 9,      /* dV accumulates dS instead of P */
  MUT_CAUSAL_OFF_BY_ONE = 10, /* visible iff j < kl - ql + i */
  MUT_DQ_NO_SCALE = 11,    /* dQ without the scale factor */
  MUT_D_FROM_DO_ONLY = 12, /* D_i = sum dO (O dropped) */
  MUT_WINDOW_OFF_BY_ONE = 13, /* left window bound one key too narrow */
  MUT_SINK_SCALED = 14,    /* sink logit multiplied by the score scale */
  MUT_DSINK_SIGN = 15,     /* dsink without its minus sign */
  MUT_V_STRIDE_D = 16,     /* v rows addressed with the q/k head dim */
  MUT_TABLE_STRIDE = 17,   /* block-table row stride = the pages a sequence uses, not its capacity */
  MUT_DECODE_TOP_LEFT = 18, /* paged causal aligned to the first key (q_abs = i) */
};
static int g_mutation = 0;

void fa_oracle_set_mutation(int m) { g_mutation = m; }
int fa_oracle_get_mutation(void) { return g_mutation; }

static inline size_t q_index(const prob_t *p, int b, int h, int i) {
  return (((size_t)b * p->H + h) * p->ql + i) * (size_t)p->d;
}
static inline size_t kv_index(const prob_t *p, int b, int kh, int j) {
  return (((size_t)b * p->Hk + kh) * p->kl + j) * (size_t)p->d;
}
/* row j of v (dv columns), and row i of O / dO (dv columns) */
static inline size_t v_index(const prob_t *p, int b, int kh, int j) {
  const size_t w = (g_mutation == MUT_V_STRIDE_D) ? (size_t)p->d : (size_t)p->dv;
  return (((size_t)b * p->Hk + kh) * p->kl + j) * w;
}
static inline size_t o_index(const prob_t *p, int b, int h, int i) {
  return (((size_t)b * p->H + h) * p->ql + i) * (size_t)p->dv;
}
/* the sink logit of head h in natural-log units, or -inf without sinks */
static inline double sink_logit(const prob_t *p, int h) {
  if (!p->sinks) return -INFINITY;
  double s = (double)p->sinks[h];
  if (g_mutation == MUT_SINK_SCALED) s *= p->scale;
  return s;
}
static inline int kv_head(const prob_t *p, int h) {
  if (g_mutation == MUT_GQA_MODULO) return h % p->Hk;
  return h / (p->H / p->Hk);
}
static inline int visible(const prob_t *p, int i, int j) {
  long off = (long)p->kl - (long)p->ql;
  if (g_mutation == MUT_TOP_LEFT) off = 0;
  const long qa = off + (long)i; /* query position aligned to the end of the keys */
  if (p->wl >= 0 && (long)j < qa - p->wl + (g_mutation == MUT_WINDOW_OFF_BY_ONE ? 1 : 0)) return 0;
  if (p->wr >= 0 && (long)j > qa + p->wr) return 0;
  if (!p->causal) return 1;
  if (g_mutation == MUT_CAUSAL_OFF_BY_ONE) return (long)j < qa;
  return (long)j <= qa;
}

/* Scores of row (b, h, i) into s[kl]: natural-log domain, -inf where hidden. */
static void row_scores(const prob_t *p, int b, int h, int i, double *s) {
  const int kh = kv_head(p, h);
  const float *qi = p->q + q_index(p, b, h, i);
  const double sc = (g_mutation == MUT_NO_SCALE) ? 1.0 : p->scale;
  for (int j = 0; j < p->kl; ++j) {
    if (!visible(p, i, j)) { s[j] = -INFINITY; continue; }
    const float *kj = p->k + kv_index(p, b, kh, j);
    double dot = 0.0;
    for (int c = 0; c < p->d; ++c) dot += (double)qi[c] * (double)kj[c];
    double v = sc * dot;
    if (p->mask) {
      double m = (double)p->mask[(((size_t)b * p->H + h) * p->ql + i) * (size_t)p->kl + j];
      if (g_mutation == MUT_MASK_SIGN) m = -m;
      v += m; /* an entry of -inf gives -inf */
    }
    s[j] = v;
  }
}

/* Forward of one row, natural-log mode: L and O[dv] from the scores (and the head's sink). */
static double row_forward_nat(const prob_t *p, int b, int h, int i, const double *s, double *o) {
  (void)i;
  const int kh = kv_head(p, h);
  const double sink = sink_logit(p, h);
  double m = sink;
  for (int j = 0; j < p->kl; ++j) if (s[j] > m) m = s[j];
  for (int c = 0; c < p->dv; ++c) o[c] = 0.0;
  if (m == -INFINITY) return -INFINITY; /* fully masked row, no sink: O = 0, L = -inf */
  double z = exp(sink - m);             /* the sink's share of the normaliser (0 without) */
  for (int j = 0; j < p->kl; ++j) z += exp(s[j] - m);
  for (int j = 0; j < p->kl; ++j) {
    if (s[j] == -INFINITY) continue;
    double w = exp(s[j] - m);
    if (g_mutation != MUT_NO_NORMALISE) w /= z;
    const float *vj = p->v + v_index(p, b, kh, j);
    for (int c = 0; c < p->dv; ++c) o[c] += w * (double)vj[c];
  }
  if (g_mutation == MUT_L_NO_MAX) return log(z);
  return m + log(z);
}

/* Forward of one row in the mlx-native base-2 form (steps of `sdpa_reference_with_logsumexp`,
 * carried out in f64). Recomputes its own scores so that it owns every step. */
static double row_forward_base2(const prob_t *p, int b, int h, int i, double *o) {
  const double LOG2E = 1.4426950408889634074;
  const double LN2 = 0.69314718055994530942;
  const int kh = kv_head(p, h);
  const float *qi = p->q + q_index(p, b, h, i);
  const double sc = ((g_mutation == MUT_NO_SCALE) ? 1.0 : p->scale) * LOG2E; /* q pre-scale */
  double *s2 = (double *)malloc(sizeof(double) * (size_t)p->kl);
  for (int j = 0; j < p->kl; ++j) {
    const float *kj = p->k + kv_index(p, b, kh, j);
    double dot = 0.0;
    for (int c = 0; c < p->d; ++c) dot += (double)qi[c] * (double)kj[c];
    s2[j] = dot * sc;
    if (p->mask) {
      double m = (double)p->mask[(((size_t)b * p->H + h) * p->ql + i) * (size_t)p->kl + j];
      if (g_mutation == MUT_MASK_SIGN) m = -m;
      s2[j] += LOG2E * m;
    }
    if (!visible(p, i, j)) s2[j] = -INFINITY;
  }
  double mx = -(double)FLT_MAX / 2.0; /* finite sentinel */
  const double sink2 = sink_logit(p, h) * LOG2E; /* -inf without sinks */
  if (sink2 > mx) mx = sink2;
  for (int j = 0; j < p->kl; ++j) if (s2[j] > mx) mx = s2[j];
  double sum = exp2(sink2 - mx);
  for (int j = 0; j < p->kl; ++j) { s2[j] = exp2(s2[j] - mx); sum += s2[j]; }
  double lse = (g_mutation == MUT_L_NO_MAX) ? log(sum) : mx * LN2 + log(sum);
  double safe = (sum == 0.0) ? 1.0 : sum;
  if (g_mutation == MUT_NO_NORMALISE) safe = 1.0;
  for (int c = 0; c < p->dv; ++c) o[c] = 0.0;
  for (int j = 0; j < p->kl; ++j) {
    const float *vj = p->v + v_index(p, b, kh, j);
    double w = s2[j] / safe;
    for (int c = 0; c < p->dv; ++c) o[c] += w * (double)vj[c];
  }
  free(s2);
  return lse;
}

/* ------------------------------------------------------------------ tiny thread pool */
typedef struct {
  void (*fn)(void *ctx, long task, int worker);
  void *ctx;
  long ntasks;
  long next;
  pthread_mutex_t mu;
  int worker_seq;
} pool_t;

static void *pool_main(void *arg) {
  pool_t *pl = (pool_t *)arg;
  pthread_mutex_lock(&pl->mu);
  int me = pl->worker_seq++;
  pthread_mutex_unlock(&pl->mu);
  for (;;) {
    pthread_mutex_lock(&pl->mu);
    long t = pl->next++;
    pthread_mutex_unlock(&pl->mu);
    if (t >= pl->ntasks) break;
    pl->fn(pl->ctx, t, me);
  }
  return NULL;
}

static void parallel_for(long ntasks, int nthreads, void (*fn)(void *, long, int), void *ctx) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > ntasks) nthreads = (int)(ntasks > 0 ? ntasks : 1);
  pool_t pl;
  pl.fn = fn; pl.ctx = ctx; pl.ntasks = ntasks; pl.next = 0; pl.worker_seq = 0;
  pthread_mutex_init(&pl.mu, NULL);
  if (nthreads == 1) {
    pool_main(&pl);
  } else {
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, pool_main, &pl);
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
  }
  pthread_mutex_destroy(&pl.mu);
}

static int g_wl = -1, g_wr = -1; /* window of the next calls (fa_oracle_set_window) */
static const float *g_sinks = NULL; /* sinks of the next calls (fa_oracle_set_sinks) */

void fa_oracle_set_window(int wl, int wr) { g_wl = wl; g_wr = wr; }
/* [H] sink logits read by the following calls (the caller keeps the array alive), or NULL. */
void fa_oracle_set_sinks(const float *sinks) { g_sinks = sinks; }

static prob_t make_prob(const float *q, const float *k, const float *v, const float *mask,
                        const float *dO, int B, int H, int Hk, int ql, int kl, int d, int dv,
                        double scale, int causal) {
  prob_t p;
  p.B = B; p.H = H; p.Hk = Hk; p.ql = ql; p.kl = kl; p.d = d; p.dv = dv;
  p.scale = scale; p.causal = causal;
  p.wl = g_wl; p.wr = g_wr;
  p.q = q; p.k = k; p.v = v; p.mask = mask; p.dO = dO;
  p.sinks = g_sinks;
  return p;
}

static int bad_sizes(int B, int H, int Hk, int ql, int kl, int d, int dv) {
  return B <= 0 || H <= 0 || Hk <= 0 || ql <= 0 || kl <= 0 || d <= 0 || dv <= 0 || H % Hk;
}

/* ------------------------------------------------------------------ forward, by rows */
typedef struct {
  const prob_t *p;
  const int64_t *rows; /* flat (b*H + h)*ql + i */
  double *o, *lse;
  int base2;
} fwd_ctx;

static void fwd_task(void *vctx, long t, int worker) {
  (void)worker;
  fwd_ctx *c = (fwd_ctx *)vctx;
  const prob_t *p = c->p;
  int64_t r = c->rows ? c->rows[t] : (int64_t)t;
  int i = (int)(r % p->ql);
  int h = (int)((r / p->ql) % p->H);
  int b = (int)(r / ((int64_t)p->ql * p->H));
  double *o = c->o + (size_t)t * p->dv;
  if (c->base2) {
    c->lse[t] = row_forward_base2(p, b, h, i, o);
  } else {
    double *s = (double *)malloc(sizeof(double) * (size_t)p->kl);
    row_scores(p, b, h, i, s);
    c->lse[t] = row_forward_nat(p, b, h, i, s, o);
    free(s);
  }
}

/* O and L of the listed rows (rows == NULL: all B*H*ql rows in order). Output o[nrows*dv],
 * lse[nrows]. Returns 0, or -1 on bad sizes. */
int fa_oracle_fwd_rows(const float *q, const float *k, const float *v, const float *mask,
                       int B, int H, int Hk, int ql, int kl, int d, int dv, double scale,
                       int causal, const int64_t *rows, long nrows, int base2, double *o,
                       double *lse, int nthreads) {
  if (bad_sizes(B, H, Hk, ql, kl, d, dv)) return -1;
  prob_t p = make_prob(q, k, v, mask, NULL, B, H, Hk, ql, kl, d, dv, scale, causal);
  fwd_ctx c = {&p, rows, o, lse, base2};
  parallel_for(nrows, nthreads, fwd_task, &c);
  return 0;
}

/* ------------------------------------------------------------------ backward pieces */

/* Everything the backward needs about one query row: P row (kl), dS row (kl), O, L and D. */
typedef struct {
  double *s, *o, *pr, *ds; /* scores, O row (dv), P row, dS row */
  double L, D;
} rowbuf;

static rowbuf rowbuf_new(const prob_t *p) {
  rowbuf r;
  r.s = (double *)malloc(sizeof(double) * (size_t)p->kl);
  r.pr = (double *)malloc(sizeof(double) * (size_t)p->kl);
  r.ds = (double *)malloc(sizeof(double) * (size_t)p->kl);
  r.o = (double *)malloc(sizeof(double) * (size_t)p->dv);
  r.L = 0.0;
  r.D = 0.0;
  return r;
}
static void rowbuf_free(rowbuf *r) { free(r->s); free(r->pr); free(r->ds); free(r->o); }

/* Fills r.pr with the P row, r.ds with the dS row, r.L and r.D of query row (b, h, i). */
static void row_backward_prep(const prob_t *p, int b, int h, int i, rowbuf *r) {
  const int kh = kv_head(p, h);
  row_scores(p, b, h, i, r->s);
  double L = row_forward_nat(p, b, h, i, r->s, r->o);
  const float *doi = p->dO + o_index(p, b, h, i);
  double D = 0.0;
  for (int c = 0; c < p->dv; ++c)
    D += (double)doi[c] * ((g_mutation == MUT_D_FROM_DO_ONLY) ? 1.0 : r->o[c]);
  for (int j = 0; j < p->kl; ++j) {
    double P = (r->s[j] == -INFINITY || L == -INFINITY) ? 0.0 : exp(r->s[j] - L);
    const float *vj = p->v + v_index(p, b, kh, j);
    double dP = 0.0;
    for (int c = 0; c < p->dv; ++c) dP += (double)doi[c] * (double)vj[c];
    r->pr[j] = P;
    r->ds[j] = (g_mutation == MUT_DS_NO_D) ? P * dP : P * (dP - D);
  }
  r->L = L;
  r->D = D;
}

typedef struct {
  const prob_t *p;
  const int64_t *rows;
  double *dq;
} dq_ctx;

static void dq_task(void *vctx, long t, int worker) {
  (void)worker;
  dq_ctx *c = (dq_ctx *)vctx;
  const prob_t *p = c->p;
  int64_t r = c->rows ? c->rows[t] : (int64_t)t;
  int i = (int)(r % p->ql);
  int h = (int)((r / p->ql) % p->H);
  int b = (int)(r / ((int64_t)p->ql * p->H));
  const int kh = kv_head(p, h);
  rowbuf rb = rowbuf_new(p);
  row_backward_prep(p, b, h, i, &rb);
  double *dq = c->dq + (size_t)t * p->d;
  const double sc = (g_mutation == MUT_DQ_NO_SCALE) ? 1.0 : p->scale;
  for (int cc = 0; cc < p->d; ++cc) dq[cc] = 0.0;
  for (int j = 0; j < p->kl; ++j) {
    double ds = rb.ds[j];
    if (ds == 0.0) continue;
    const float *kj = p->k + kv_index(p, b, kh, j);
    for (int cc = 0; cc < p->d; ++cc) dq[cc] += sc * ds * (double)kj[cc];
  }
  rowbuf_free(&rb);
}

/* dQ of the listed query rows (rows == NULL: all). Output dq[nrows*d]. */
int fa_oracle_bwd_q_rows(const float *q, const float *k, const float *v, const float *mask,
                         const float *dO, int B, int H, int Hk, int ql, int kl, int d, int dv,
                         double scale, int causal, const int64_t *rows, long nrows, double *dq,
                         int nthreads) {
  if (bad_sizes(B, H, Hk, ql, kl, d, dv)) return -1;
  prob_t p = make_prob(q, k, v, mask, dO, B, H, Hk, ql, kl, d, dv, scale, causal);
  dq_ctx c = {&p, rows, dq};
  parallel_for(nrows, nthreads, dq_task, &c);
  return 0;
}

/* dK, dV rows of one (b, kh): tasks run over (h in group, i), each worker owning a private
 * accumulator that is summed at the end (the sum order over workers is fixed). */
typedef struct {
  const prob_t *p;
  int b, kh;
  const int32_t *js;
  int nj;
  double *acc; /* [nworkers][nj * (d + dv)]: dK rows, then dV rows */
  int nworkers;
} dkv_ctx;

static void dkv_task(void *vctx, long t, int worker) {
  dkv_ctx *c = (dkv_ctx *)vctx;
  const prob_t *p = c->p;
  const int G = p->H / p->Hk;
  int gh = (int)(t / p->ql), i = (int)(t % p->ql);
  int h = c->kh * G + gh;
  if (g_mutation == MUT_GQA_MODULO) h = c->kh + gh * p->Hk; /* heads with h % Hk == kh */
  rowbuf rb = rowbuf_new(p);
  row_backward_prep(p, c->b, h, i, &rb);
  const float *qi = p->q + q_index(p, c->b, h, i);
  const float *doi = p->dO + o_index(p, c->b, h, i);
  double *dk = c->acc + (size_t)worker * c->nj * (p->d + p->dv);
  double *dv = dk + (size_t)c->nj * p->d;
  for (int n = 0; n < c->nj; ++n) {
    int j = c->js[n];
    double P = rb.pr[j], ds = rb.ds[j];
    if (P == 0.0 && ds == 0.0) continue;
    const float *kj = p->k + kv_index(p, c->b, c->kh, j);
    const float *src = (g_mutation == MUT_DK_USES_K) ? kj : qi;
    const double pv = (g_mutation == MUT_DV_USES_DS) ? ds : P;
    for (int cc = 0; cc < p->d; ++cc) dk[(size_t)n * p->d + cc] += p->scale * ds * (double)src[cc];
    for (int cc = 0; cc < p->dv; ++cc) dv[(size_t)n * p->dv + cc] += pv * (double)doi[cc];
  }
  rowbuf_free(&rb);
}

/* dK and dV rows js[0..nj) of kv head kh in batch b. Outputs dk[nj*d], dv[nj*dv]. */
int fa_oracle_bwd_kv_rows(const float *q, const float *k, const float *v, const float *mask,
                          const float *dO, int B, int H, int Hk, int ql, int kl, int d, int dv,
                          double scale, int causal, int b, int kh, const int32_t *js, int nj,
                          double *dk, double *dvo, int nthreads) {
  if (bad_sizes(B, H, Hk, ql, kl, d, dv)) return -1;
  if (b < 0 || b >= B || kh < 0 || kh >= Hk) return -1;
  for (int n = 0; n < nj; ++n) if (js[n] < 0 || js[n] >= kl) return -1;
  prob_t p = make_prob(q, k, v, mask, dO, B, H, Hk, ql, kl, d, dv, scale, causal);
  const int G = H / Hk;
  long ntasks = (long)G * ql;
  int nw = nthreads < 1 ? 1 : nthreads;
  if (nw > ntasks) nw = (int)ntasks;
  const size_t per = (size_t)nj * (d + dv);
  dkv_ctx c;
  c.p = &p; c.b = b; c.kh = kh; c.js = js; c.nj = nj; c.nworkers = nw;
  c.acc = (double *)calloc((size_t)nw * per, sizeof(double));
  if (!c.acc) return -2;
  parallel_for(ntasks, nw, dkv_task, &c);
  for (size_t e = 0; e < (size_t)nj * d; ++e) dk[e] = 0.0;
  for (size_t e = 0; e < (size_t)nj * dv; ++e) dvo[e] = 0.0;
  for (int w = 0; w < nw; ++w) {
    const double *a = c.acc + (size_t)w * per;
    for (size_t e = 0; e < (size_t)nj * d; ++e) dk[e] += a[e];
    for (size_t e = 0; e < (size_t)nj * dv; ++e) dvo[e] += a[(size_t)nj * d + e];
  }
  free(c.acc);
  return 0;
}

/* Full backward: dq [B,H,ql,d], dk [B,Hk,kl,d] and dv [B,Hk,kl,dv]. */
int fa_oracle_bwd(const float *q, const float *k, const float *v, const float *mask,
                  const float *dO, int B, int H, int Hk, int ql, int kl, int d, int dv,
                  double scale, int causal, double *dq, double *dk, double *dvo, int nthreads) {
  int rc = fa_oracle_bwd_q_rows(q, k, v, mask, dO, B, H, Hk, ql, kl, d, dv, scale, causal, NULL,
                                (long)B * H * ql, dq, nthreads);
  if (rc) return rc;
  int32_t *js = (int32_t *)malloc(sizeof(int32_t) * (size_t)kl);
  for (int j = 0; j < kl; ++j) js[j] = j;
  for (int b = 0; b < B && !rc; ++b)
    for (int kh = 0; kh < Hk && !rc; ++kh) {
      const size_t row0 = ((size_t)b * Hk + kh) * kl;
      rc = fa_oracle_bwd_kv_rows(q, k, v, mask, dO, B, H, Hk, ql, kl, d, dv, scale, causal, b,
                                 kh, js, kl, dk + row0 * d, dvo + row0 * dv, nthreads);
    }
  free(js);
  return rc;
}

/* ------------------------------------------------------------------ sink gradient */
typedef struct {
  const prob_t *p;
  double *term; /* [B*H*ql]: -exp(sink_h - L_i) D_i of every row */
} dsink_ctx;

static void dsink_task(void *vctx, long t, int worker) {
  (void)worker;
  dsink_ctx *c = (dsink_ctx *)vctx;
  const prob_t *p = c->p;
  int i = (int)(t % p->ql);
  int h = (int)((t / p->ql) % p->H);
  int b = (int)(t / ((int64_t)p->ql * p->H));
  rowbuf rb = rowbuf_new(p);
  row_backward_prep(p, b, h, i, &rb);
  const double sink = sink_logit(p, h);
  const double psink = (rb.L == -INFINITY) ? 0.0 : exp(sink - rb.L); /* the sink's P */
  c->term[t] = (g_mutation == MUT_DSINK_SIGN) ? psink * rb.D : -psink * rb.D;
  rowbuf_free(&rb);
}

/* Gradient of sum(O * dO) with respect to the sink logits set by fa_oracle_set_sinks:
 * dsinks[h] = -sum_b sum_i exp(sink_h - L_bhi) D_bhi. Returns -1 on bad sizes or when no
 * sinks are set. */
int fa_oracle_dsinks(const float *q, const float *k, const float *v, const float *mask,
                     const float *dO, int B, int H, int Hk, int ql, int kl, int d, int dv,
                     double scale, int causal, double *dsinks, int nthreads) {
  if (bad_sizes(B, H, Hk, ql, kl, d, dv) || !g_sinks) return -1;
  prob_t p = make_prob(q, k, v, mask, dO, B, H, Hk, ql, kl, d, dv, scale, causal);
  const long n = (long)B * H * ql;
  dsink_ctx c = {&p, (double *)malloc(sizeof(double) * (size_t)n)};
  if (!c.term) return -2;
  parallel_for(n, nthreads, dsink_task, &c);
  for (int h = 0; h < H; ++h) dsinks[h] = 0.0;
  for (long t = 0; t < n; ++t) dsinks[(t / ql) % H] += c.term[t]; /* fixed order */
  free(c.term);
  return 0;
}

/* ------------------------------------------------------------------ paged KV cache */
typedef struct {
  const float *q, *kc, *vc;
  const int32_t *table, *lens;
  int B, H, Hk, lq, d, bs, max_pages, num_pages, causal;
  double scale;
  double *o, *lse;
} paged_ctx;

/* physical (page, slot) of logical key j of sequence b */
static void paged_locate(const paged_ctx *c, int b, int j, int *page, int *slot) {
  long stride = c->max_pages;
  if (g_mutation == MUT_TABLE_STRIDE) stride = (c->lens[b] + c->bs - 1) / c->bs;
  *page = c->table[(long)b * stride + j / c->bs];
  *slot = j % c->bs;
}

static void paged_task(void *vctx, long t, int worker) {
  (void)worker;
  const paged_ctx *c = (const paged_ctx *)vctx;
  const int i = (int)(t % c->lq);
  const int h = (int)((t / c->lq) % c->H);
  const int b = (int)(t / ((long)c->lq * c->H));
  const int kh = h / (c->H / c->Hk);
  const int len = c->lens[b];
  const float *qi = c->q + (size_t)t * c->d;
  double *o = c->o + (size_t)t * c->d;
  const long qa = (g_mutation == MUT_DECODE_TOP_LEFT) ? (long)i : (long)len - c->lq + i;
  double *s = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1));
  double m = -INFINITY;
  for (int j = 0; j < len; ++j) {
    s[j] = -INFINITY;
    if (c->causal && (long)j > qa) continue;
    int page, slot;
    paged_locate(c, b, j, &page, &slot);
    const float *kj = c->kc + ((((size_t)page * c->Hk + kh) * c->bs + slot) * (size_t)c->d);
    double dot = 0.0;
    for (int e = 0; e < c->d; ++e) dot += (double)qi[e] * (double)kj[e];
    s[j] = c->scale * dot;
    if (s[j] > m) m = s[j];
  }
  for (int e = 0; e < c->d; ++e) o[e] = 0.0;
  if (m == -INFINITY) {
    c->lse[t] = -INFINITY; /* a query that sees no key: O = 0, L = -inf */
    free(s);
    return;
  }
  double z = 0.0;
  for (int j = 0; j < len; ++j) z += exp(s[j] - m);
  const double L = m + log(z);
  for (int j = 0; j < len; ++j) {
    if (s[j] == -INFINITY) continue;
    int page, slot;
    paged_locate(c, b, j, &page, &slot);
    const float *vj = c->vc + ((((size_t)page * c->Hk + kh) * c->bs + slot) * (size_t)c->d);
    const double w = exp(s[j] - L);
    for (int e = 0; e < c->d; ++e) o[e] += w * (double)vj[e];
  }
  c->lse[t] = L;
  free(s);
}

/* O [B, H, lq, d] and L [B, H, lq] of queries q [B, H, lq, d] over paged caches
 * kc, vc [num_pages, Hk, bs, d] with block table [B, max_pages] and lengths [B]. Returns -1 on
 * bad sizes, a length outside [0, max_pages * bs] or a used table entry outside
 * [0, num_pages). */
int fa_oracle_paged_fwd(const float *q, const float *kc, const float *vc, const int32_t *table,
                        const int32_t *lens, int B, int H, int Hk, int lq, int d, int bs,
                        int max_pages, int num_pages, double scale, int causal, double *o,
                        double *lse, int nthreads) {
  if (B <= 0 || H <= 0 || Hk <= 0 || lq <= 0 || d <= 0 || bs <= 0 || max_pages <= 0 ||
      num_pages <= 0 || H % Hk)
    return -1;
  for (int b = 0; b < B; ++b) {
    if (lens[b] < 0 || (long)lens[b] > (long)max_pages * bs) return -1;
    for (int p = 0; p < (lens[b] + bs - 1) / bs; ++p) {
      const int32_t e = table[(long)b * max_pages + p];
      if (e < 0 || e >= num_pages) return -1;
    }
  }
  paged_ctx c = {q, kc, vc, table, lens, B, H, Hk, lq, d, bs, max_pages, num_pages,
                 causal ? 1 : 0, scale, o, lse};
  parallel_for((long)B * H * lq, nthreads, paged_task, &c);
  return 0;
}
