/*
 * dsa_oracle.c -- plain, slow, CPU oracle for the gated DSA attention step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; the two meet only in the seeded input buffers.
 *
 * Every function evaluates the plain definition in double precision from the
 * same BF16 inputs the CUDA path reads (decoded exactly), one query row at a
 * time, with no blocking, fusion or reordering beyond what the definition
 * states.  Rows are spread over POSIX threads; each row is computed by one
 * thread in a fixed order, so results do not depend on the thread count.
 *
 * Sources (page title, section):
 *   [K31]  "Kimi-K3.1-Pro", NeMo AutoModel model coverage:
 *          - Implementation Limits, bullet 1: a fused indexer produces top-k
 *            coordinates; sparse MLA attends directly to the selected latent KV.
 *          - Implementation Limits, bullet 2: BF16 indexer projections with FP32
 *            score accumulation; the indexer scans all causal keys; sparse MLA
 *            neither expands per-head K/V nor attends to unselected keys.
 *          - Implementation Limits, bullet 4: a sequence of at most 2,048 valid
 *            tokens keeps every causal key.
 *          - Implementation Limits, closing paragraph: the output gate is kept.
 *   [ARCH] "Kimi K3.1 Pro" (archdiff, attn-gate): summary line (24 gated DSA
 *          layers, top-2,048, no positional encoding); blueprint list items
 *          "LayerNorm on the indexer key", "Partial RoPE / NoPE", and
 *          "Output gate + sink: sigma(x W_g) (.) o".
 *   [CFG]  "nemo_automodel.components.models.kimi_k3" (v0.4 API),
 *          KimiK3TextConfig: kv_lora_rank 512, qk_nope_head_dim 128,
 *          qk_rope_head_dim 64, v_head_dim 128, num_attention_heads 96,
 *          mla_use_nope True, mla_use_output_gate True.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - indexer score I[t,s] = sum_j w[t,j] * max(0, q[t,j,:] . k[s,:]), one shared
 *     key per token, no extra scale (the pages do not give the indexer's form);
 *   - causal means s <= t, self included, and self is not forced into the set;
 *   - ordering for top-k: larger score first, then smaller key index;
 *   - value vector = the first 512 latent dims; the 64 k_pe dims only enter
 *     the logits; no rotation anywhere (NoPE);
 *   - the gate acts element-wise on the per-head value after W_UV, i.e. on the
 *     H*dv = 96*128 wide attention output, with W_g shaped [H*dv, hid].
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_OK 0
#define OR_BAD_ARG 1
#define OR_BAD_INDEX 2
#define OR_NOMEM 3

/* ------------------------------------------------------------------------- */
/* BF16 decode (exact) and threading                                          */
/* ------------------------------------------------------------------------- */

static double bf(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static int g_threads = 0;

int oracle_set_threads(int n) {
  g_threads = n;
  return OR_OK;
}

int oracle_get_threads(void) {
  if (g_threads > 0) return g_threads;
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

typedef void (*row_fn)(void* ctx, int64_t r);

typedef struct {
  row_fn fn;
  void* ctx;
  int64_t n;
  int64_t next;
  pthread_mutex_t mu;
} pool_t;

static void* pool_worker(void* arg) {
  pool_t* p = (pool_t*)arg;
  for (;;) {
    pthread_mutex_lock(&p->mu);
    int64_t r = p->next++;
    pthread_mutex_unlock(&p->mu);
    if (r >= p->n) break;
    p->fn(p->ctx, r);
  }
  return NULL;
}

static void parallel_rows(int64_t n, row_fn fn, void* ctx) {
  int nt = oracle_get_threads();
  if (nt > n) nt = (int)(n > 0 ? n : 1);
  pool_t p;
  p.fn = fn;
  p.ctx = ctx;
  p.n = n;
  p.next = 0;
  pthread_mutex_init(&p.mu, NULL);
  if (nt <= 1) {
    pool_worker(&p);
  } else {
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
    int started = 0;
    for (int i = 0; i < nt; ++i)
      if (pthread_create(&th[i], NULL, pool_worker, &p) == 0) ++started;
    if (started == 0) pool_worker(&p);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
  }
  pthread_mutex_destroy(&p.mu);
}

/* ------------------------------------------------------------------------- */
/* Indexer scores  [K31 Impl. Limits b2; ARCH summary; reading above]         */
/* ------------------------------------------------------------------------- */

typedef struct {
  const uint16_t *q, *w, *k;
  const int32_t *q_start, *kv_len;
  int Tq, S_max, H_I, D_I;
  const int64_t* rows;
  double* out;
  int err;
} idx_ctx;

static void indexer_row(void* vctx, int64_t r) {
  idx_ctx* c = (idx_ctx*)vctx;
  int64_t flat = c->rows[r];
  int b = (int)(flat / c->Tq), i = (int)(flat % c->Tq);
  int64_t t = (int64_t)c->q_start[b] + i; /* absolute query position */
  double* o = c->out + r * (int64_t)c->S_max;
  for (int64_t s = 0; s < c->S_max; ++s) o[s] = NAN;
  if (t >= c->kv_len[b] || t >= c->S_max) { c->err = OR_BAD_ARG; return; }
  const uint16_t* q = c->q + flat * (int64_t)c->H_I * c->D_I;
  const uint16_t* w = c->w + flat * (int64_t)c->H_I;
  const uint16_t* kb = c->k + (int64_t)b * c->S_max * c->D_I;
  /* every causal key s <= t is scored */
  for (int64_t s = 0; s <= t; ++s) {
    const uint16_t* k = kb + s * c->D_I;
    double score = 0.0;
    for (int j = 0; j < c->H_I; ++j) {
      double dot = 0.0;
      for (int d = 0; d < c->D_I; ++d) dot += bf(q[j * c->D_I + d]) * bf(k[d]);
      double relu = dot > 0.0 ? dot : 0.0;
      score += bf(w[j]) * relu;
    }
    o[s] = score;
  }
}

/* q_idx [B,Tq,H_I,D_I], w [B,Tq,H_I], k_idx [B,S_max,D_I] (BF16 bits);
 * out [n_rows, S_max]: score of key s for s <= t, NaN beyond. */
int oracle_indexer_scores(const uint16_t* q_idx, const uint16_t* w, const uint16_t* k_idx,
                          const int32_t* q_start, const int32_t* kv_len, int B, int Tq,
                          int S_max, int H_I, int D_I, int64_t n_rows, const int64_t* rows,
                          double* out) {
  if (!q_idx || !w || !k_idx || !q_start || !kv_len || !rows || !out) return OR_BAD_ARG;
  if (B <= 0 || Tq <= 0 || S_max <= 0 || H_I <= 0 || D_I <= 0 || n_rows < 0) return OR_BAD_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= (int64_t)B * Tq) return OR_BAD_ARG;
  idx_ctx c = {q_idx, w, k_idx, q_start, kv_len, Tq, S_max, H_I, D_I, rows, out, OR_OK};
  parallel_rows(n_rows, indexer_row, &c);
  return c.err;
}

/* ------------------------------------------------------------------------- */
/* Top-k selection  [K31 Impl. Limits b1 (coordinates), b4 (<= k keeps all)]  */
/* ------------------------------------------------------------------------- */

typedef struct {
  double score;
  int32_t s;
} cand_t;

static int cand_cmp(const void* a, const void* b) {
  const cand_t* x = (const cand_t*)a;
  const cand_t* y = (const cand_t*)b;
  if (x->score > y->score) return -1; /* larger score first */
  if (x->score < y->score) return 1;
  return (x->s < y->s) ? -1 : (x->s > y->s); /* then smaller index */
}

typedef struct {
  const double* scores;
  const int32_t* n_valid;
  int S_max, topk;
  int32_t* out_idx;
  double* kth;
  int err;
} topk_ctx;

static void topk_row(void* vctx, int64_t r) {
  topk_ctx* c = (topk_ctx*)vctx;
  int n = c->n_valid[r];
  int32_t* o = c->out_idx + r * (int64_t)c->topk;
  for (int j = 0; j < c->topk; ++j) o[j] = -1;
  if (n <= c->topk) {
    /* a query with at most k causal keys keeps every one of them */
    for (int s = 0; s < n; ++s) o[s] = s;
    c->kth[r] = -INFINITY;
    return;
  }
  cand_t* v = (cand_t*)malloc(sizeof(cand_t) * (size_t)n);
  if (!v) { c->err = OR_NOMEM; return; }
  const double* sc = c->scores + r * (int64_t)c->S_max;
  for (int s = 0; s < n; ++s) { v[s].score = sc[s]; v[s].s = s; }
  qsort(v, (size_t)n, sizeof(cand_t), cand_cmp);
  for (int j = 0; j < c->topk; ++j) o[j] = v[j].s;
  c->kth[r] = v[c->topk - 1].score;
  free(v);
}

/* scores [n_rows, S_max] (first n_valid[r] entries used); out_idx [n_rows, topk]
 * sorted by (score desc, index asc), -1 padded; kth[r] = k-th largest score, or
 * -inf when every key is kept. */
int oracle_topk(const double* scores, const int32_t* n_valid, int64_t n_rows, int S_max,
                int topk, int32_t* out_idx, double* kth) {
  if (!scores || !n_valid || !out_idx || !kth || topk <= 0 || S_max <= 0) return OR_BAD_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (n_valid[r] < 0 || n_valid[r] > S_max) return OR_BAD_ARG;
  topk_ctx c = {scores, n_valid, S_max, topk, out_idx, kth, OR_OK};
  parallel_rows(n_rows, topk_row, &c);
  return c.err;
}

/* ------------------------------------------------------------------------- */
/* Sparse MLA in latent space  [K31 Impl. Limits b1-b2; ARCH NoPE; CFG dims]  */
/* ------------------------------------------------------------------------- */

#define RLAT 576
#define VLAT 512

typedef struct {
  const uint16_t *q, *kv;
  const int32_t *idx, *q_start, *kv_len;
  int Tq, S_max, H, topk;
  double scale;
  const int64_t* rows;
  double *o, *lse;
  const double* sink; /* [H] learnable sink logits (natural log), or NULL */
  int err;
} mla_ctx;

static void mla_row(void* vctx, int64_t r) {
  mla_ctx* c = (mla_ctx*)vctx;
  int64_t flat = c->rows[r];
  int b = (int)(flat / c->Tq), i = (int)(flat % c->Tq);
  int64_t t = (int64_t)c->q_start[b] + i;
  const uint16_t* kvb = c->kv + (int64_t)b * c->S_max * RLAT;
  double* o = c->o + r * (int64_t)c->H * VLAT;
  double* lse = c->lse + r * (int64_t)c->H;
  if (t >= c->kv_len[b] || t >= c->S_max) { c->err = OR_BAD_ARG; return; }

  /* the set of attended keys: the given indices, skipping -1 */
  int n = 0;
  const int32_t* ix = c->idx + flat * (int64_t)c->topk;
  int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (size_t)c->topk);
  if (!sel) { c->err = OR_NOMEM; return; }
  for (int j = 0; j < c->topk; ++j) {
    int32_t s = ix[j];
    if (s < 0) continue;
    if (s > t || s >= c->kv_len[b]) { c->err = OR_BAD_INDEX; continue; }
    sel[n++] = s;
  }
  double* z = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  if (!z) { free(sel); c->err = OR_NOMEM; return; }
  for (int h = 0; h < c->H; ++h) {
    const uint16_t* q = c->q + (flat * c->H + h) * (int64_t)RLAT;
    double* oh = o + (int64_t)h * VLAT;
    for (int d = 0; d < VLAT; ++d) oh[d] = 0.0;
    /* no attended key: all weight on the sink (if any), whose value is zero */
    if (n == 0) { lse[h] = c->sink ? c->sink[h] : -INFINITY; continue; }
    /* logits over the full 576-wide row: 512 c_kv dims + 64 unrotated k_pe dims */
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
      const uint16_t* row = kvb + (int64_t)sel[j] * RLAT;
      double dot = 0.0;
      for (int d = 0; d < RLAT; ++d) dot += bf(q[d]) * bf(row[d]);
      z[j] = dot * c->scale;
      if (z[j] > m) m = z[j];
    }
    /* learnable sink ([ARCH] "Output gate + sink"): one more logit in the
     * denominator with no value row */
    if (c->sink && c->sink[h] > m) m = c->sink[h];
    double l = 0.0;
    for (int j = 0; j < n; ++j) {
      double p = exp(z[j] - m);
      l += p;
      const uint16_t* row = kvb + (int64_t)sel[j] * RLAT;
      for (int d = 0; d < VLAT; ++d) oh[d] += p * bf(row[d]); /* value = first 512 dims */
    }
    if (c->sink) l += exp(c->sink[h] - m);
    for (int d = 0; d < VLAT; ++d) oh[d] /= l;
    lse[h] = m + log(l);
  }
  free(z);
  free(sel);
}

static int mla_common(const uint16_t* q_lat, const uint16_t* kv, const int32_t* idx,
                      const int32_t* q_start, const int32_t* kv_len, int B, int Tq, int S_max,
                      int H, int topk, double scale, int64_t n_rows, const int64_t* rows,
                      double* o, double* lse, const double* sink) {
  if (!q_lat || !kv || !q_start || !kv_len || !rows || !o || !lse) return OR_BAD_ARG;
  if (!idx || topk <= 0) return OR_BAD_ARG;
  if (B <= 0 || Tq <= 0 || S_max <= 0 || H <= 0 || n_rows < 0) return OR_BAD_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= (int64_t)B * Tq) return OR_BAD_ARG;
  mla_ctx c = {q_lat, kv, idx, q_start, kv_len, Tq, S_max, H, topk, scale,
               rows, o, lse, sink, OR_OK};
  parallel_rows(n_rows, mla_row, &c);
  return c.err;
}

/* q_lat [B,Tq,H,576], kv [B,S_max,576] (BF16 bits), idx [B,Tq,topk] (-1 = unused);
 * o [n_rows,H,512], lse [n_rows,H] (natural log). */
int oracle_sparse_mla(const uint16_t* q_lat, const uint16_t* kv, const int32_t* idx,
                      const int32_t* q_start, const int32_t* kv_len, int B, int Tq, int S_max,
                      int H, int topk, double scale, int64_t n_rows, const int64_t* rows,
                      double* o, double* lse) {
  return mla_common(q_lat, kv, idx, q_start, kv_len, B, Tq, S_max, H, topk, scale, n_rows,
                    rows, o, lse, NULL);
}

/* The same with a learnable sink: sink [H] logits (natural log) that join the
 * softmax denominator and carry no value: o = sum_s e^{z_s} v_s / (e^{sink} +
 * sum_s e^{z_s}), lse = log(e^{sink} + sum_s e^{z_s}). */
int oracle_sparse_mla_sink(const uint16_t* q_lat, const uint16_t* kv, const int32_t* idx,
                           const int32_t* q_start, const int32_t* kv_len, int B, int Tq, int S_max,
                           int H, int topk, double scale, const double* sink, int64_t n_rows,
                           const int64_t* rows, double* o, double* lse) {
  if (!sink) return OR_BAD_ARG;
  return mla_common(q_lat, kv, idx, q_start, kv_len, B, Tq, S_max, H, topk, scale, n_rows,
                    rows, o, lse, sink);
}

/* Dense causal MLA over every key s <= t: the dense-mask reference path, with
 * no index list at all.  Written as its own loops (keys outer, heads inner for
 * the logits; then one normalisation per head) so that it does not share the
 * sparse path's code: the "a sequence of at most k tokens keeps every causal
 * key" check ("Kimi-K3.1-Pro", Implementation Limits, bullet 4) then compares
 * two programs. */
typedef struct {
  const uint16_t *q, *kv;
  const int32_t *q_start, *kv_len;
  int Tq, S_max, H;
  double scale;
  const int64_t* rows;
  double *o, *lse;
  int err;
} dense_ctx;

static void dense_row(void* vctx, int64_t r) {
  dense_ctx* c = (dense_ctx*)vctx;
  const int64_t flat = c->rows[r];
  const int b = (int)(flat / c->Tq), i = (int)(flat % c->Tq);
  const int64_t t = (int64_t)c->q_start[b] + i;
  if (t < 0 || t >= c->kv_len[b] || t >= c->S_max) { c->err = OR_BAD_ARG; return; }
  const int64_t nk = t + 1;
  const uint16_t* qrow = c->q + flat * c->H * (int64_t)RLAT;
  const uint16_t* keys = c->kv + (int64_t)b * c->S_max * RLAT;
  /* z[h * nk + s]: every head's logit against every causal key */
  double* z = (double*)malloc(sizeof(double) * (size_t)(nk * c->H));
  if (!z) { c->err = OR_NOMEM; return; }
  for (int64_t s = 0; s < nk; ++s) {
    const uint16_t* krow = keys + s * RLAT;
    for (int h = 0; h < c->H; ++h) {
      const uint16_t* qh = qrow + (int64_t)h * RLAT;
      double acc = 0.0;
      for (int d = 0; d < RLAT; ++d) acc += bf(qh[d]) * bf(krow[d]);
      z[(int64_t)h * nk + s] = c->scale * acc;
    }
  }
  for (int h = 0; h < c->H; ++h) {
    const double* zh = z + (int64_t)h * nk;
    double m = zh[0];
    for (int64_t s = 1; s < nk; ++s) m = zh[s] > m ? zh[s] : m;
    double denom = 0.0;
    for (int64_t s = 0; s < nk; ++s) denom += exp(zh[s] - m);
    double* oh = c->o + (r * c->H + h) * (int64_t)VLAT;
    for (int d = 0; d < VLAT; ++d) {
      double num = 0.0;
      for (int64_t s = 0; s < nk; ++s) num += exp(zh[s] - m) * bf(keys[s * RLAT + d]);
      oh[d] = num / denom;
    }
    c->lse[r * c->H + h] = m + log(denom);
  }
  free(z);
}

int oracle_dense_mla(const uint16_t* q_lat, const uint16_t* kv, const int32_t* q_start,
                     const int32_t* kv_len, int B, int Tq, int S_max, int H, double scale,
                     int64_t n_rows, const int64_t* rows, double* o, double* lse) {
  if (!q_lat || !kv || !q_start || !kv_len || !rows || !o || !lse) return OR_BAD_ARG;
  if (B <= 0 || Tq <= 0 || S_max <= 0 || H <= 0 || n_rows < 0) return OR_BAD_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= (int64_t)B * Tq) return OR_BAD_ARG;
  dense_ctx c = {q_lat, kv, q_start, kv_len, Tq, S_max, H, scale, rows, o, lse, OR_OK};
  parallel_rows(n_rows, dense_row, &c);
  return c.err;
}

/* ------------------------------------------------------------------------- */
/* Explicit (non-absorbed) MLA: per-head K/V expanded through W_UK / W_UV      */
/* [K31 Impl. Limits b2: sparse MLA avoids this expansion; CFG dims]          */
/* ------------------------------------------------------------------------- */

typedef struct {
  const double *q_nope, *q_pe, *W_UK, *W_UV, *c_kv, *k_pe;
  const int32_t* sel;
  int H, dn, dr, R, dv, K;
  double scale;
  double* out;
} exp_ctx;

static void explicit_row(void* vctx, int64_t r) {
  exp_ctx* c = (exp_ctx*)vctx;
  const int32_t* sel = c->sel + r * (int64_t)c->K;
  int n = 0;
  for (int j = 0; j < c->K; ++j)
    if (sel[j] >= 0) ++n;
  double* z = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double* kh = (double*)malloc(sizeof(double) * (size_t)c->dn);
  double* vh = (double*)malloc(sizeof(double) * (size_t)c->dv);
  for (int h = 0; h < c->H; ++h) {
    const double* qn = c->q_nope + (r * c->H + h) * (int64_t)c->dn;
    const double* qp = c->q_pe + (r * c->H + h) * (int64_t)c->dr;
    const double* Wk = c->W_UK + (int64_t)h * c->dn * c->R; /* [dn, R] */
    const double* Wv = c->W_UV + (int64_t)h * c->dv * c->R; /* [dv, R] */
    double* oh = c->out + (r * c->H + h) * (int64_t)c->dv;
    for (int e = 0; e < c->dv; ++e) oh[e] = 0.0;
    if (n == 0) continue;
    double m = -INFINITY;
    int jj = 0;
    for (int j = 0; j < c->K; ++j) {
      int s = sel[j];
      if (s < 0) continue;
      const double* ck = c->c_kv + (int64_t)s * c->R;
      /* k_nope_h[s] = W_UK_h c_kv[s] */
      for (int a = 0; a < c->dn; ++a) {
        double acc = 0.0;
        for (int d = 0; d < c->R; ++d) acc += Wk[(int64_t)a * c->R + d] * ck[d];
        kh[a] = acc;
      }
      double dot = 0.0;
      for (int a = 0; a < c->dn; ++a) dot += qn[a] * kh[a];
      const double* kp = c->k_pe + (int64_t)s * c->dr;
      for (int a = 0; a < c->dr; ++a) dot += qp[a] * kp[a];
      z[jj] = dot * c->scale;
      if (z[jj] > m) m = z[jj];
      ++jj;
    }
    double l = 0.0;
    jj = 0;
    for (int j = 0; j < c->K; ++j) {
      int s = sel[j];
      if (s < 0) continue;
      double p = exp(z[jj++] - m);
      l += p;
      const double* ck = c->c_kv + (int64_t)s * c->R;
      /* v_h[s] = W_UV_h c_kv[s] */
      for (int e = 0; e < c->dv; ++e) {
        double acc = 0.0;
        for (int d = 0; d < c->R; ++d) acc += Wv[(int64_t)e * c->R + d] * ck[d];
        vh[e] = acc;
      }
      for (int e = 0; e < c->dv; ++e) oh[e] += p * vh[e];
    }
    for (int e = 0; e < c->dv; ++e) oh[e] /= l;
  }
  free(z);
  free(kh);
  free(vh);
}

/* q_nope [n,H,dn], q_pe [n,H,dr], W_UK [H,dn,R], W_UV [H,dv,R], c_kv [S,R],
 * k_pe [S,dr], sel [n,K] (-1 = unused) -> out [n,H,dv]; all double. */
int oracle_explicit_mla(const double* q_nope, const double* q_pe, const double* W_UK,
                        const double* W_UV, const double* c_kv, const double* k_pe,
                        const int32_t* sel, int64_t n, int H, int dn, int dr, int R, int dv,
                        int K, double scale, double* out) {
  if (!q_nope || !q_pe || !W_UK || !W_UV || !c_kv || !k_pe || !sel || !out) return OR_BAD_ARG;
  if (n < 0 || H <= 0 || dn <= 0 || dr < 0 || R <= 0 || dv <= 0 || K <= 0) return OR_BAD_ARG;
  exp_ctx c = {q_nope, q_pe, W_UK, W_UV, c_kv, k_pe, sel, H, dn, dr, R, dv, K, scale, out};
  parallel_rows(n, explicit_row, &c);
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Output gate  [ARCH "Output gate + sink"; K31 Impl. Limits closing para;    */
/*               CFG mla_use_output_gate, v_head_dim]                        */
/* ------------------------------------------------------------------------- */

typedef struct {
  const uint16_t *x, *W_g, *W_uv;
  const double* o_lat;
  int hid, H, dv, R;
  const int64_t* rows;
  double* out;
} gate_ctx;

static void gate_row(void* vctx, int64_t r) {
  gate_ctx* c = (gate_ctx*)vctx;
  int64_t t = c->rows[r];
  const uint16_t* x = c->x + t * (int64_t)c->hid;
  double* o = c->out + r * (int64_t)c->H * c->dv;
  for (int h = 0; h < c->H; ++h) {
    const double* ol = c->o_lat + (t * c->H + h) * (int64_t)c->R;
    for (int e = 0; e < c->dv; ++e) {
      int64_t col = (int64_t)h * c->dv + e;
      /* g = x . W_g[col, :] */
      const uint16_t* wg = c->W_g + col * c->hid;
      double g = 0.0;
      for (int d = 0; d < c->hid; ++d) g += bf(x[d]) * bf(wg[d]);
      /* per-head value after the up-projection: u = W_UV_h[e, :] . o_lat_h */
      const uint16_t* wu = c->W_uv + ((int64_t)h * c->dv + e) * c->R;
      double u = 0.0;
      for (int d = 0; d < c->R; ++d) u += bf(wu[d]) * ol[d];
      o[col] = u / (1.0 + exp(-g)); /* sigma(g) * u */
    }
  }
}

/* x [N,hid], W_g [H*dv,hid], W_uv [H,dv,R] (BF16 bits); o_lat [N,H,R] double;
 * out [n_rows, H*dv]. */
int oracle_gate(const uint16_t* x, const uint16_t* W_g, const double* o_lat, const uint16_t* W_uv,
                int64_t N, int hid, int H, int dv, int R, int64_t n_rows, const int64_t* rows,
                double* out) {
  if (!x || !W_g || !o_lat || !W_uv || !rows || !out) return OR_BAD_ARG;
  if (N <= 0 || hid <= 0 || H <= 0 || dv <= 0 || R <= 0 || n_rows < 0) return OR_BAD_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return OR_BAD_ARG;
  gate_ctx c = {x, W_g, W_uv, o_lat, hid, H, dv, R, rows, out};
  parallel_rows(n_rows, gate_row, &c);
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Indexer-key LayerNorm  [ARCH "LayerNorm on the indexer key"; CFG          */
/*                         rms_norm_eps for eps]                             */
/* ------------------------------------------------------------------------- */

/* x [n, D] float -> y [n, D] double:  y = (x - mean x) / sqrt(var x + eps),
 * population variance over the row, unit gain and zero bias (the blueprint
 * names the normalisation and nothing else).  Mean and variance are the plain
 * sums of the definition in double, the variance over the centred values. */
int oracle_layernorm(const float* x, int64_t n, int D, double eps, double* y) {
  if (!x || !y || n < 0 || D <= 0 || !(eps >= 0.0)) return OR_BAD_ARG;
  for (int64_t r = 0; r < n; ++r) {
    const float* xr = x + r * (int64_t)D;
    double* yr = y + r * (int64_t)D;
    double mean = 0.0;
    for (int d = 0; d < D; ++d) mean += (double)xr[d];
    mean /= D;
    double var = 0.0;
    for (int d = 0; d < D; ++d) var += ((double)xr[d] - mean) * ((double)xr[d] - mean);
    var /= D;
    const double inv = 1.0 / sqrt(var + eps);
    for (int d = 0; d < D; ++d) yr[d] = ((double)xr[d] - mean) * inv;
  }
  return OR_OK;
}

/* Round each double to the nearest BF16 value (8 significant bits, ties to
 * even) and return the 16-bit patterns.  Written from the definition: the
 * significand is scaled to [128, 256), rounded to an integer with the default
 * round-half-even mode, and the result (exactly a float) gives the top half of
 * its float bit pattern.  Finite values of normal float magnitude only. */
int oracle_bf16_rne(const double* v, int64_t n, uint16_t* out) {
  if (!v || !out || n < 0) return OR_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) {
    const double a = v[i];
    if (a == 0.0) {
      out[i] = signbit(a) ? 0x8000u : 0x0000u;
      continue;
    }
    if (!isfinite(a) || fabs(a) < 0x1p-126 || fabs(a) >= 0x1p127) return OR_BAD_ARG;
    int e;
    const double m = frexp(fabs(a), &e);   /* |a| = m * 2^e, m in [0.5, 1) */
    double r = nearbyint(m * 256.0);       /* 8 significant bits */
    if (r == 256.0) { r = 128.0; e += 1; }
    const float f = (float)ldexp(a < 0 ? -r : r, e - 8);
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    out[i] = (uint16_t)(bits >> 16);
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* FP8 indexer variant  [K31 Impl. Limits b2: the FP8 indexer some serving    */
/*                       kernels use, set against the BF16 one]              */
/* ------------------------------------------------------------------------- */
/* The pages name the FP8 indexer and nothing more.  Readings (also in the
 * design notes):
 *   - the 8-bit format is E4M3: sign, 4 exponent bits with bias 7, 3 mantissa
 *     bits; exponent field 0 holds the subnormals m * 2^-9; the all-ones
 *     pattern S.1111.111 is NaN, so the largest finite magnitude is
 *     1.75 * 2^8 = 448; there is no infinity.  Encoding rounds to the nearest
 *     representable value, ties to the even mantissa, and saturates to +-448;
 *   - every row of D values (one indexer key, or one head of one query) has its
 *     own FP32 scale: amax = max |x| over the BF16 row,
 *     scale = max(amax, 2^-100) / 448, inv = 1 / scale, code = E4M3(x * inv),
 *     each of the three a single IEEE float operation rounded to nearest;
 *     the value a code stands for is scale * decode(code);
 *   - scores are the BF16 indexer's formula on those values.
 * The 2^-100 floor only keeps inv finite for an all-zero row (its codes are
 * all zero, so its values are exactly zero). */

#define E4M3_MAX 448.0

/* Magnitude of an E4M3 code (sign ignored). */
static double e4m3_mag(uint8_t c) {
  const int ex = (c >> 3) & 15, m = c & 7;
  if (ex == 0) return ldexp((double)m, -9);
  return ldexp(8.0 + m, ex - 10); /* (1 + m/8) * 2^(ex-7) */
}

static uint8_t e4m3_encode1(float xf) {
  const double x = (double)xf;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  const double a = fabs(x);
  if (!(a < E4M3_MAX)) return sign | 0x7E; /* saturate (also catches +-inf) */
  /* quantum of the binade [2^e, 2^(e+1)) is 2^(e-3); the subnormal range
   * [0, 2^-6) shares the quantum 2^-9 of the smallest normal binade */
  int e2;
  frexp(a, &e2);
  int e = e2 - 1;
  if (a == 0.0 || e < -6) e = -6;
  const double q = ldexp(1.0, e - 3);
  const double v = nearbyint(a / q) * q; /* a / q is exact; ties to even */
  if (v >= E4M3_MAX) return sign | 0x7E;
  /* find the code of v: exact search over the 127 finite magnitudes */
  for (int c = 0; c <= 0x7E; ++c)
    if (e4m3_mag((uint8_t)c) == v) return sign | (uint8_t)c;
  return 0xFF; /* unreachable: v is on the E4M3 grid */
}

/* float -> E4M3 codes (round to nearest even, saturating). */
int oracle_e4m3_encode(const float* x, int64_t n, uint8_t* out) {
  if (!x || !out || n < 0) return OR_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) {
    if (isnan(x[i])) return OR_BAD_ARG;
    out[i] = e4m3_encode1(x[i]);
  }
  return OR_OK;
}

/* E4M3 codes -> values (NaN for the two NaN patterns). */
int oracle_e4m3_decode(const uint8_t* c, int64_t n, double* out) {
  if (!c || !out || n < 0) return OR_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) {
    const uint8_t m = c[i] & 0x7F;
    const double v = m == 0x7F ? NAN : e4m3_mag(m);
    out[i] = (c[i] & 0x80) ? -v : v;
  }
  return OR_OK;
}

/* x [n, D] BF16 -> codes [n, D] E4M3 and scale [n] float, as stated above. */
int oracle_quant_fp8(const uint16_t* x, int64_t n, int D, uint8_t* codes, float* scale) {
  if (!x || !codes || !scale || n < 0 || D <= 0) return OR_BAD_ARG;
  for (int64_t r = 0; r < n; ++r) {
    const uint16_t* xr = x + r * (int64_t)D;
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
      const float a = (float)fabs(bf(xr[d]));
      if (isnan(a) || isinf(a)) return OR_BAD_ARG;
      if (a > amax) amax = a;
    }
    const float floor_ = 0x1p-100f;
    const float s = (amax > floor_ ? amax : floor_) / 448.0f;
    const float inv = 1.0f / s;
    scale[r] = s;
    for (int d = 0; d < D; ++d) {
      const float t = (float)bf(xr[d]) * inv;
      codes[r * (int64_t)D + d] = e4m3_encode1(t);
    }
  }
  return OR_OK;
}

typedef struct {
  const uint8_t *q, *k;
  const float *qs, *ks;
  const uint16_t* w;
  const int32_t *q_start, *kv_len;
  int Tq, S_max, H_I, D_I;
  const int64_t* rows;
  double* out;
  int err;
} idx8_ctx;

static double dec8(uint8_t c) {
  const double v = e4m3_mag(c & 0x7F);
  return (c & 0x80) ? -v : v;
}

static void indexer_row_fp8(void* vctx, int64_t r) {
  idx8_ctx* c = (idx8_ctx*)vctx;
  int64_t flat = c->rows[r];
  int b = (int)(flat / c->Tq), i = (int)(flat % c->Tq);
  int64_t t = (int64_t)c->q_start[b] + i;
  double* o = c->out + r * (int64_t)c->S_max;
  for (int64_t s = 0; s < c->S_max; ++s) o[s] = NAN;
  if (t >= c->kv_len[b] || t >= c->S_max) { c->err = OR_BAD_ARG; return; }
  const uint8_t* q = c->q + flat * (int64_t)c->H_I * c->D_I;
  const float* qs = c->qs + flat * (int64_t)c->H_I;
  const uint16_t* w = c->w + flat * (int64_t)c->H_I;
  const uint8_t* kb = c->k + (int64_t)b * c->S_max * c->D_I;
  const float* ksb = c->ks + (int64_t)b * c->S_max;
  for (int64_t s = 0; s <= t; ++s) {
    const uint8_t* k = kb + s * c->D_I;
    const double ks = (double)ksb[s];
    double score = 0.0;
    for (int j = 0; j < c->H_I; ++j) {
      const double qsj = (double)qs[j];
      double dot = 0.0;
      for (int d = 0; d < c->D_I; ++d) dot += (qsj * dec8(q[j * c->D_I + d])) * (ks * dec8(k[d]));
      const double pos = dot > 0.0 ? dot : 0.0; /* ReLU */
      score += bf(w[j]) * pos;
    }
    o[s] = score;
  }
}

/* q codes [B,Tq,H_I,D_I] + q_scale [B,Tq,H_I]; w [B,Tq,H_I] BF16;
 * k codes [B,S_max,D_I] + k_scale [B,S_max]: the indexer scores of the
 * dequantised rows, every causal key, NaN beyond t (as oracle_indexer_scores). */
int oracle_indexer_scores_fp8(const uint8_t* q_codes, const float* q_scale, const uint16_t* w,
                              const uint8_t* k_codes, const float* k_scale,
                              const int32_t* q_start, const int32_t* kv_len, int B, int Tq,
                              int S_max, int H_I, int D_I, int64_t n_rows, const int64_t* rows,
                              double* out) {
  if (!q_codes || !q_scale || !w || !k_codes || !k_scale || !q_start || !kv_len || !rows || !out)
    return OR_BAD_ARG;
  if (B <= 0 || Tq <= 0 || S_max <= 0 || H_I <= 0 || D_I <= 0 || n_rows < 0) return OR_BAD_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= (int64_t)B * Tq) return OR_BAD_ARG;
  idx8_ctx c = {q_codes, k_codes, q_scale, k_scale, w, q_start, kv_len, Tq, S_max, H_I, D_I,
                rows, out, OR_OK};
  parallel_rows(n_rows, indexer_row_fp8, &c);
  return c.err;
}

/* ------------------------------------------------------------------------- */
/* Sparse MLA backward  [K31 Impl. Limits b1-b2 (attention over the selected  */
/* rows only), the paragraph after b4 (a native 96-head backward), b3 (hard   */
/* top-k gives the indexer no gradient: the index set is a constant here)]    */
/* ------------------------------------------------------------------------- */
/* The forward, per query row and head, over the selected positions s_j:
 *   z_j = scale * q . kv[s_j]          (576 dims)
 *   p_j = exp(z_j - lse),  lse = log sum_j exp(z_j)
 *   o   = sum_j p_j kv[s_j, 0:512]
 * and its gradient for an upstream gradient dO of o (the plain chain rule):
 *   dp_j = dO . kv[s_j, 0:512],   D = sum_j p_j dp_j = dO . o
 *   dz_j = p_j (dp_j - D)
 *   dq   = scale * sum_j dz_j kv[s_j, 0:576]
 *   dkv[s_j, 0:576] += scale * dz_j q,   dkv[s_j, 0:512] += p_j dO
 * (the latent row is both the key, 576 dims, and the value, its first 512).
 * Entries -1 are skipped; any other entry must be causal (else OR_BAD_INDEX).
 * With a learnable sink (one logit per head, no value row) the sink joins the
 * denominator: lse = log(e^sink + sum_j e^z_j); p_j, o, D and the gradients
 * above keep their form (the sink carries no value and depends on neither q
 * nor the latent rows).
 * Inputs and outputs are double: the gradient of the function on exact values. */

typedef struct {
  const double *q, *kv, *dO;
  const int32_t *idx, *q_start, *kv_len;
  int Tq, S_max, H, topk;
  double scale;
  const int64_t* rows;
  double *o, *lse, *D, *dq; /* o / D / dq may be NULL */
  const double* sink;       /* [H] natural-log sink logits, or NULL */
  int err;
} mlab_ctx;

/* forward row (o, lse) and, when dO is given, D and dq */
static void mlab_row(void* vctx, int64_t r) {
  mlab_ctx* c = (mlab_ctx*)vctx;
  int64_t flat = c->rows[r];
  int b = (int)(flat / c->Tq), i = (int)(flat % c->Tq);
  int64_t t = (int64_t)c->q_start[b] + i;
  const int32_t* ix = c->idx + flat * (int64_t)c->topk;
  const double* kvb = c->kv + (int64_t)b * c->S_max * RLAT;
  double* z = (double*)malloc(sizeof(double) * (size_t)c->topk);
  if (!z) { c->err = OR_NOMEM; return; }
  for (int h = 0; h < c->H; ++h) {
    const double* qh = c->q + (flat * c->H + h) * (int64_t)RLAT;
    double m = -INFINITY;
    int n = 0;
    for (int j = 0; j < c->topk; ++j) {
      int s = ix[j];
      z[j] = -INFINITY;
      if (s < 0) continue;
      if (s > t || s >= c->kv_len[b] || s >= c->S_max) { c->err = OR_BAD_INDEX; continue; }
      const double* row = kvb + (int64_t)s * RLAT;
      double dot = 0.0;
      for (int d = 0; d < RLAT; ++d) dot += qh[d] * row[d];
      z[j] = c->scale * dot;
      if (z[j] > m) m = z[j];
      ++n;
    }
    const double sk = c->sink ? c->sink[h] : -INFINITY;
    if (sk > m) m = sk;
    double l = 0.0;
    for (int j = 0; j < c->topk; ++j)
      if (z[j] != -INFINITY) l += exp(z[j] - m);
    if (sk != -INFINITY) l += exp(sk - m);
    const double lse = m != -INFINITY ? m + log(l) : -INFINITY;
    if (c->lse) c->lse[r * c->H + h] = lse;
    double o[VLAT];
    for (int d = 0; d < VLAT; ++d) o[d] = 0.0;
    for (int j = 0; j < c->topk; ++j) {
      if (z[j] == -INFINITY) continue;
      const double p = exp(z[j] - lse);
      const double* row = kvb + (int64_t)ix[j] * RLAT;
      for (int d = 0; d < VLAT; ++d) o[d] += p * row[d];
    }
    if (c->o)
      for (int d = 0; d < VLAT; ++d) c->o[(r * c->H + h) * (int64_t)VLAT + d] = o[d];
    if (!c->dO) continue;
    const double* dOh = c->dO + (flat * c->H + h) * (int64_t)VLAT;
    double Dv = 0.0;
    for (int d = 0; d < VLAT; ++d) Dv += dOh[d] * o[d];
    if (c->D) c->D[r * c->H + h] = Dv;
    double* dqh = c->dq + (r * c->H + h) * (int64_t)RLAT;
    for (int d = 0; d < RLAT; ++d) dqh[d] = 0.0;
    for (int j = 0; j < c->topk; ++j) {
      if (z[j] == -INFINITY) continue;
      const double p = exp(z[j] - lse);
      const double* row = kvb + (int64_t)ix[j] * RLAT;
      double dp = 0.0;
      for (int d = 0; d < VLAT; ++d) dp += dOh[d] * row[d];
      const double dz = p * (dp - Dv);
      for (int d = 0; d < RLAT; ++d) dqh[d] += c->scale * dz * row[d];
    }
  }
  free(z);
}

/* Double-input sparse MLA forward: o [n_rows, H, 512], lse [n_rows, H] (natural log).
 * The same function as oracle_sparse_mla on exact values; the backward is its gradient. */
int oracle_sparse_mla_f64(const double* q, const double* kv, const int32_t* idx,
                          const int32_t* q_start, const int32_t* kv_len, int B, int Tq, int S_max,
                          int H, int topk, double scale, const double* sink, int64_t n_rows,
                          const int64_t* rows, double* o, double* lse) {
  if (!q || !kv || !idx || !q_start || !kv_len || !rows || !o || !lse) return OR_BAD_ARG;
  if (B <= 0 || Tq <= 0 || S_max <= 0 || H <= 0 || topk <= 0 || n_rows < 0) return OR_BAD_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= (int64_t)B * Tq) return OR_BAD_ARG;
  mlab_ctx c = {q, kv, NULL, idx, q_start, kv_len, Tq, S_max, H, topk, scale, rows,
                o, lse, NULL, NULL, sink, OR_OK};
  parallel_rows(n_rows, mlab_row, &c);
  return c.err;
}

typedef struct {
  const double *q, *kv, *dO, *lse, *D;
  const int32_t* idx;
  const int64_t *start, *list; /* inverted lists: for key row kr, entries start[kr]..start[kr+1] */
  int Tq, S_max, H, topk;
  double scale;
  double* dkv;
} dkv_ctx;

/* dkv of one key row (b, s): the sum over every (query row, head) that selected it */
static void dkv_row(void* vctx, int64_t kr) {
  dkv_ctx* c = (dkv_ctx*)vctx;
  int b = (int)(kr / c->S_max);
  const double* row = c->kv + kr * RLAT;
  double* out = c->dkv + kr * RLAT;
  for (int d = 0; d < RLAT; ++d) out[d] = 0.0;
  for (int64_t e = c->start[kr]; e < c->start[kr + 1]; ++e) {
    const int64_t flat = c->list[e]; /* query row b*Tq + i (one entry per selection) */
    (void)b;
    for (int h = 0; h < c->H; ++h) {
      const double* qh = c->q + (flat * c->H + h) * (int64_t)RLAT;
      const double* dOh = c->dO + (flat * c->H + h) * (int64_t)VLAT;
      double dot = 0.0;
      for (int d = 0; d < RLAT; ++d) dot += qh[d] * row[d];
      const double p = exp(dot * c->scale - c->lse[flat * c->H + h]);
      double dp = 0.0;
      for (int d = 0; d < VLAT; ++d) dp += dOh[d] * row[d];
      const double dz = p * (dp - c->D[flat * c->H + h]);
      for (int d = 0; d < RLAT; ++d) out[d] += c->scale * dz * qh[d];
      for (int d = 0; d < VLAT; ++d) out[d] += p * dOh[d];
    }
  }
}

/* q [B,Tq,H,576], kv [B,S_max,576], dO [B,Tq,H,512] (double); idx [B,Tq,topk].
 * Outputs: dq [B,Tq,H,576] and dkv [B,S_max,576] (every row written; rows no
 * query selected are zero). */
int oracle_sparse_mla_bwd(const double* q, const double* kv, const int32_t* idx,
                          const int32_t* q_start, const int32_t* kv_len, int B, int Tq, int S_max,
                          int H, int topk, double scale, const double* sink, const double* dO,
                          double* dq, double* dkv) {
  if (!q || !kv || !idx || !q_start || !kv_len || !dO || !dq || !dkv) return OR_BAD_ARG;
  if (B <= 0 || Tq <= 0 || S_max <= 0 || H <= 0 || topk <= 0) return OR_BAD_ARG;
  const int64_t nq = (int64_t)B * Tq, nk = (int64_t)B * S_max;
  int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)nq);
  double* lse = (double*)malloc(sizeof(double) * (size_t)(nq * H));
  double* D = (double*)malloc(sizeof(double) * (size_t)(nq * H));
  int64_t* start = (int64_t*)calloc((size_t)(nk + 1), sizeof(int64_t));
  if (!rows || !lse || !D || !start) { free(rows); free(lse); free(D); free(start); return OR_NOMEM; }
  for (int64_t r = 0; r < nq; ++r) rows[r] = r;
  /* pass 1: per query row, lse, D = dO . o and dq */
  mlab_ctx c = {q, kv, dO, idx, q_start, kv_len, Tq, S_max, H, topk, scale, rows,
                NULL, lse, D, dq, sink, OR_OK};
  parallel_rows(nq, mlab_row, &c);
  int err = c.err;
  /* inverted lists of the selections (valid entries only, query order) */
  for (int64_t r = 0; r < nq && err == OR_OK; ++r) {
    const int b = (int)(r / Tq);
    for (int j = 0; j < topk; ++j) {
      const int s = idx[r * topk + j];
      if (s >= 0) start[(int64_t)b * S_max + s + 1] += 1;
    }
  }
  for (int64_t k = 0; k < nk; ++k) start[k + 1] += start[k];
  int64_t* list = (int64_t*)malloc(sizeof(int64_t) * (size_t)(start[nk] > 0 ? start[nk] : 1));
  int64_t* fill = (int64_t*)malloc(sizeof(int64_t) * (size_t)nk);
  if (!list || !fill) { err = OR_NOMEM; }
  if (err == OR_OK) {
    for (int64_t k = 0; k < nk; ++k) fill[k] = start[k];
    for (int64_t r = 0; r < nq; ++r) {
      const int b = (int)(r / Tq);
      for (int j = 0; j < topk; ++j) {
        const int s = idx[r * topk + j];
        if (s >= 0) list[fill[(int64_t)b * S_max + s]++] = r;
      }
    }
    /* pass 2: per key row, dkv */
    dkv_ctx k2 = {q, kv, dO, lse, D, idx, start, list, Tq, S_max, H, topk, scale, dkv};
    parallel_rows(nk, dkv_row, &k2);
  }
  free(rows); free(lse); free(D); free(start); free(list); free(fill);
  return err;
}
