/*
 * fp64 CPU oracle for the DeepSeek Sparse Attention (DSA) layer hot path.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * definition that the CUDA path is checked against. Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the library's
 * product path never does. It shares no code, header or table with the CUDA
 * sources.
 *
 * What is computed, and where the pages define it:
 *
 *  valid(t, s)  "Support Ring Attention with DeepSeek DSA Sparse Indexer",
 *               Forward Flow step 3: the indexer mask is combined with the
 *               causal mask q_pos >= kv_pos (diagonal included). With segment
 *               ids (same page, Tests: indexer mask with / without segment
 *               ids; document packing in "Add Flash Attention Support to
 *               Deepseek v4") a key is valid only inside the query's document:
 *               seg[s] == seg[t].
 *
 *  index score  "DeepSeek3.2: Onboard sparse attention", Background: the
 *               indexer is a per-head q.k product giving an index score;
 *               "Implement QK attention head chunking for CSA", Description:
 *               per-head [B,H,S,S] products are reduced over the heads. The
 *               exact form used by this library:
 *                   I[t,s] = sum_h w[t,h] * max(0, sum_d q[t,h,d] * k[s,d])
 *               for valid (t,s); -inf elsewhere in s <= t.
 *
 *  fp8 scores   Same page, What this PR does item 4: the original indexer is an
 *               fp8 kernel over quantized activations. Inputs are OCP FP8
 *               E4M3 bytes (1 sign, 4 exponent bits with bias 7, 3 mantissa
 *               bits; exponent 0 is subnormal; S.1111.111 is NaN; no
 *               infinities), decoded exactly, and k carries a per-key scale:
 *                   I[t,s] = sum_h w[t,h] * max(0, sum_d q[t,h,d] * c_s * k[s,d])
 *               computed as written (the scale inside the dot product).
 *
 *  top-k        "DeepSeek3.2: Onboard sparse attention", Background / What
 *               this PR does: per query, the top-k keys by index score give
 *               the index mask. Ties go to the lower key index; -0.0 and +0.0
 *               are equal. m(t) = min(k, n(t)) valid keys are selected
 *               (n(t) = number of valid keys), emitted in ascending order,
 *               and the remaining k - m(t) slots hold -1.
 *
 *  attention    "Support Ring Attention with DeepSeek DSA Sparse Indexer",
 *               Forward Flow step 5: logits = where(mask, Q.K^T * scale,
 *               -inf), softmax over the keys, output P.V. The selected set is
 *               shared by all query heads; key/value head g = h / (H / Hkv).
 *               LSE = log sum_j exp(l_j). A query with no selected key gets
 *               O = 0 and LSE = -inf.
 *
 *  backward     Same page, Backward Flow step 6: dQ = dP.K, dK = dP^T.Q,
 *               dV = P^T.dO over the same mask, where "dP" is read as the
 *               gradient with respect to the logits: with
 *               dP_j = dO.V[s_j] and Delta = sum_c dO[c] O[c],
 *               dS_j = P_j (dP_j - Delta), dQ = scale sum_j dS_j K[s_j],
 *               dK[s_j] += scale dS_j Q, dV[s_j] += P_j dO.
 *
 * All arithmetic is fp64. bf16 inputs are widened exactly. Rows are spread
 * over POSIX threads; per-thread dK/dV partial sums are added in thread order.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* OCP FP8 E4M3 byte -> its exact value */
static double e4m3_to_double(uint8_t b) {
  const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);          /* subnormal: 0.m * 2^(1-7) */
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);        /* normal: 1.m * 2^(e-7) */
  return sign ? -v : v;
}

/* causal and same-document test */
static int valid_pair(const int32_t* seg_row, int64_t t, int64_t s) {
  if (s > t || s < 0) return 0;
  if (seg_row && seg_row[s] != seg_row[t]) return 0;
  return 1;
}

/* ------------------------------------------------------------------ threads */

typedef void (*row_fn)(void* ctx, int64_t r, int tid);

typedef struct {
  row_fn fn;
  void* ctx;
  int64_t nrows;
  int tid, nthreads;
} worker_t;

static void* worker_main(void* p) {
  worker_t* w = (worker_t*)p;
  /* rows interleaved over threads: row cost grows with t */
  for (int64_t r = w->tid; r < w->nrows; r += w->nthreads) w->fn(w->ctx, r, w->tid);
  return NULL;
}

static void for_rows(row_fn fn, void* ctx, int64_t nrows, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  worker_t ws[512];
  pthread_t th[512];
  for (int i = 0; i < nthreads; ++i) {
    ws[i].fn = fn; ws[i].ctx = ctx; ws[i].nrows = nrows; ws[i].tid = i; ws[i].nthreads = nthreads;
  }
  for (int i = 1; i < nthreads; ++i)
    if (pthread_create(&th[i], NULL, worker_main, &ws[i]) != 0) th[i] = 0;
  worker_main(&ws[0]);
  for (int i = 1; i < nthreads; ++i) {
    if (th[i]) pthread_join(th[i], NULL);
    else worker_main(&ws[i]);
  }
}

/* ------------------------------------------------------------ index scores */

typedef struct {
  const uint16_t *q, *k;     /* bf16 inputs, or NULL when q8 / k8 are given */
  const uint8_t *q8, *k8;    /* e4m3 inputs */
  const float* kscale;       /* per-key scale of k8, or NULL */
  const float* w;
  const int32_t* seg;
  int B, S, Hi, Di;
  const int64_t* rows;
  double* out;
} scores_ctx;

static double q_value(const scores_ctx* c, int64_t i) {
  return c->q8 ? e4m3_to_double(c->q8[i]) : bf16_to_double(c->q[i]);
}

static double k_value(const scores_ctx* c, int64_t b, int64_t s, int d) {
  const int64_t i = (b * c->S + s) * c->Di + d;
  if (!c->k8) return bf16_to_double(c->k[i]);
  const double scale = c->kscale ? (double)c->kscale[b * c->S + s] : 1.0;
  return scale * e4m3_to_double(c->k8[i]);
}

static void scores_row(void* p, int64_t r, int tid) {
  (void)tid;
  scores_ctx* c = (scores_ctx*)p;
  int64_t row = c->rows[r];
  int64_t b = row / c->S, t = row % c->S;
  const int32_t* seg_row = c->seg ? c->seg + b * c->S : NULL;
  double* out = c->out + r * (int64_t)c->S;
  double* qd = (double*)malloc(sizeof(double) * (size_t)c->Hi * c->Di);
  for (int64_t i = 0; i < (int64_t)c->Hi * c->Di; ++i)
    qd[i] = q_value(c, row * c->Hi * c->Di + i);
  for (int64_t s = 0; s < c->S; ++s) {
    if (s > t) { out[s] = NAN; continue; }              /* undefined above the diagonal */
    if (!valid_pair(seg_row, t, s)) { out[s] = -INFINITY; continue; }
    double acc = 0.0;
    for (int h = 0; h < c->Hi; ++h) {
      double dot = 0.0;
      for (int d = 0; d < c->Di; ++d) dot += qd[h * c->Di + d] * k_value(c, b, s, d);
      double relu = dot > 0.0 ? dot : 0.0;
      acc += (double)c->w[row * c->Hi + h] * relu;
    }
    out[s] = acc;
  }
  free(qd);
}

/*
 * Index scores for the query rows listed in rows[] (flat b*S + t).
 * q_idx [B,S,Hi,Di] bf16, k_idx [B,S,Di] bf16, w [B,S,Hi] f32, seg [B,S] or NULL.
 * out [nrows, S]: s <= t -> score, or -inf when invalid; s > t -> NaN.
 */
void oracle_index_scores(const uint16_t* q_idx, const uint16_t* k_idx, const float* w,
                         const int32_t* seg, int B, int S, int Hi, int Di, const int64_t* rows,
                         int64_t nrows, double* out, int nthreads) {
  scores_ctx c = {q_idx, k_idx, NULL, NULL, NULL, w, seg, B, S, Hi, Di, rows, out};
  for_rows(scores_row, &c, nrows, nthreads);
}

/*
 * The same scores from e4m3 bytes: q8 [B,S,Hi,Di], k8 [B,S,Di], kscale [B,S] or NULL.
 */
void oracle_index_scores_fp8(const uint8_t* q8, const uint8_t* k8, const float* kscale,
                             const float* w, const int32_t* seg, int B, int S, int Hi, int Di,
                             const int64_t* rows, int64_t nrows, double* out, int nthreads) {
  scores_ctx c = {NULL, NULL, q8, k8, kscale, w, seg, B, S, Hi, Di, rows, out};
  for_rows(scores_row, &c, nrows, nthreads);
}

/* Decode n e4m3 bytes. */
void oracle_e4m3_decode(const uint8_t* in, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_to_double(in[i]);
}

/* ------------------------------------------------------------------- top-k */

typedef struct {
  double v;
  int32_t s;
} cand_t;

/* larger score first; equal scores (including -0 == +0): lower index first */
static int cmp_score_desc(const void* a, const void* b) {
  const cand_t* x = (const cand_t*)a;
  const cand_t* y = (const cand_t*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->s > y->s) - (x->s < y->s);
}

static int cmp_int_asc(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

typedef struct {
  const double* scores;
  const int32_t* seg;
  int S, k;
  const int64_t* rows;
  int32_t *idx, *count;
} topk_ctx;

static void topk_row(void* p, int64_t r, int tid) {
  (void)tid;
  topk_ctx* c = (topk_ctx*)p;
  int64_t row = c->rows[r];
  int64_t b = row / c->S, t = row % c->S;
  const int32_t* seg_row = c->seg ? c->seg + b * c->S : NULL;
  const double* sc = c->scores + r * (int64_t)c->S;
  cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)(t + 1));
  int64_t n = 0;
  for (int64_t s = 0; s <= t; ++s)
    if (valid_pair(seg_row, t, s)) { cand[n].v = sc[s]; cand[n].s = (int32_t)s; ++n; }
  qsort(cand, (size_t)n, sizeof(cand_t), cmp_score_desc);
  int64_t m = n < c->k ? n : c->k;
  int32_t* out = c->idx + r * (int64_t)c->k;
  for (int64_t j = 0; j < m; ++j) out[j] = cand[j].s;
  qsort(out, (size_t)m, sizeof(int32_t), cmp_int_asc);
  for (int64_t j = m; j < c->k; ++j) out[j] = -1;
  if (c->count) c->count[r] = (int32_t)m;
  free(cand);
}

/*
 * Top-k over the valid keys of each listed row. scores [nrows, S] (only
 * s <= t is read). idx [nrows, k] ascending, -1 padded; count [nrows] or NULL.
 */
void oracle_topk(const double* scores, const int32_t* seg, int S, int k, const int64_t* rows,
                 int64_t nrows, int32_t* idx, int32_t* count, int nthreads) {
  topk_ctx c = {scores, seg, S, k, rows, idx, count};
  for_rows(topk_row, &c, nrows, nthreads);
}

/* ------------------------------------------------------- sparse attention */

typedef struct {
  const uint16_t *Q, *K, *V, *dO;
  const int32_t* idx;
  int B, S, H, Hkv, Dqk, Dv, k;
  double scale;
  const int64_t* rows;
  double *O, *lse;                 /* forward outputs per listed row */
  double *dQ;                      /* backward: per listed row */
  double *dK_part, *dV_part;       /* backward: per thread [B*S*Hkv*D] */
  int bad_index;                   /* set when an index is out of [-1, S) */
} attn_ctx;

/* the selected keys of row (b,t): causal & index mask */
static int64_t gather_keys(const attn_ctx* c, int64_t row, int64_t t, int32_t* keys, int* bad) {
  int64_t m = 0;
  for (int j = 0; j < c->k; ++j) {
    int32_t s = c->idx[row * c->k + j];
    if (s < -1 || s >= c->S) { *bad = 1; continue; }
    if (s < 0 || s > t) continue;
    keys[m++] = s;
  }
  return m;
}

/* forward for one (row, head): P (length m), O (Dv), LSE */
static void attn_head(const attn_ctx* c, int64_t row, int64_t b, int h, const int32_t* keys,
                      int64_t m, double* P, double* O, double* lse) {
  int g = h / (c->H / c->Hkv);
  const uint16_t* q = c->Q + (row * c->H + h) * c->Dqk;
  double mx = -INFINITY;
  for (int64_t j = 0; j < m; ++j) {
    const uint16_t* kr = c->K + ((b * c->S + keys[j]) * c->Hkv + g) * c->Dqk;
    double dot = 0.0;
    for (int d = 0; d < c->Dqk; ++d) dot += bf16_to_double(q[d]) * bf16_to_double(kr[d]);
    P[j] = dot * c->scale;
    if (P[j] > mx) mx = P[j];
  }
  for (int d = 0; d < c->Dv; ++d) O[d] = 0.0;
  if (m == 0) { *lse = -INFINITY; return; }
  double z = 0.0;
  for (int64_t j = 0; j < m; ++j) { P[j] = exp(P[j] - mx); z += P[j]; }
  for (int64_t j = 0; j < m; ++j) {
    P[j] /= z;
    const uint16_t* vr = c->V + ((b * c->S + keys[j]) * c->Hkv + g) * c->Dv;
    for (int d = 0; d < c->Dv; ++d) O[d] += P[j] * bf16_to_double(vr[d]);
  }
  *lse = mx + log(z);
}

static void fwd_row(void* p, int64_t r, int tid) {
  (void)tid;
  attn_ctx* c = (attn_ctx*)p;
  int64_t row = c->rows[r];
  int64_t b = row / c->S, t = row % c->S;
  int32_t* keys = (int32_t*)malloc(sizeof(int32_t) * (size_t)(c->k > 0 ? c->k : 1));
  double* P = (double*)malloc(sizeof(double) * (size_t)(c->k > 0 ? c->k : 1));
  int bad = 0;
  int64_t m = gather_keys(c, row, t, keys, &bad);
  if (bad) c->bad_index = 1;
  for (int h = 0; h < c->H; ++h)
    attn_head(c, row, b, h, keys, m, P, c->O + (r * c->H + h) * c->Dv, c->lse + r * c->H + h);
  free(keys);
  free(P);
}

/*
 * Sparse attention forward for the listed rows.
 * Q [B,S,H,Dqk], K [B,S,Hkv,Dqk], V [B,S,Hkv,Dv] bf16; idx [B,S,k] int32.
 * O [nrows,H,Dv], lse [nrows,H] fp64. Returns 0, or 1 if an index was outside [-1, S).
 */
int oracle_attn_fwd(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* idx,
                    int B, int S, int H, int Hkv, int Dqk, int Dv, int k, double scale,
                    const int64_t* rows, int64_t nrows, double* O, double* lse, int nthreads) {
  if (Hkv < 1 || H % Hkv != 0) return 2;
  attn_ctx c;
  memset(&c, 0, sizeof(c));
  c.Q = Q; c.K = K; c.V = V; c.idx = idx;
  c.B = B; c.S = S; c.H = H; c.Hkv = Hkv; c.Dqk = Dqk; c.Dv = Dv; c.k = k; c.scale = scale;
  c.rows = rows; c.O = O; c.lse = lse;
  for_rows(fwd_row, &c, nrows, nthreads);
  return c.bad_index;
}

static void bwd_row(void* p, int64_t r, int tid) {
  attn_ctx* c = (attn_ctx*)p;
  int64_t row = c->rows[r];
  int64_t b = row / c->S, t = row % c->S;
  int kk = c->k > 0 ? c->k : 1;
  int32_t* keys = (int32_t*)malloc(sizeof(int32_t) * (size_t)kk);
  double* P = (double*)malloc(sizeof(double) * (size_t)kk);
  double* O = (double*)malloc(sizeof(double) * (size_t)c->Dv);
  int bad = 0;
  int64_t m = gather_keys(c, row, t, keys, &bad);
  if (bad) c->bad_index = 1;
  size_t kd = (size_t)c->Dqk, vd = (size_t)c->Dv;
  double* dKp = c->dK_part + (size_t)tid * (size_t)c->B * c->S * c->Hkv * kd;
  double* dVp = c->dV_part + (size_t)tid * (size_t)c->B * c->S * c->Hkv * vd;
  for (int h = 0; h < c->H; ++h) {
    int g = h / (c->H / c->Hkv);
    double lse;
    attn_head(c, row, b, h, keys, m, P, O, &lse);
    const uint16_t* q = c->Q + (row * c->H + h) * c->Dqk;
    const uint16_t* dO = c->dO + (row * c->H + h) * c->Dv;
    double* dQ = c->dQ + (r * c->H + h) * c->Dqk;
    for (int d = 0; d < c->Dqk; ++d) dQ[d] = 0.0;
    double delta = 0.0;
    for (int d = 0; d < c->Dv; ++d) delta += bf16_to_double(dO[d]) * O[d];
    for (int64_t j = 0; j < m; ++j) {
      int64_t kv = (b * c->S + keys[j]) * c->Hkv + g;
      const uint16_t* kr = c->K + kv * c->Dqk;
      const uint16_t* vr = c->V + kv * c->Dv;
      double dp = 0.0;
      for (int d = 0; d < c->Dv; ++d) dp += bf16_to_double(dO[d]) * bf16_to_double(vr[d]);
      double ds = P[j] * (dp - delta);
      for (int d = 0; d < c->Dqk; ++d) {
        dQ[d] += c->scale * ds * bf16_to_double(kr[d]);
        dKp[kv * kd + d] += c->scale * ds * bf16_to_double(q[d]);
      }
      for (int d = 0; d < c->Dv; ++d) dVp[kv * vd + d] += P[j] * bf16_to_double(dO[d]);
    }
  }
  free(keys);
  free(P);
  free(O);
}

/*
 * Sparse attention backward. dQ [nrows,H,Dqk] for the listed rows; dK
 * [B,S,Hkv,Dqk] and dV [B,S,Hkv,Dv] collect the contributions of the listed
 * rows only (all rows -> the full gradient). Returns as oracle_attn_fwd.
 */
int oracle_attn_bwd(const uint16_t* Q, const uint16_t* K, const uint16_t* V, const int32_t* idx,
                    const uint16_t* dO, int B, int S, int H, int Hkv, int Dqk, int Dv, int k,
                    double scale, const int64_t* rows, int64_t nrows, double* dQ, double* dK,
                    double* dV, int nthreads) {
  if (Hkv < 1 || H % Hkv != 0) return 2;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  size_t nk = (size_t)B * S * Hkv * Dqk, nv = (size_t)B * S * Hkv * Dv;
  attn_ctx c;
  memset(&c, 0, sizeof(c));
  c.Q = Q; c.K = K; c.V = V; c.dO = dO; c.idx = idx;
  c.B = B; c.S = S; c.H = H; c.Hkv = Hkv; c.Dqk = Dqk; c.Dv = Dv; c.k = k; c.scale = scale;
  c.rows = rows; c.dQ = dQ;
  c.dK_part = (double*)calloc(nk * (size_t)nthreads, sizeof(double));
  c.dV_part = (double*)calloc(nv * (size_t)nthreads, sizeof(double));
  if (!c.dK_part || !c.dV_part) { free(c.dK_part); free(c.dV_part); return 3; }
  for_rows(bwd_row, &c, nrows, nthreads);
  for (size_t i = 0; i < nk; ++i) {
    double a = 0.0;
    for (int tI = 0; tI < nthreads; ++tI) a += c.dK_part[(size_t)tI * nk + i];
    dK[i] = a;
  }
  for (size_t i = 0; i < nv; ++i) {
    double a = 0.0;
    for (int tI = 0; tI < nthreads; ++tI) a += c.dV_part[(size_t)tI * nv + i];
    dV[i] = a;
  }
  free(c.dK_part);
  free(c.dV_part);
  return c.bad_index;
}

/* ------------------------------------------------------ indexer loss (f3) */
/*
 * The indexer's auxiliary loss. "Implement QK attention head chunking for CSA"
 * (the teacher of the indexer loss): the attention scores of every head are
 * turned into fp32 softmax probabilities over the keys, zeroed outside the
 * valid tokens and summed over the heads; the result is a stop-gradient target.
 * "Support Ring Attention with DeepSeek DSA Sparse Indexer" (Loss Harvesting &
 * Objective Injection): the loss is added to the training objective and its
 * gradient reaches the indexer's query and key projections.
 *
 * Plainest reading of what the pages leave open:
 *   - the valid tokens are the attention's own mask, the selected slots j of
 *     the row with 0 <= idx[t,j] <= t (a key listed twice counts twice);
 *   - the target is made a distribution by dividing the head sum by H:
 *         pbar_j = (1/H) sum_h softmax_j(scale * Q[t,h] . K[s_j, g(h)]);
 *   - the student is the softmax of the index scores over the same slots,
 *         q_j = exp(I[t,s_j]) / sum_i exp(I[t,s_i]);
 *   - the loss of row t is KL(pbar || q) = sum_j pbar_j (log pbar_j - log q_j),
 *     with 0 log 0 = 0; a row without a selected key has loss 0;
 *   - dL/dI[t,s_j] = g (q_j - pbar_j) for the objective g * sum_t L_t (the
 *     target is constant), and the chain rule through
 *         I[t,s] = sum_h w[t,h] max(0, z_h),  z_h = q_idx[t,h] . k_idx[s]
 *     takes the derivative of max(0, z) at z = 0 as 0:
 *         dw[t,h]      = sum_j dI_j max(0, z_hj)
 *         dq_idx[t,h]  = sum_j dI_j w[t,h] [z_hj > 0] k_idx[s_j]
 *         dk_idx[s_j] += sum_h dI_j w[t,h] [z_hj > 0] q_idx[t,h]
 */

typedef struct {
  const uint16_t *Q, *K;
  const int32_t* idx;
  const double* scores;   /* [nrows, S]: the index scores of each listed row */
  int B, S, H, Hkv, Dqk, k;
  double scale, grad_scale;
  const int64_t* rows;
  double *kl, *dI, *pbar;  /* [nrows], [nrows,k], [nrows,k] (pbar may be NULL) */
  int bad_index;
} iloss_ctx;

static void iloss_row(void* p, int64_t r, int tid) {
  (void)tid;
  iloss_ctx* c = (iloss_ctx*)p;
  int64_t row = c->rows[r];
  int64_t b = row / c->S, t = row % c->S;
  int kk = c->k > 0 ? c->k : 1;
  int* slot = (int*)malloc(sizeof(int) * (size_t)kk);
  int32_t* keys = (int32_t*)malloc(sizeof(int32_t) * (size_t)kk);
  double* pb = (double*)calloc((size_t)kk, sizeof(double));
  double* l = (double*)malloc(sizeof(double) * (size_t)kk);
  int64_t m = 0;
  for (int j = 0; j < c->k; ++j) {
    int32_t s = c->idx[row * c->k + j];
    if (s < -1 || s >= c->S) { c->bad_index = 1; continue; }
    if (s < 0 || s > t) continue;
    slot[m] = j;
    keys[m] = s;
    ++m;
  }
  for (int j = 0; j < c->k; ++j) c->dI[r * c->k + j] = 0.0;
  if (c->pbar)
    for (int j = 0; j < c->k; ++j) c->pbar[r * c->k + j] = 0.0;
  c->kl[r] = 0.0;
  if (m > 0) {
    /* teacher: per-head softmax of the attention logits, averaged over heads */
    for (int h = 0; h < c->H; ++h) {
      int g = h / (c->H / c->Hkv);
      const uint16_t* q = c->Q + (row * c->H + h) * c->Dqk;
      double mx = -INFINITY;
      for (int64_t i = 0; i < m; ++i) {
        const uint16_t* kr = c->K + ((b * c->S + keys[i]) * c->Hkv + g) * c->Dqk;
        double dot = 0.0;
        for (int d = 0; d < c->Dqk; ++d) dot += bf16_to_double(q[d]) * bf16_to_double(kr[d]);
        l[i] = dot * c->scale;
        if (l[i] > mx) mx = l[i];
      }
      double z = 0.0;
      for (int64_t i = 0; i < m; ++i) { l[i] = exp(l[i] - mx); z += l[i]; }
      for (int64_t i = 0; i < m; ++i) pb[i] += l[i] / z;
    }
    for (int64_t i = 0; i < m; ++i) pb[i] /= c->H;
    /* student: softmax of the index scores over the same slots */
    const double* I = c->scores + r * (int64_t)c->S;
    double mx = -INFINITY;
    for (int64_t i = 0; i < m; ++i)
      if (I[keys[i]] > mx) mx = I[keys[i]];
    double z = 0.0;
    for (int64_t i = 0; i < m; ++i) z += exp(I[keys[i]] - mx);
    double logz = mx + log(z);
    double kl = 0.0;
    for (int64_t i = 0; i < m; ++i) {
      double logq = I[keys[i]] - logz;
      if (pb[i] > 0.0) kl += pb[i] * (log(pb[i]) - logq);
      c->dI[r * c->k + slot[i]] = c->grad_scale * (exp(logq) - pb[i]);
      if (c->pbar) c->pbar[r * c->k + slot[i]] = pb[i];
    }
    c->kl[r] = kl;
  }
  free(slot);
  free(keys);
  free(pb);
  free(l);
}

/*
 * Indexer loss of the listed rows. Q [B,S,H,Dqk], K [B,S,Hkv,Dqk] bf16, idx
 * [B,S,k], scores [nrows,S] (the listed rows' index scores; only the selected
 * keys are read). kl [nrows]; dI [nrows,k] = dL/dI at each slot (0 at slots
 * that hold no selected key); pbar [nrows,k] (optional) = the target. Returns
 * 0, 1 if an index was outside [-1, S), 2 on bad head counts.
 */
int oracle_indexer_loss(const uint16_t* Q, const uint16_t* K, const int32_t* idx,
                        const double* scores, int B, int S, int H, int Hkv, int Dqk, int k,
                        double scale, double grad_scale, const int64_t* rows, int64_t nrows,
                        double* kl, double* dI, double* pbar, int nthreads) {
  if (Hkv < 1 || H % Hkv != 0) return 2;
  iloss_ctx c;
  memset(&c, 0, sizeof(c));
  c.Q = Q; c.K = K; c.idx = idx; c.scores = scores;
  c.B = B; c.S = S; c.H = H; c.Hkv = Hkv; c.Dqk = Dqk; c.k = k;
  c.scale = scale; c.grad_scale = grad_scale;
  c.rows = rows; c.kl = kl; c.dI = dI; c.pbar = pbar;
  for_rows(iloss_row, &c, nrows, nthreads);
  return c.bad_index;
}

typedef struct {
  const uint16_t *qi, *ki; /* q_idx [B,S,Hi,Di], k_idx [B,S,Di] bf16 */
  const float* w;          /* [B,S,Hi] */
  const int32_t* idx;
  const double* dI;        /* [nrows,k] */
  int B, S, Hi, Di, k;
  const int64_t* rows;
  double *dq, *dw;         /* [nrows,Hi,Di], [nrows,Hi] */
  double* dk_part;         /* per thread [B*S*Di] */
  int bad_index;
} ibwd_ctx;

static void ibwd_row(void* p, int64_t r, int tid) {
  ibwd_ctx* c = (ibwd_ctx*)p;
  int64_t row = c->rows[r];
  int64_t b = row / c->S, t = row % c->S;
  double* dq = c->dq + r * (int64_t)c->Hi * c->Di;
  double* dw = c->dw + r * (int64_t)c->Hi;
  double* dk = c->dk_part + (size_t)tid * (size_t)c->B * c->S * c->Di;
  for (int64_t i = 0; i < (int64_t)c->Hi * c->Di; ++i) dq[i] = 0.0;
  for (int h = 0; h < c->Hi; ++h) dw[h] = 0.0;
  for (int j = 0; j < c->k; ++j) {
    int32_t s = c->idx[row * c->k + j];
    if (s < -1 || s >= c->S) { c->bad_index = 1; continue; }
    if (s < 0 || s > t) continue;
    double g = c->dI[r * c->k + j];
    const uint16_t* kr = c->ki + (b * c->S + s) * c->Di;
    for (int h = 0; h < c->Hi; ++h) {
      const uint16_t* qr = c->qi + (row * c->Hi + h) * c->Di;
      double z = 0.0;
      for (int d = 0; d < c->Di; ++d) z += bf16_to_double(qr[d]) * bf16_to_double(kr[d]);
      if (z > 0.0) {
        dw[h] += g * z;
        double gw = g * (double)c->w[row * c->Hi + h];
        for (int d = 0; d < c->Di; ++d) {
          dq[h * c->Di + d] += gw * bf16_to_double(kr[d]);
          dk[(b * c->S + s) * c->Di + d] += gw * bf16_to_double(qr[d]);
        }
      }
    }
  }
}

/*
 * Gradient of the indexer loss into the indexer inputs, given dI [nrows,k]
 * (dL/dI at each slot of the listed rows). dq [nrows,Hi,Di], dw [nrows,Hi] for
 * the listed rows; dk [B,S,Di] collects the contributions of the listed rows
 * (all rows: the full gradient). Returns as oracle_indexer_loss.
 */
int oracle_indexer_loss_bwd(const uint16_t* q_idx, const uint16_t* k_idx, const float* w,
                            const int32_t* idx, const double* dI, int B, int S, int Hi, int Di,
                            int k, const int64_t* rows, int64_t nrows, double* dq, double* dk,
                            double* dw, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  size_t nk = (size_t)B * S * Di;
  ibwd_ctx c;
  memset(&c, 0, sizeof(c));
  c.qi = q_idx; c.ki = k_idx; c.w = w; c.idx = idx; c.dI = dI;
  c.B = B; c.S = S; c.Hi = Hi; c.Di = Di; c.k = k;
  c.rows = rows; c.dq = dq; c.dw = dw;
  c.dk_part = (double*)calloc(nk * (size_t)nthreads, sizeof(double));
  if (!c.dk_part) return 3;
  for_rows(ibwd_row, &c, nrows, nthreads);
  for (size_t i = 0; i < nk; ++i) {
    double a = 0.0;
    for (int tI = 0; tI < nthreads; ++tI) a += c.dk_part[(size_t)tI * nk + i];
    dk[i] = a;
  }
  free(c.dk_part);
  return c.bad_index;
}
