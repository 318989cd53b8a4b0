/*
 * CPU oracle for MLA tree-verify attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the CPU-baseline leg of the benchmark
 * load this library.  The product path (the CUDA library) never calls it and
 * shares no code, header or table with it.
 *
 * What it computes is the plain definition of the verify step, written out in
 * fp64 from the exact bf16 input values, one (request, tree token, head) row at
 * a time:
 *
 *   keys(r,i) = { kv_pool[kv_indices[kv_indptr[r] + j]] : j < p_r }          (prefix)
 *             U { kv_pool[out_cache_loc[qo_indptr[r] + t]] : mask(r,i,t) }  (tree)
 *   s_k   = scale * sum_{d<576} q[qo_indptr[r]+i, h, d] * k[d]
 *   out   = sum_k exp(s_k - m) * k[0:512] / sum_k exp(s_k - m),  m = max_k s_k
 *   lse   = m + ln(sum_k exp(s_k - m))
 *
 * Sources (page title -- section):
 *  - prefix slots through kv_indices/kv_indptr, tree slots through
 *    out_cache_loc, mask through custom_mask + mask_indptr: "The Final Solder
 *    Joint" -- "The Three-Edits Sequence" (item 1) and "The Investigation".
 *  - absorbed query [num_tok, H, 576], latent pool [num_slots, 576]: "The Glue
 *    That Binds" -- "The Broader Engineering Effort".
 *  - masked keys take -inf before the softmax, online softmax over arbitrary
 *    prefix lengths: "The Glue That Connects" -- "Design Decisions and
 *    Trade-Offs" (mask handling; online softmax).
 *  - V is the first 512 latent dims of the same row (MLA latent shared by K
 *    and V): "The Glue That Connects" -- "The Context".
 *
 * Readings where the pages are silent (listed again in the design notes):
 *  - mask layout FULL_ROW: request r's mask is row-major [n_r, p_r + n_r] at
 *    mask_indptr[r]; tree column t lives at p_r + t; prefix columns are not
 *    read (the prefix is always visible).  TREE_ONLY: [n_r, n_r].
 *  - LSE is the natural log of the sum of exp(scaled score).
 *  - A row with no visible key: out = 0, lse = -inf.
 *
 * Built with gcc -O2, no fast-math; fp64 throughout; two passes (max, then
 * sums) exactly as the definition reads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EBADARG -1
#define ORACLE_EINDEX -2
#define ORACLE_ENOMEM -3

#define MASK_FULL_ROW 0
#define MASK_TREE_ONLY 1

/* bf16 bit pattern -> exact double (bf16 is the top half of an IEEE fp32). */
static double bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

typedef struct {
  const uint16_t *q, *kv_pool;
  int64_t num_slots;
  const int64_t *kv_indices;
  const int32_t *kv_indptr;
  const int64_t *out_cache_loc, *qo_indptr;
  const uint8_t *custom_mask;
  const int64_t *mask_indptr;
  int mask_layout, bs, num_heads, d_latent, d_rope;
  double scale;
  /* work list: (request, tree token, head) triples or "all heads" */
  const int64_t *rows; /* NULL: every (token, head); else token*H + h ids */
  int64_t nwork;
  double *out, *lse;
  /* shared counter */
  int64_t next;
  pthread_mutex_t mu;
  int err;
} job_t;

static int64_t find_request(const job_t *J, int64_t tok) {
  /* linear search is fine: bs is small */
  for (int r = 0; r < J->bs; ++r)
    if (tok >= J->qo_indptr[r] && tok < J->qo_indptr[r + 1]) return r;
  return -1;
}

/* mask(r,i,t): may tree token i of request r see tree token t? */
static int tree_visible(const job_t *J, int r, int64_t i, int64_t t, int64_t p, int64_t n) {
  int64_t base = J->mask_indptr[r];
  int64_t off = (J->mask_layout == MASK_FULL_ROW) ? base + i * (p + n) + p + t
                                                  : base + i * n + t;
  return J->custom_mask[off] != 0;
}

/* Computes one (token, head) row into out_row[d_latent], *lse_row.
 * scratch: room for p+n doubles of scores and p+n slot ids. */
static int one_row(const job_t *J, int64_t tok, int h, double *out_row, double *lse_row,
                   double *scores, int64_t *slots) {
  const int dqk = J->d_latent + J->d_rope;
  int64_t r = find_request(J, tok);
  if (r < 0) return ORACLE_EBADARG;
  const int64_t p = (int64_t)J->kv_indptr[r + 1] - (int64_t)J->kv_indptr[r];
  const int64_t n = J->qo_indptr[r + 1] - J->qo_indptr[r];
  const int64_t i = tok - J->qo_indptr[r];

  /* the visible key list */
  int64_t nk = 0;
  for (int64_t j = 0; j < p; ++j) slots[nk++] = J->kv_indices[(int64_t)J->kv_indptr[r] + j];
  for (int64_t t = 0; t < n; ++t)
    if (tree_visible(J, (int)r, i, t, p, n)) slots[nk++] = J->out_cache_loc[J->qo_indptr[r] + t];
  for (int64_t k = 0; k < nk; ++k)
    if (slots[k] < 0 || slots[k] >= J->num_slots) return ORACLE_EINDEX;

  for (int d = 0; d < J->d_latent; ++d) out_row[d] = 0.0;
  if (nk == 0) {
    *lse_row = -INFINITY;
    return ORACLE_OK;
  }
  const uint16_t *qrow = J->q + (tok * J->num_heads + h) * (int64_t)dqk;

  /* scores */
  double m = -INFINITY;
  for (int64_t k = 0; k < nk; ++k) {
    const uint16_t *krow = J->kv_pool + slots[k] * (int64_t)dqk;
    double acc = 0.0;
    for (int d = 0; d < dqk; ++d) acc += bf16_to_double(qrow[d]) * bf16_to_double(krow[d]);
    scores[k] = J->scale * acc;
    if (scores[k] > m) m = scores[k];
  }
  /* weights, normaliser, weighted sum of the first d_latent dims */
  double l = 0.0;
  for (int64_t k = 0; k < nk; ++k) {
    double w = exp(scores[k] - m);
    l += w;
    const uint16_t *vrow = J->kv_pool + slots[k] * (int64_t)dqk;
    for (int d = 0; d < J->d_latent; ++d) out_row[d] += w * bf16_to_double(vrow[d]);
  }
  for (int d = 0; d < J->d_latent; ++d) out_row[d] /= l;
  *lse_row = m + log(l);
  return ORACLE_OK;
}

static void *worker(void *arg) {
  job_t *J = (job_t *)arg;
  int64_t maxk = 0;
  for (int r = 0; r < J->bs; ++r) {
    int64_t k = (int64_t)J->kv_indptr[r + 1] - J->kv_indptr[r] + J->qo_indptr[r + 1] - J->qo_indptr[r];
    if (k > maxk) maxk = k;
  }
  double *scores = (double *)malloc(sizeof(double) * (size_t)(maxk + 1));
  int64_t *slots = (int64_t *)malloc(sizeof(int64_t) * (size_t)(maxk + 1));
  if (!scores || !slots) {
    pthread_mutex_lock(&J->mu);
    J->err = ORACLE_ENOMEM;
    pthread_mutex_unlock(&J->mu);
    free(scores);
    free(slots);
    return NULL;
  }
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int64_t w = J->next++;
    int stop = J->err != ORACLE_OK;
    pthread_mutex_unlock(&J->mu);
    if (stop || w >= J->nwork) break;
    int64_t id = J->rows ? J->rows[w] : w;
    int64_t tok = id / J->num_heads;
    int h = (int)(id % J->num_heads);
    int rc = one_row(J, tok, h, J->out + w * (int64_t)J->d_latent, J->lse + w, scores, slots);
    if (rc != ORACLE_OK) {
      pthread_mutex_lock(&J->mu);
      J->err = rc;
      pthread_mutex_unlock(&J->mu);
    }
  }
  free(scores);
  free(slots);
  return NULL;
}

/* Rows: NULL -> all total_q*H rows in (token, head) order; else nrows ids of the
 * form token*H + h.  out: [nrows, d_latent] doubles, lse: [nrows] doubles. */
int oracle_mla_tree_verify_rows(const uint16_t *q, const uint16_t *kv_pool, int64_t num_slots,
                                const int64_t *kv_indices, const int32_t *kv_indptr,
                                const int64_t *out_cache_loc, const int64_t *qo_indptr,
                                const uint8_t *custom_mask, const int64_t *mask_indptr,
                                int mask_layout, int bs, int num_heads, int d_latent, int d_rope,
                                double scale, const int64_t *rows, int64_t nrows, double *out,
                                double *lse, int num_threads) {
  if (!q || !kv_pool || !kv_indptr || !qo_indptr || !mask_indptr || !out || !lse) return ORACLE_EBADARG;
  if (bs < 0 || num_heads <= 0 || d_latent <= 0 || d_rope < 0) return ORACLE_EBADARG;
  if (mask_layout != MASK_FULL_ROW && mask_layout != MASK_TREE_ONLY) return ORACLE_EBADARG;
  job_t J;
  memset(&J, 0, sizeof J);
  J.q = q; J.kv_pool = kv_pool; J.num_slots = num_slots;
  J.kv_indices = kv_indices; J.kv_indptr = kv_indptr;
  J.out_cache_loc = out_cache_loc; J.qo_indptr = qo_indptr;
  J.custom_mask = custom_mask; J.mask_indptr = mask_indptr; J.mask_layout = mask_layout;
  J.bs = bs; J.num_heads = num_heads; J.d_latent = d_latent; J.d_rope = d_rope; J.scale = scale;
  J.rows = rows;
  J.nwork = rows ? nrows : (bs > 0 ? qo_indptr[bs] : 0) * num_heads;
  J.out = out; J.lse = lse;
  pthread_mutex_init(&J.mu, NULL);
  if (num_threads < 1) num_threads = 1;
  if (num_threads > 1024) num_threads = 1024;
  pthread_t th[1024];
  int started = 0;
  for (int t = 1; t < num_threads; ++t)
    if (pthread_create(&th[started], NULL, worker, &J) == 0) ++started;
  worker(&J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&J.mu);
  return J.err;
}

/* Merge of per-split partial results by log-sum-exp weights -- the plain
 * definition of combining split-K softmax partials:
 *   lse = ln sum_s exp(lse_s);  out = sum_s exp(lse_s - lse) * o_s.
 * Splits with lse_s = -inf carry no weight; if all are -inf, out = 0, lse = -inf.
 * o: [nsplit, nrows, d] doubles, lse_in: [nsplit, nrows]. */
int oracle_lse_combine(const double *o, const double *lse_in, int nsplit, int64_t nrows, int d,
                       double *out, double *lse) {
  if (!o || !lse_in || !out || !lse || nsplit < 1 || nrows < 0 || d < 1) return ORACLE_EBADARG;
  for (int64_t r = 0; r < nrows; ++r) {
    double m = -INFINITY;
    for (int s = 0; s < nsplit; ++s)
      if (lse_in[s * nrows + r] > m) m = lse_in[s * nrows + r];
    for (int j = 0; j < d; ++j) out[r * d + j] = 0.0;
    if (m == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double sum = 0.0;
    for (int s = 0; s < nsplit; ++s) sum += exp(lse_in[s * nrows + r] - m);
    double L = m + log(sum);
    for (int s = 0; s < nsplit; ++s) {
      double w = exp(lse_in[s * nrows + r] - L);
      if (w == 0.0) continue;
      for (int j = 0; j < d; ++j) out[r * d + j] += w * o[((int64_t)s * nrows + r) * d + j];
    }
    lse[r] = L;
  }
  return ORACLE_OK;
}
