/*
 * dsa_oracle.c -- plain fp64 CPU oracle for diagonal-aware sparse decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or load
 * this file: only the tests, the package smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code with the CUDA library.
 *
 * Sources (page title, then section):
 *   [DAS-abstract]  "Understanding and Exploiting Diagonal Attention Sparsity in
 *                   Autoregressive Image Generation", arXiv abstract.
 *   [DAS-method]    same title, paper-daily summary, section "技术方法详解"
 *                   (method details).
 *   [DAS-formula]   same title, paper-daily summary, section "核心公式"
 *                   (core formula: masked softmax attention, the band mask M,
 *                   the sparsity 1 - sum(M)/N^2).
 *   [DAS-example]   same title, paper-daily summary, section "具体技术细节示例"
 *                   (worked example N=8, W=4, B=2, query i=6).
 *
 * Readings of the pages that this file follows (each is listed in the design
 * notes of the repository):
 *   - The decode kept set of request b and KV head hk, at query position
 *     i = L-1, is every prompt row j < P, the query row itself (offset 0), and
 *     every row j = i - o with 1 <= o <= W whose mask bit (o-1) is set.  The
 *     summary's band |i-j| <= B, j >= i-W is the mask with bits 0..B-1 set;
 *     decode is causal, so j <= i always.
 *   - "softmax(QK^T/sqrt(d) (.) M) V" removes masked entries from the softmax
 *     (their score is minus infinity), since the abstract says those KV entries
 *     are skipped and the worked example counts only the kept ones as reads.
 *   - Inputs are taken as stored (fp32 or bf16) and widened exactly to fp64;
 *     every operation after that is fp64.
 *
 * Everything is written as the plain definition, one (request, head) at a time.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1 };

/* Status codes returned by the entry points. */
enum {
  OR_OK = 0,
  OR_BAD_ARG = -1,      /* a size or pointer is out of range */
  OR_BAD_REQUEST = -2,  /* a per-request value (L, P, W, page id) is invalid */
  OR_NO_MEMORY = -3
};

typedef struct {
  int32_t batch, hq, hkv, head_dim;
  int32_t num_pages, max_pages, max_window, mask_words;
  int32_t q_dtype, kv_dtype;
  const void* q;              /* [batch][hq][head_dim]                    */
  const void* k_pages;        /* [num_pages][16][hkv][head_dim]           */
  const void* v_pages;        /* [num_pages][16][hkv][head_dim]           */
  const int32_t* page_table;  /* [batch][max_pages]                       */
  const int32_t* seq_len;     /* [batch]                                  */
  const int32_t* prompt_len;  /* [batch]                                  */
  const int32_t* window;      /* [batch]                                  */
  const int32_t* grid_w;      /* [batch]  (attention mass only)           */
  const uint32_t* keep_mask;  /* [batch][hkv][mask_words]                 */
  double scale;               /* softmax scale, 1/sqrt(head_dim)          */
} oracle_problem;

#define OR_PAGE 16

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double widen(const void* base, size_t idx, int32_t dtype) {
  if (dtype == OR_F32) return (double)((const float*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static int mask_bit(const uint32_t* mask, int32_t bit) {
  return (int)((mask[bit >> 5] >> (bit & 31)) & 1u);
}

/* ---------------------------------------------------------------------------
 * Kept set of one decode query [DAS-formula], [DAS-example], [DAS-abstract]:
 * every j in 0..i that is a prompt row, the query row, or a window row whose
 * offset bit is set.  Rows are listed in ascending j.  Returns the count.
 * ------------------------------------------------------------------------- */
int32_t oracle_kept_set(int32_t L, int32_t P, int32_t W, const uint32_t* mask,
                        int32_t* out_idx) {
  if (L < 1 || P < 0 || W < 0) return OR_BAD_REQUEST;
  int32_t i = L - 1, n = 0;
  for (int32_t j = 0; j <= i; ++j) {
    int32_t o = i - j;
    int keep = (j < P) || (o == 0) || (o >= 1 && o <= W && mask_bit(mask, o - 1));
    if (keep) out_idx[n++] = j;
  }
  return n;
}

/* ---------------------------------------------------------------------------
 * Pages that no later decode step can read [DAS-formula], [DAS-abstract]:
 * the kept set of any query i' >= i = L-1 holds prompt rows and rows of its
 * window i'-W .. i', so a row j with P <= j < i - W lies below every later
 * window and outside the prompt: it is never read again (reading: P and W of
 * a request stay fixed while it decodes).  Page p holds rows 16p .. 16p+15;
 * flags[p] = 1 when every one of them is such a row, for the ceil(L/16) pages
 * a request of length L maps.  Returns the count, or OR_BAD_REQUEST.
 * ------------------------------------------------------------------------- */
int32_t oracle_evictable_pages(int32_t L, int32_t P, int32_t W, uint8_t* flags) {
  if (L < 1 || P < 0 || W < 0) return OR_BAD_REQUEST;
  int32_t i = L - 1, pages = (L + OR_PAGE - 1) / OR_PAGE, count = 0;
  for (int32_t p = 0; p < pages; ++p) {
    int never = 1;
    for (int32_t j = p * OR_PAGE; j < (p + 1) * OR_PAGE; ++j)
      if (!(j >= P && j < i - W)) never = 0;
    flags[p] = (uint8_t)never;
    count += never;
  }
  return count;
}

/* ---------------------------------------------------------------------------
 * The summary's literal N x N mask [DAS-formula]: M_ij = 1 iff |i-j| <= B and
 * j >= i-W.  With causal != 0 the entries j > i are also cleared (decode).
 * ------------------------------------------------------------------------- */
void oracle_mask_matrix(int32_t N, int32_t W, int32_t B, int32_t causal, uint8_t* M) {
  for (int32_t i = 0; i < N; ++i)
    for (int32_t j = 0; j < N; ++j) {
      int32_t d = i > j ? i - j : j - i;
      int keep = (d <= B) && (j >= i - W);
      if (causal && j > i) keep = 0;
      M[(size_t)i * N + j] = (uint8_t)keep;
    }
}

/* Sparsity = 1 - sum_ij M_ij / N^2 [DAS-formula]. */
double oracle_sparsity(int32_t N, const uint8_t* M) {
  double s = 0.0;
  for (size_t t = 0; t < (size_t)N * N; ++t) s += (double)M[t];
  return 1.0 - s / ((double)N * (double)N);
}

/* ---------------------------------------------------------------------------
 * Softmax attention of one query over an explicit list of n rows [DAS-formula]:
 *   s_j = scale * sum_t q_t k_jt,  a_j = exp(s_j - m) / sum exp(s - m),
 *   out = sum_j a_j v_j,  lse = m + ln sum exp(s - m).
 * q, k, v are fp64; k and v are [n][D].  With n == 0 the output is NaN.
 * ------------------------------------------------------------------------- */
void oracle_attend_rows(int32_t D, const double* q, const double* k, const double* v,
                        int32_t n, double scale, double* out, double* lse) {
  if (n <= 0) {
    for (int32_t t = 0; t < D; ++t) out[t] = NAN;
    if (lse) *lse = NAN;
    return;
  }
  double* s = (double*)malloc((size_t)n * sizeof(double));
  if (!s) {
    for (int32_t t = 0; t < D; ++t) out[t] = NAN;
    if (lse) *lse = NAN;
    return;
  }
  double m = -INFINITY;
  for (int32_t r = 0; r < n; ++r) {
    double dot = 0.0;
    for (int32_t t = 0; t < D; ++t) dot += q[t] * k[(size_t)r * D + t];
    s[r] = dot * scale;
    if (s[r] > m) m = s[r];
  }
  double z = 0.0;
  for (int32_t r = 0; r < n; ++r) {
    s[r] = exp(s[r] - m);
    z += s[r];
  }
  for (int32_t t = 0; t < D; ++t) out[t] = 0.0;
  for (int32_t r = 0; r < n; ++r) {
    double a = s[r] / z;
    for (int32_t t = 0; t < D; ++t) out[t] += a * v[(size_t)r * D + t];
  }
  if (lse) *lse = m + log(z);
  free(s);
}

/* Row j of request b, KV head hk lives at page_table[b][j/16], slot j%16. */
static int row_offset(const oracle_problem* pr, int32_t b, int32_t hk, int32_t j,
                      size_t* off) {
  int32_t page_slot = j / OR_PAGE;
  if (page_slot < 0 || page_slot >= pr->max_pages) return 0;
  int32_t page = pr->page_table[(size_t)b * pr->max_pages + page_slot];
  if (page < 0 || page >= pr->num_pages) return 0;
  size_t prow = (size_t)page * OR_PAGE + (size_t)(j % OR_PAGE);
  *off = (prow * (size_t)pr->hkv + (size_t)hk) * (size_t)pr->head_dim;
  return 1;
}

static int check_problem(const oracle_problem* pr) {
  if (!pr || pr->batch < 0 || pr->hq < 1 || pr->hkv < 1 || pr->head_dim < 1) return 0;
  if (pr->hq % pr->hkv != 0) return 0;
  if (pr->max_pages < 1 || pr->num_pages < 1) return 0;
  if (pr->q_dtype != OR_F32 && pr->q_dtype != OR_BF16) return 0;
  if (pr->kv_dtype != OR_F32 && pr->kv_dtype != OR_BF16) return 0;
  return 1;
}

/* One (request, query head) of decode attention: gather the rows of its kept
 * set (sparse) or of 0..i (dense) through the page table, then attend. */
static int decode_one(const oracle_problem* pr, int sparse, int32_t b, int32_t h,
                      double* out, double* lse) {
  const int32_t D = pr->head_dim;
  const int32_t g = pr->hq / pr->hkv;
  const int32_t hk = h / g;
  const int32_t L = pr->seq_len[b];
  if (L < 1 || L > pr->max_pages * OR_PAGE) return OR_BAD_REQUEST;

  int32_t* idx = (int32_t*)malloc((size_t)L * sizeof(int32_t));
  if (!idx) return OR_NO_MEMORY;
  int32_t n;
  if (sparse) {
    int32_t P = pr->prompt_len[b], W = pr->window[b];
    if (W > pr->max_window || W > pr->mask_words * 32) {
      free(idx);
      return OR_BAD_REQUEST;
    }
    n = oracle_kept_set(L, P, W, pr->keep_mask + ((size_t)b * pr->hkv + hk) * pr->mask_words,
                        idx);
    if (n < 0) {
      free(idx);
      return n;
    }
  } else {
    n = L;
    for (int32_t j = 0; j < L; ++j) idx[j] = j;
  }

  double* q = (double*)malloc((size_t)D * sizeof(double));
  double* k = (double*)malloc((size_t)n * D * sizeof(double));
  double* v = (double*)malloc((size_t)n * D * sizeof(double));
  int rc = OR_OK;
  if (!q || !k || !v) rc = OR_NO_MEMORY;
  if (rc == OR_OK) {
    for (int32_t t = 0; t < D; ++t)
      q[t] = widen(pr->q, ((size_t)b * pr->hq + h) * D + t, pr->q_dtype);
    for (int32_t r = 0; r < n && rc == OR_OK; ++r) {
      size_t off;
      if (!row_offset(pr, b, hk, idx[r], &off)) {
        rc = OR_BAD_REQUEST;
        break;
      }
      for (int32_t t = 0; t < D; ++t) {
        k[(size_t)r * D + t] = widen(pr->k_pages, off + t, pr->kv_dtype);
        v[(size_t)r * D + t] = widen(pr->v_pages, off + t, pr->kv_dtype);
      }
    }
  }
  if (rc == OR_OK) oracle_attend_rows(D, q, k, v, n, pr->scale, out, lse);
  free(q);
  free(k);
  free(v);
  free(idx);
  return rc;
}

/* ---------------------------------------------------------------------------
 * Several query tokens of one request under the same mask [DAS-formula],
 * [DAS-abstract]: the last n rows of the cache are the query tokens
 * i = L-n .. L-1 (their K/V rows are already in the cache, as when a chunk of
 * prompt or image tokens is prefilled at once).  Query i attends over its own
 * causal kept set, the decode rule of oracle_kept_set with L = i+1 (reading:
 * the pages define the mask per query position, so every query of the chunk
 * uses it unchanged).  One (request, query slot t, query head h).
 * ------------------------------------------------------------------------- */
static int multi_one(const oracle_problem* pr, const int32_t* q_len, int32_t max_q, int32_t b,
                     int32_t t, int32_t h, double* out, double* lse) {
  const int32_t D = pr->head_dim;
  const int32_t g = pr->hq / pr->hkv;
  const int32_t hk = h / g;
  const int32_t L = pr->seq_len[b], n = q_len[b];
  const int32_t P = pr->prompt_len[b], W = pr->window[b];
  if (L < 1 || L > pr->max_pages * OR_PAGE || n < 0 || n > L || n > max_q || t < 0 || t >= n ||
      W > pr->max_window || W > pr->mask_words * 32)
    return OR_BAD_REQUEST;
  const int32_t i = L - n + t;
  int32_t* idx = (int32_t*)malloc((size_t)(i + 1) * sizeof(int32_t));
  if (!idx) return OR_NO_MEMORY;
  const int32_t cnt = oracle_kept_set(i + 1, P, W,
                                      pr->keep_mask + ((size_t)b * pr->hkv + hk) * pr->mask_words,
                                      idx);
  if (cnt < 0) {
    free(idx);
    return cnt;
  }
  double* q = (double*)malloc((size_t)D * sizeof(double));
  double* k = (double*)malloc((size_t)(cnt > 0 ? cnt : 1) * D * sizeof(double));
  double* v = (double*)malloc((size_t)(cnt > 0 ? cnt : 1) * D * sizeof(double));
  int rc = OR_OK;
  if (!q || !k || !v) rc = OR_NO_MEMORY;
  if (rc == OR_OK) {
    for (int32_t e = 0; e < D; ++e)
      q[e] = widen(pr->q, (((size_t)b * max_q + t) * pr->hq + h) * D + e, pr->q_dtype);
    for (int32_t r = 0; r < cnt && rc == OR_OK; ++r) {
      size_t off;
      if (!row_offset(pr, b, hk, idx[r], &off)) {
        rc = OR_BAD_REQUEST;
        break;
      }
      for (int32_t e = 0; e < D; ++e) {
        k[(size_t)r * D + e] = widen(pr->k_pages, off + e, pr->kv_dtype);
        v[(size_t)r * D + e] = widen(pr->v_pages, off + e, pr->kv_dtype);
      }
    }
  }
  if (rc == OR_OK) oracle_attend_rows(D, q, k, v, cnt, pr->scale, out, lse);
  free(q);
  free(k);
  free(v);
  free(idx);
  return rc;
}

/* ---------------------------------------------------------------------------
 * Attention mass of one (request, query head) over the dense causal softmax
 * [DAS-abstract: concentration on prompt and local tokens, diagonal pattern],
 * [DAS-method: raster order puts spatial neighbours at offsets k*w +- r].
 * Each row j of 0..i, offset o = i-j, goes to exactly one bin:
 *   0 prompt   j < P
 *   1 local    j >= P and o <= r_local
 *   2 diagonal j >= P, r_local < o <= W, and |o - k*w| <= r_diag for a k >= 1
 *   3 other    everything else.
 * offset_mass[o] = a_{i-o} for 0 <= o <= min(W, i); other entries are 0.
 * ------------------------------------------------------------------------- */
static int mass_one(const oracle_problem* pr, int32_t b, int32_t h, int32_t r_local,
                    int32_t r_diag, double* mass4, double* offset_mass) {
  const int32_t D = pr->head_dim;
  const int32_t g = pr->hq / pr->hkv;
  const int32_t hk = h / g;
  const int32_t L = pr->seq_len[b];
  const int32_t P = pr->prompt_len[b], W = pr->window[b], w = pr->grid_w[b];
  if (L < 1 || L > pr->max_pages * OR_PAGE || P < 0 || W < 0 || W > pr->max_window || w < 1)
    return OR_BAD_REQUEST;
  const int32_t i = L - 1;

  double* q = (double*)malloc((size_t)D * sizeof(double));
  double* s = (double*)malloc((size_t)L * sizeof(double));
  if (!q || !s) {
    free(q);
    free(s);
    return OR_NO_MEMORY;
  }
  for (int32_t t = 0; t < D; ++t)
    q[t] = widen(pr->q, ((size_t)b * pr->hq + h) * D + t, pr->q_dtype);
  double m = -INFINITY;
  for (int32_t j = 0; j <= i; ++j) {
    size_t off;
    if (!row_offset(pr, b, hk, j, &off)) {
      free(q);
      free(s);
      return OR_BAD_REQUEST;
    }
    double dot = 0.0;
    for (int32_t t = 0; t < D; ++t) dot += q[t] * widen(pr->k_pages, off + t, pr->kv_dtype);
    s[j] = dot * pr->scale;
    if (s[j] > m) m = s[j];
  }
  double z = 0.0;
  for (int32_t j = 0; j <= i; ++j) {
    s[j] = exp(s[j] - m);
    z += s[j];
  }
  for (int c = 0; c < 4; ++c) mass4[c] = 0.0;
  if (offset_mass)
    for (int32_t o = 0; o <= pr->max_window; ++o) offset_mass[o] = 0.0;
  for (int32_t j = 0; j <= i; ++j) {
    double a = s[j] / z;
    int32_t o = i - j;
    int bin;
    if (j < P) {
      bin = 0;
    } else if (o <= r_local) {
      bin = 1;
    } else {
      int near_row = 0;
      if (o <= W)
        for (int32_t k = 1; (int64_t)k * w - r_diag <= o; ++k)
          if (labs((long)o - (long)k * w) <= r_diag) near_row = 1;
      bin = near_row ? 2 : 3;
    }
    mass4[bin] += a;
    if (offset_mass && o <= W) offset_mass[o] = a;
  }
  free(q);
  free(s);
  return OR_OK;
}

/* ---------------------------------------------------------------------------
 * Thread pool over a list of (request, query head) tasks.
 * ------------------------------------------------------------------------- */
typedef struct {
  const oracle_problem* pr;
  int kind; /* 0 dense, 1 sparse, 2 mass, 3 several queries per request */
  const int32_t* q_len;
  int32_t max_q;
  const int32_t* bh;
  int32_t n_bh;
  int32_t r_local, r_diag;
  double* out;
  double* lse;
  double* mass;
  double* offset_mass;
  int32_t next;
  int32_t status;
  pthread_mutex_t lock;
} task_set;

static void* worker(void* arg) {
  task_set* ts = (task_set*)arg;
  const oracle_problem* pr = ts->pr;
  for (;;) {
    pthread_mutex_lock(&ts->lock);
    int32_t t = ts->next++;
    pthread_mutex_unlock(&ts->lock);
    if (t >= ts->n_bh) break;
    int32_t b, h, qt = 0;
    if (ts->kind == 3) {
      /* task t = (b, query slot, head) in row-major order over [batch][max_q][hq] */
      b = t / (ts->max_q * pr->hq);
      qt = (t / pr->hq) % ts->max_q;
      h = t % pr->hq;
    } else if (ts->bh) {
      b = ts->bh[2 * t];
      h = ts->bh[2 * t + 1];
    } else {
      b = t / pr->hq;
      h = t % pr->hq;
    }
    int rc;
    if (b < 0 || b >= pr->batch || h < 0 || h >= pr->hq) {
      rc = OR_BAD_ARG;
    } else if (ts->kind == 3) {
      rc = qt < ts->q_len[b] ? multi_one(pr, ts->q_len, ts->max_q, b, qt, h,
                                         ts->out + (size_t)t * pr->head_dim, ts->lse + t)
                             : OR_OK; /* slots past q_len are left as they are */
    } else if (ts->kind == 2) {
      rc = mass_one(pr, b, h, ts->r_local, ts->r_diag, ts->mass + (size_t)t * 4,
                    ts->offset_mass ? ts->offset_mass + (size_t)t * (pr->max_window + 1) : NULL);
    } else {
      rc = decode_one(pr, ts->kind, b, h, ts->out + (size_t)t * pr->head_dim,
                      ts->lse ? ts->lse + t : NULL);
    }
    if (rc != OR_OK) {
      pthread_mutex_lock(&ts->lock);
      if (ts->status == OR_OK) ts->status = rc;
      pthread_mutex_unlock(&ts->lock);
    }
  }
  return NULL;
}

static int run_tasks(task_set* ts, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 1024) nthreads = 1024;
  ts->next = 0;
  ts->status = OR_OK;
  pthread_mutex_init(&ts->lock, NULL);
  pthread_t* th = (pthread_t*)malloc((size_t)nthreads * sizeof(pthread_t));
  if (!th) {
    pthread_mutex_destroy(&ts->lock);
    return OR_NO_MEMORY;
  }
  int started = 0;
  for (int t = 0; t < nthreads; ++t)
    if (pthread_create(&th[t], NULL, worker, ts) == 0) ++started;
  if (started == 0) worker(ts);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  free(th);
  pthread_mutex_destroy(&ts->lock);
  return ts->status;
}

/* Decode attention for the listed (b, h) pairs (bh = [n_bh][2]), or for all
 * batch*hq pairs in (b, h) order when bh is NULL.  sparse != 0 uses the kept
 * set; sparse == 0 is dense causal attention over 0..i.  out is [n][head_dim],
 * lse is [n] or NULL. */
int32_t oracle_decode(const oracle_problem* pr, int32_t sparse, const int32_t* bh,
                      int32_t n_bh, double* out, double* lse, int32_t nthreads) {
  if (!check_problem(pr) || !out) return OR_BAD_ARG;
  task_set ts;
  memset(&ts, 0, sizeof ts);
  ts.pr = pr;
  ts.kind = sparse ? 1 : 0;
  ts.bh = bh;
  ts.n_bh = bh ? n_bh : pr->batch * pr->hq;
  ts.out = out;
  ts.lse = lse;
  return run_tasks(&ts, nthreads);
}

/* Attention-mass bins ([n][4]) and per-offset mass ([n][max_window+1] or NULL)
 * for the listed (b, h) pairs, or all pairs when bh is NULL. */
int32_t oracle_mass(const oracle_problem* pr, int32_t r_local, int32_t r_diag,
                    const int32_t* bh, int32_t n_bh, double* mass, double* offset_mass,
                    int32_t nthreads) {
  if (!check_problem(pr) || !mass || !pr->grid_w || r_local < 0 || r_diag < 0) return OR_BAD_ARG;
  task_set ts;
  memset(&ts, 0, sizeof ts);
  ts.pr = pr;
  ts.kind = 2;
  ts.bh = bh;
  ts.n_bh = bh ? n_bh : pr->batch * pr->hq;
  ts.r_local = r_local;
  ts.r_diag = r_diag;
  ts.mass = mass;
  ts.offset_mass = offset_mass;
  return run_tasks(&ts, nthreads);
}

/* Attention of several query tokens per request (multi_one) for every
 * (request, query slot t < q_len[b], head): q is [batch][max_q][hq][head_dim],
 * out [batch][max_q][hq][head_dim], lse [batch][max_q][hq]; slots t >= q_len[b]
 * are not written. */
int32_t oracle_multi(const oracle_problem* pr, const int32_t* q_len, int32_t max_q, double* out,
                     double* lse, int32_t nthreads) {
  if (!check_problem(pr) || !q_len || max_q < 0 || !out || !lse) return OR_BAD_ARG;
  task_set ts;
  memset(&ts, 0, sizeof ts);
  ts.pr = pr;
  ts.kind = 3;
  ts.q_len = q_len;
  ts.max_q = max_q;
  ts.n_bh = pr->batch * max_q * pr->hq;
  ts.out = out;
  ts.lse = lse;
  return run_tasks(&ts, nthreads);
}
