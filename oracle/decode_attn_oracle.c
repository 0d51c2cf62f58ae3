/*
 * Plain f64 CPU oracle for paged grouped-query decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header, table or constant with the
 * CUDA library; the two are compared on the same seeded inputs.
 *
 * What it computes (the plain definition; the GPU path reaches the same
 * real-valued result by a faster route):
 *
 *   apache/tvm pull request 20426 "webgpu-decode-attention", commit message
 *   of the sharded nest: a paged decode attention kernel, whose output is
 *   checked against an f64 reference at 1..3060 positions.
 *   BackendStack21/mlx-runner pull request 3, commit "GQA-shared split
 *   attention": every query head of a GQA group reads the same K/V rows.
 *
 * For batch entry b, query head hq, KV head h = hq / G (G = Hq / Hkv, query
 * heads h*G .. h*G+G-1 share KV head h), L = seq_lens[b] and
 * lo = (window > 0) ? max(0, L - window) : 0:
 *   k_t  = K[page_table[b][t / PS]][t % PS][h][:]     (likewise v_t)
 *   s_t  = scale * sum_d q[b][hq][d] * k_t[d]          t in [lo, L)
 *   m    = max_t s_t,  w_t = exp(s_t - m),  Z = sum_t w_t
 *   out  = sum_t w_t * v_t / Z                         (zero row if L == lo)
 * All arithmetic is IEEE double; fp16 inputs are decoded exactly.  Each
 * output row is computed by one thread in ascending t, so the result does not
 * depend on the thread count.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes): contiguous head grouping hq -> hq / G; seq_lens counts every cached
 * position to attend (the new token's K/V is already in the cache, no mask
 * inside the step); a window attends the last min(L, window) positions; a
 * row with L == 0 is zero; a row whose attended pages fall outside [0, P) or
 * whose L is negative or above max_pages * PS is invalid: it is written as
 * zero and flagged in row_err.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -pthread (no FMA
 * contraction, so x86 and Arm builds round identically).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int32_t batch;           /* B */
  int32_t num_q_heads;     /* Hq */
  int32_t num_kv_heads;    /* Hkv, Hq % Hkv == 0 */
  int32_t head_dim;        /* D */
  int32_t page_size;       /* PS */
  int32_t max_pages;       /* columns of page_table */
  int32_t num_pages;       /* P, rows of k_pages / v_pages */
  int32_t dtype;           /* element format of q, K, V: 0 = IEEE binary16, 1 = bfloat16 */
} oracle_shape;

/* ---- IEEE 754 binary16 -> binary64, from the format's definition ------- */

/* sign s (1 bit), biased exponent e (5 bits, bias 15), fraction f (10 bits):
 *   e == 0:         (-1)^s * 2^-14 * (f / 1024)        (zero / subnormal)
 *   0 < e < 31:     (-1)^s * 2^(e-15) * (1 + f / 1024)
 *   e == 31:        infinity (f == 0) or NaN           */
double oracle_half_to_double(uint16_t bits) {
  int s = (bits >> 15) & 1;
  int e = (bits >> 10) & 0x1f;
  int f = bits & 0x3ff;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -24);
  } else if (e == 31) {
    mag = (f == 0) ? INFINITY : NAN;
  } else {
    mag = ldexp(1024.0 + (double)f, e - 25);
  }
  return s ? -mag : mag;
}

/* bfloat16 -> binary64: the upper half of an IEEE binary32, i.e. sign (1
 * bit), biased exponent e (8 bits, bias 127), fraction f (7 bits):
 *   e == 0:         (-1)^s * 2^-126 * (f / 128)        (zero / subnormal)
 *   0 < e < 255:    (-1)^s * 2^(e-127) * (1 + f / 128)
 *   e == 255:       infinity (f == 0) or NaN           */
double oracle_bf16_to_double(uint16_t bits) {
  int s = (bits >> 15) & 1;
  int e = (bits >> 7) & 0xff;
  int f = bits & 0x7f;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -133);
  } else if (e == 255) {
    mag = (f == 0) ? INFINITY : NAN;
  } else {
    mag = ldexp(128.0 + (double)f, e - 134);
  }
  return s ? -mag : mag;
}

static double g_half_table[65536];
static double g_bf16_table[65536];
static pthread_once_t g_half_once = PTHREAD_ONCE_INIT;
static void build_half_table(void) {
  for (uint32_t i = 0; i < 65536u; ++i) {
    g_half_table[i] = oracle_half_to_double((uint16_t)i);
    g_bf16_table[i] = oracle_bf16_to_double((uint16_t)i);
  }
}
/* decoding table of the shape's element format */
static const double* elem_table(const oracle_shape* sh) {
  pthread_once(&g_half_once, build_half_table);
  return sh->dtype == 1 ? g_bf16_table : g_half_table;
}

/* ---- gather through the page table ------------------------------------- */

/* Row of KV head h at logical position t of sequence b; NULL if the page id
 * the table holds for it is outside [0, P). */
static const uint16_t* kv_row(const oracle_shape* sh, const uint16_t* pages,
                              const int32_t* page_table, int b, int64_t t, int h) {
  int32_t phys = page_table[(int64_t)b * sh->max_pages + t / sh->page_size];
  if (phys < 0 || phys >= sh->num_pages) return NULL;
  int64_t slot = t % sh->page_size;
  int64_t off = (((int64_t)phys * sh->page_size + slot) * sh->num_kv_heads + h) * sh->head_dim;
  return pages + off;
}

/* Attended range [*lo, *hi) of sequence b; returns 0 if seq_len is valid. */
static int attended_range(const oracle_shape* sh, const int32_t* seq_lens, int b,
                          int32_t window, int64_t* lo, int64_t* hi) {
  int64_t L = seq_lens[b];
  int64_t cap = (int64_t)sh->max_pages * sh->page_size;
  if (L < 0 || L > cap) {
    *lo = *hi = 0;
    return -1;
  }
  *hi = L;
  *lo = (window > 0 && L > window) ? L - window : 0;
  return 0;
}

/* ---- one output row: two-pass exact softmax ---------------------------- */

static int one_row(const oracle_shape* sh, const uint16_t* q, const uint16_t* k_pages,
                   const uint16_t* v_pages, const int32_t* page_table, const int32_t* seq_lens,
                   double scale, int32_t window, int32_t row, double* out) {
  const double* H = elem_table(sh);
  const int D = sh->head_dim;
  const int G = sh->num_q_heads / sh->num_kv_heads;
  const int b = row / sh->num_q_heads;
  const int hq = row % sh->num_q_heads;
  const int h = hq / G;
  const uint16_t* qrow = q + (int64_t)row * D;
  for (int d = 0; d < D; ++d) out[d] = 0.0;

  int64_t lo, hi;
  if (attended_range(sh, seq_lens, b, window, &lo, &hi) != 0) return -1;
  for (int64_t t = lo; t < hi; ++t)
    if (!kv_row(sh, k_pages, page_table, b, t, h)) return -1;
  int64_t n = hi - lo;
  if (n <= 0) return 0;

  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  if (!s) return -2;
  /* pass 1: scores and their maximum */
  double m = -INFINITY;
  for (int64_t t = lo; t < hi; ++t) {
    const uint16_t* k = kv_row(sh, k_pages, page_table, b, t, h);
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += H[qrow[d]] * H[k[d]];
    s[t - lo] = scale * dot;
    if (s[t - lo] > m) m = s[t - lo];
  }
  /* pass 2: weights, their sum and the weighted sum of V rows */
  double Z = 0.0;
  for (int64_t t = lo; t < hi; ++t) {
    const uint16_t* v = kv_row(sh, v_pages, page_table, b, t, h);
    double w = exp(s[t - lo] - m);
    Z += w;
    for (int d = 0; d < D; ++d) out[d] += w * H[v[d]];
  }
  for (int d = 0; d < D; ++d) out[d] /= Z;
  free(s);
  return 0;
}

/* ---- threaded driver over output rows ---------------------------------- */

typedef struct {
  const oracle_shape* sh;
  const uint16_t *q, *k, *v;
  const int32_t *page_table, *seq_lens, *rows;
  double scale;
  int32_t window;
  int32_t begin, end;   /* slice of the row list handled by this thread */
  double* out;
  int32_t* row_err;
} row_job;

static void* run_rows(void* arg) {
  row_job* j = (row_job*)arg;
  for (int32_t i = j->begin; i < j->end; ++i) {
    int32_t row = j->rows ? j->rows[i] : i;
    int st = one_row(j->sh, j->q, j->k, j->v, j->page_table, j->seq_lens, j->scale, j->window,
                     row, j->out + (int64_t)i * j->sh->head_dim);
    if (j->row_err) j->row_err[i] = st ? 1 : 0;
  }
  return NULL;
}

static int shape_ok(const oracle_shape* sh) {
  return sh && sh->batch >= 0 && sh->num_q_heads > 0 && sh->num_kv_heads > 0 &&
         sh->num_q_heads % sh->num_kv_heads == 0 && sh->head_dim > 0 && sh->page_size > 0 &&
         sh->max_pages >= 0 && sh->num_pages >= 0 && (sh->dtype == 0 || sh->dtype == 1);
}

/*
 * Decode attention for the rows listed in rows[0..n_rows) (row = b*Hq + hq),
 * or for all B*Hq rows when rows is NULL.  q is [B][Hq][D], k_pages and
 * v_pages are [P][PS][Hkv][D], all fp16 bit patterns; page_table is
 * [B][max_pages], seq_lens [B].  out is [n_rows][D] f64.  row_err (nullable)
 * gets 1 for each invalid row.  Returns the number of invalid rows, or -1 for
 * a bad shape.
 */
int oracle_decode_attn_f64(const oracle_shape* sh, const uint16_t* q, const uint16_t* k_pages,
                           const uint16_t* v_pages, const int32_t* page_table,
                           const int32_t* seq_lens, double scale, int32_t window,
                           const int32_t* rows, int32_t n_rows, int32_t n_threads, double* out,
                           int32_t* row_err) {
  if (!shape_ok(sh)) return -1;
  if (!rows) n_rows = sh->batch * sh->num_q_heads;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > n_rows) n_threads = n_rows > 0 ? n_rows : 1;
  int32_t* errs = row_err ? row_err : (int32_t*)calloc((size_t)(n_rows > 0 ? n_rows : 1), 4);
  pthread_t* tid = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
  row_job* jobs = (row_job*)malloc(sizeof(row_job) * (size_t)n_threads);
  for (int i = 0; i < n_threads; ++i) {
    row_job j = {sh, q, k_pages, v_pages, page_table, seq_lens, rows, scale, window,
                 (int32_t)((int64_t)n_rows * i / n_threads),
                 (int32_t)((int64_t)n_rows * (i + 1) / n_threads), out, errs};
    jobs[i] = j;
  }
  for (int i = 1; i < n_threads; ++i) pthread_create(&tid[i], NULL, run_rows, &jobs[i]);
  run_rows(&jobs[0]);
  for (int i = 1; i < n_threads; ++i) pthread_join(tid[i], NULL);
  int bad = 0;
  for (int32_t i = 0; i < n_rows; ++i) bad += errs[i] ? 1 : 0;
  if (!row_err) free(errs);
  free(tid);
  free(jobs);
  return bad;
}

/* ---- shard partial and ordered merge ------------------------------------ */

/*
 * apache/tvm pull request 20426, sharded nest: each shard of the context keeps
 * an online-softmax state; BackendStack21/mlx-runner pull request 3: the
 * combine merges per-shard partials.  Partial of row (b, hq) over logical
 * positions [lo, hi) (clipped to nothing else: the caller picks the range):
 *   m = max s_t,  l = sum exp(s_t - m),  acc[:] = sum exp(s_t - m) * v_t[:]
 * An empty range gives m = -inf, l = 0, acc = 0.  Returns -1 on a bad page.
 */
int oracle_partial_f64(const oracle_shape* sh, const uint16_t* q, const uint16_t* k_pages,
                       const uint16_t* v_pages, const int32_t* page_table, int32_t b, int32_t hq,
                       double scale, int64_t lo, int64_t hi, double* m_out, double* l_out,
                       double* acc) {
  if (!shape_ok(sh)) return -1;
  const double* H = elem_table(sh);
  const int D = sh->head_dim;
  const int h = hq / (sh->num_q_heads / sh->num_kv_heads);
  const uint16_t* qrow = q + ((int64_t)b * sh->num_q_heads + hq) * D;
  for (int d = 0; d < D; ++d) acc[d] = 0.0;
  *m_out = -INFINITY;
  *l_out = 0.0;
  if (hi <= lo) return 0;
  double m = -INFINITY;
  for (int64_t t = lo; t < hi; ++t) {
    const uint16_t* k = kv_row(sh, k_pages, page_table, b, t, h);
    if (!k) return -1;
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += H[qrow[d]] * H[k[d]];
    if (scale * dot > m) m = scale * dot;
  }
  double l = 0.0;
  for (int64_t t = lo; t < hi; ++t) {
    const uint16_t* k = kv_row(sh, k_pages, page_table, b, t, h);
    const uint16_t* v = kv_row(sh, v_pages, page_table, b, t, h);
    if (!v) return -1;
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += H[qrow[d]] * H[k[d]];
    double w = exp(scale * dot - m);
    l += w;
    for (int d = 0; d < D; ++d) acc[d] += w * H[v[d]];
  }
  *m_out = m;
  *l_out = l;
  return 0;
}

/*
 * Merge n partials (m[i], l[i], acc[i*D..]) in ascending i:
 *   M = max_i m_i,  c_i = exp(m_i - M) (0 for an empty partial),
 *   out = sum_i c_i * acc_i / sum_i c_i * l_i      (zero row if the sum is 0)
 */
void oracle_merge_f64(int32_t n, int32_t D, const double* m, const double* l, const double* acc,
                      double* out) {
  double M = -INFINITY;
  for (int32_t i = 0; i < n; ++i)
    if (m[i] > M) M = m[i];
  double L = 0.0;
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  for (int32_t i = 0; i < n; ++i) {
    if (l[i] == 0.0) continue;
    double c = exp(m[i] - M);
    L += c * l[i];
    for (int d = 0; d < D; ++d) out[d] += c * acc[(int64_t)i * D + d];
  }
  if (L == 0.0) {
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    return;
  }
  for (int d = 0; d < D; ++d) out[d] /= L;
}

/* ---- paged K/V append ---------------------------------------------------- */

/*
 * idle-intelligence/llm-web pull request 8, suffix-prefill commit: new K/V
 * rows are scattered into the cache at their positions after the resident
 * prefix (the step before attention reads them).  For every b with
 * positions[b] >= 0 and every KV head h:
 *   k_pages[page_table[b][t / PS]][t % PS][h][:] = k_new[b][h][:],  t = positions[b]
 * (likewise v).  A position < 0 means no new row for that sequence.  A
 * position >= max_pages * PS or a page id outside [0, P) is invalid: nothing
 * is written for that sequence and row_err[b] (nullable) is set.  Plain
 * element copies of the fp16 bit patterns.  Returns the number of invalid
 * sequences, -1 for a bad shape.
 */
int oracle_kv_append_u16(const oracle_shape* sh, const uint16_t* k_new, const uint16_t* v_new,
                         const int32_t* positions, const int32_t* page_table, uint16_t* k_pages,
                         uint16_t* v_pages, int32_t* row_err) {
  if (!shape_ok(sh)) return -1;
  int bad = 0;
  for (int b = 0; b < sh->batch; ++b) {
    int64_t t = positions[b];
    int err = 0;
    if (t >= 0) {
      int64_t cap = (int64_t)sh->max_pages * sh->page_size;
      if (t >= cap) {
        err = 1;
      } else {
        int32_t phys = page_table[(int64_t)b * sh->max_pages + t / sh->page_size];
        if (phys < 0 || phys >= sh->num_pages) err = 1;
      }
      if (!err) {
        for (int h = 0; h < sh->num_kv_heads; ++h) {
          /* kv_row is const; the same offset arithmetic written out here */
          int32_t phys = page_table[(int64_t)b * sh->max_pages + t / sh->page_size];
          int64_t off =
              (((int64_t)phys * sh->page_size + t % sh->page_size) * sh->num_kv_heads + h) *
              sh->head_dim;
          const uint16_t* kn = k_new + ((int64_t)b * sh->num_kv_heads + h) * sh->head_dim;
          const uint16_t* vn = v_new + ((int64_t)b * sh->num_kv_heads + h) * sh->head_dim;
          for (int d = 0; d < sh->head_dim; ++d) {
            k_pages[off + d] = kn[d];
            v_pages[off + d] = vn[d];
          }
        }
      }
    }
    if (row_err) row_err[b] = err;
    bad += err;
  }
  return bad;
}

/* ---- several new query positions per sequence (causal) ------------------ */

/*
 * idle-intelligence/llm-web pull request 8, suffix-prefill commit: new tokens
 * attend to the resident cache and to each other (their K/V already
 * appended).  With T new tokens per sequence and L = seq_lens[b] counting
 * them, query t (0 <= t < T) of sequence b sits at position P = L - T + t and
 * attends the positions [lo, P + 1) with lo = (window > 0) ? max(0, P + 1 -
 * window) : 0: causal order among the new tokens, the window counted from
 * each query's own position.  A query with P < 0 (fewer cached positions
 * than queries) gives a zero row.  q is [B][T][Hq][D], out [B*T*Hq][D] in the
 * same order.  Each row is the single-query definition above with the
 * sequence length P + 1.  Returns the number of invalid rows, -1 on a bad
 * shape.
 */
int oracle_decode_attn_multi_f64(const oracle_shape* sh, int32_t T, const uint16_t* q,
                                 const uint16_t* k_pages, const uint16_t* v_pages,
                                 const int32_t* page_table, const int32_t* seq_lens,
                                 double scale, int32_t window, double* out, int32_t* row_err) {
  if (!shape_ok(sh) || T < 1) return -1;
  const int D = sh->head_dim;
  const int64_t cap = (int64_t)sh->max_pages * sh->page_size;
  int bad = 0;
  for (int b = 0; b < sh->batch; ++b) {
    for (int t = 0; t < T; ++t) {
      /* the sequence as query t sees it: one batch entry of length P + 1 */
      int64_t L = seq_lens[b];
      int32_t len_t = (L < 0 || L > cap) ? -1 : (int32_t)(L - T + t + 1);
      if (len_t < 0 && L >= 0 && L <= cap) len_t = 0;
      oracle_shape one = *sh;
      one.batch = 1;
      for (int hq = 0; hq < sh->num_q_heads; ++hq) {
        int64_t row = ((int64_t)b * T + t) * sh->num_q_heads + hq;
        int st = one_row(&one, q + ((int64_t)b * T + t) * sh->num_q_heads * D,
                         k_pages, v_pages, page_table + (int64_t)b * sh->max_pages, &len_t,
                         scale, window, hq, out + row * D);
        if (row_err) row_err[row] = st ? 1 : 0;
        bad += st ? 1 : 0;
      }
    }
  }
  return bad;
}
