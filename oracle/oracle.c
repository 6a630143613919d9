/*
 * CPU oracle for fused DiT attention + post-attention Ulysses All-to-All layout.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file; only the tests, the package's smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header or constant with the CUDA path.
 *
 * What it computes (plain definitions, fp64 throughout, no blocking or fusion):
 *
 *  1. Exact non-causal attention per (batch b, head h), the operation that
 *     FlashAttention computes exactly ("X-Stage", pith.science review page,
 *     glossary entry "FlashAttention"; Figure 5 (d): FlashAttention produces the
 *     output of each head partition):
 *        s_j   = (sum_c q[b,h,n,c] * k[b,h,j,c]) / sqrt(d)
 *        m     = max_j s_j
 *        w_j   = exp(s_j - m)
 *        o[n,:] = sum_j w_j v[b,h,j,:] / sum_j w_j
 *     Inputs are bf16 bit patterns, widened exactly (bits << 16 -> float -> double).
 *
 *  2. The post-attention All-to-All layout (Figure 5 (d)-(e): the post-attention
 *     All-to-All restores the original sequence partition; abstract: the owner of
 *     an output tile stores it to its destination). Destination p receives the
 *     contiguous sequence rows [p*N/P, (p+1)*N/P) for every head:
 *        recv[p][b][i][h][c] = o[b][h][p*(N/P)+i][c],  0 <= p < P, 0 <= i < N/P
 *     and its inverse, which takes recv back to o. Both are explicit index loops
 *     over elements of any byte size, so they move bits and never round.
 *
 * Threads: rows are split across POSIX threads; each output element is
 * computed by exactly one thread with the same sequential loop, so the result
 * does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 bit pattern -> double, exactly: bf16 is the upper half of an IEEE float. */
static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* One query row of exact attention. q_row: d values; kh, vh: N x d of this head. */
static void attention_row(const uint16_t *q_row, const uint16_t *kh,
                          const uint16_t *vh, int N, int d, double *s,
                          double *out) {
  const double inv_sqrt_d = 1.0 / sqrt((double)d);
  double m = -INFINITY;
  for (int j = 0; j < N; ++j) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c)
      acc += bf16_bits_to_double(q_row[c]) *
             bf16_bits_to_double(kh[(size_t)j * d + c]);
    s[j] = acc * inv_sqrt_d;
    if (s[j] > m) m = s[j];
  }
  double denom = 0.0;
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  for (int j = 0; j < N; ++j) {
    double w = exp(s[j] - m);
    denom += w;
    for (int c = 0; c < d; ++c)
      out[c] += w * bf16_bits_to_double(vh[(size_t)j * d + c]);
  }
  for (int c = 0; c < d; ++c) out[c] /= denom;
}

/* A work item is one (b, h, row) triple; rows are listed explicitly so the same
 * code serves the full problem and a row sample. */
typedef struct {
  const uint16_t *q, *k, *v;
  double *o;               /* output rows, d doubles per listed item */
  const int64_t *items;    /* (bh, n) pairs, flattened: items[2t], items[2t+1] */
  int64_t n_items;
  int N, d;
  int64_t begin, end;      /* this thread's item range */
  int status;
} row_job;

static void *row_worker(void *arg) {
  row_job *jb = (row_job *)arg;
  double *s = (double *)malloc(sizeof(double) * (size_t)jb->N);
  if (!s) { jb->status = 1; return NULL; }
  for (int64_t t = jb->begin; t < jb->end; ++t) {
    int64_t bh = jb->items[2 * t], n = jb->items[2 * t + 1];
    const size_t head = (size_t)bh * (size_t)jb->N * (size_t)jb->d;
    attention_row(jb->q + head + (size_t)n * jb->d, jb->k + head, jb->v + head,
                  jb->N, jb->d, s, jb->o + (size_t)t * jb->d);
  }
  free(s);
  jb->status = 0;
  return NULL;
}

static int run_items(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     double *o, const int64_t *items, int64_t n_items, int N,
                     int d, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  if ((int64_t)nthreads > n_items) nthreads = (int)(n_items > 0 ? n_items : 1);
  pthread_t tid[512];
  row_job jobs[512];
  int started[512];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].q = q; jobs[t].k = k; jobs[t].v = v; jobs[t].o = o;
    jobs[t].items = items; jobs[t].n_items = n_items;
    jobs[t].N = N; jobs[t].d = d;
    jobs[t].begin = n_items * t / nthreads;
    jobs[t].end = n_items * (t + 1) / nthreads;
    jobs[t].status = 1;
    started[t] = pthread_create(&tid[t], NULL, row_worker, &jobs[t]) == 0;
    if (!started[t]) row_worker(&jobs[t]);
  }
  int bad = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (started[t]) pthread_join(tid[t], NULL);
    bad |= jobs[t].status;
  }
  return bad ? -1 : 0;
}

/* Full attention: q, k, v are [B][H][N][d] bf16 bits; o is [B][H][N][d] fp64. */
int oracle_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     double *o, int B, int N, int H, int d, int nthreads) {
  if (!q || !k || !v || !o || B < 0 || N < 0 || H < 0 || d <= 0) return -2;
  int64_t n_items = (int64_t)B * H * N;
  if (n_items == 0) return 0;
  int64_t *items = (int64_t *)malloc(sizeof(int64_t) * 2 * (size_t)n_items);
  if (!items) return -1;
  for (int64_t t = 0; t < n_items; ++t) {
    items[2 * t] = t / N;
    items[2 * t + 1] = t % N;
  }
  int rc = run_items(q, k, v, o, items, n_items, N, d, nthreads);
  free(items);
  return rc;
}

/* Sampled attention: computes only the listed rows. rows[t] is a row index n
 * taken for every (b, h); o_rows is [B*H][n_rows][d] fp64. */
int oracle_attention_rows(const uint16_t *q, const uint16_t *k,
                          const uint16_t *v, const int64_t *rows, int n_rows,
                          double *o_rows, int B, int N, int H, int d,
                          int nthreads) {
  if (!q || !k || !v || !rows || !o_rows || B < 0 || N < 0 || H < 0 || d <= 0 ||
      n_rows < 0)
    return -2;
  for (int r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return -2;
  int64_t n_items = (int64_t)B * H * n_rows;
  if (n_items == 0) return 0;
  int64_t *items = (int64_t *)malloc(sizeof(int64_t) * 2 * (size_t)n_items);
  if (!items) return -1;
  for (int64_t t = 0; t < n_items; ++t) {
    items[2 * t] = t / n_rows;
    items[2 * t + 1] = rows[t % n_rows];
  }
  int rc = run_items(q, k, v, o_rows, items, n_items, N, d, nthreads);
  free(items);
  return rc;
}

/* Layout transform: o [B][H][N][d] -> recv [P][B][N/P][H][d], elements of
 * esize bytes, copied bit for bit. recv holds the P shards back to back. */
int oracle_shard_layout(const void *o, void *recv, int B, int N, int H, int d,
                        int P, int esize) {
  if (!o || !recv || B < 0 || N < 0 || H < 0 || d <= 0 || P <= 0 || esize <= 0 ||
      N % P != 0)
    return -2;
  const int rows = N / P;
  const char *src = (const char *)o;
  char *dst = (char *)recv;
  for (int p = 0; p < P; ++p)
    for (int b = 0; b < B; ++b)
      for (int i = 0; i < rows; ++i)
        for (int h = 0; h < H; ++h)
          for (int c = 0; c < d; ++c) {
            int n = p * rows + i;
            size_t s_idx = (((size_t)b * H + h) * N + n) * d + c;
            size_t d_idx = ((((size_t)p * B + b) * rows + i) * H + h) * d + c;
            memcpy(dst + d_idx * esize, src + s_idx * esize, (size_t)esize);
          }
  return 0;
}

/* Inverse layout transform: recv [P][B][N/P][H][d] -> o [B][H][N][d]. */
int oracle_shard_layout_inverse(const void *recv, void *o, int B, int N, int H,
                                int d, int P, int esize) {
  if (!o || !recv || B < 0 || N < 0 || H < 0 || d <= 0 || P <= 0 || esize <= 0 ||
      N % P != 0)
    return -2;
  const int rows = N / P;
  const char *src = (const char *)recv;
  char *dst = (char *)o;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h)
      for (int n = 0; n < N; ++n)
        for (int c = 0; c < d; ++c) {
          int p = n / rows, i = n % rows;
          size_t s_idx = ((((size_t)p * B + b) * rows + i) * H + h) * d + c;
          size_t d_idx = (((size_t)b * H + h) * N + n) * d + c;
          memcpy(dst + d_idx * esize, src + s_idx * esize, (size_t)esize);
        }
  return 0;
}

int oracle_abi_version(void) { return 1; }
