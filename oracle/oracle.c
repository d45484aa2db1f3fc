/*
 * fp64 CPU oracle for the Ring Attention forward step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path (the GPU library and
 * its Python binding) may link, load or call this file; only the tests, the
 * smoke check and the benchmark's CPU-baseline leg use it.  It shares no code,
 * header or constant with the GPU library.
 *
 * What it computes.  The mKernel pages describe Ring Attention as
 * sequence-parallel attention in which each ring step rotates a KV chunk and
 * the local FlashAttention consumes the chunk received before (arxivdaily
 * abstract; dataforcee and chathome "five fused kernels" tables, Ring
 * Attention row; pwwt.cn analysis, Table 3, Ring Attention row: 128-row KV
 * tiles).  The pages give no formula for the attention itself, so the oracle
 * follows the plain definition of scaled-dot-product attention with an
 * optional causal mask over global positions, plus the per-row log-sum-exp:
 *
 *   A_i   = [0, S)            (non-causal)   or   [0, i]   (causal)
 *         or {j : pos(j) <= pos(i)}   (causal over load-balanced shards, causal == 2)
 *   s_ij  = scale * sum_c Q[b,hq,i,c] * K[b,kv,j,c]      for j in A_i
 *   m_i   = max_j s_ij
 *   l_i   = sum_j exp(s_ij - m_i)
 *   O_i   = sum_j exp(s_ij - m_i) * V[b,kv,j,:] / l_i
 *   LSE_i = m_i + ln l_i                                  (natural log)
 *
 * with kv = floor(hq / (Hq / Hkv)) (consecutive query heads share a KV head).
 *
 * Load-balanced shards (causal == 2; not on the pages, the usual balancing of
 * causal ring attention): the S axis is stored shard by shard, L = S/P rows
 * each, and shard r holds the half-chunks r and 2P-1-r of the sequence (L/2
 * positions each), in that order.  pos(i) is the global position of stored
 * row i; the mask compares positions, and outputs stay in stored order.
 * Inputs are bf16 bit patterns widened exactly to fp64; every step is fp64.
 *
 * Two modes:
 *   oracle_attn_fwd          the definition above, two passes per row;
 *   oracle_attn_fwd_chunked  the same rows computed the way a ring consumes
 *                            them: the key range split into P chunks of
 *                            L = S/P keys, visited in ring order
 *                            j = (r - t) mod P for t = 0..P-1 (r = shard of
 *                            row i), each chunk's partial (O_t, lse_t) formed
 *                            in fp64, and the partials merged exactly by
 *                            lse = M + ln sum_t exp(lse_t - M),
 *                            O = sum_t exp(lse_t - lse) * O_t.
 *                            Used only to check the merge identity.
 *
 * Parity pins live in tests/test_oracle_pins.py (Decimal brute force, closed
 * forms, invariants).
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

static inline double bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* sum_c a[c]*b[c] in fp64 (four partial sums; the association differs from a
 * left-to-right sum only at the 1e-16 relative level). */
static inline double dot_bf16(const uint16_t *a, const uint16_t *b, int d) {
  double s0 = 0, s1 = 0, s2 = 0, s3 = 0;
  int c = 0;
  for (; c + 4 <= d; c += 4) {
    s0 += bf16_to_f64(a[c + 0]) * bf16_to_f64(b[c + 0]);
    s1 += bf16_to_f64(a[c + 1]) * bf16_to_f64(b[c + 1]);
    s2 += bf16_to_f64(a[c + 2]) * bf16_to_f64(b[c + 2]);
    s3 += bf16_to_f64(a[c + 3]) * bf16_to_f64(b[c + 3]);
  }
  for (; c < d; ++c) s0 += bf16_to_f64(a[c]) * bf16_to_f64(b[c]);
  return (s0 + s1) + (s2 + s3);
}

typedef struct {
  const oracle_shape *sh;
  const uint16_t *q, *k, *v;
  const int64_t *rows;
  int64_t lo, n_rows, stride; /* rows lo, lo+stride, ... < n_rows */
  const int *perm; /* chunked mode: visiting order, or NULL for ring order */
  int chunked;
  double *o, *lse;
  int err;
} job_t;

/* Key range A_i of row i: [0, S) or [0, i]. */
static inline int64_t allowed_end(const oracle_shape *sh, int64_t i) {
  return sh->causal ? i + 1 : sh->S;
}

/* Global position of stored row i: i itself, or under load-balanced shards the
 * position inside half-chunk r (rows 0 .. L/2-1 of shard r) or 2P-1-r (the rest). */
static inline int64_t position(const oracle_shape *sh, int64_t i) {
  if (sh->causal != 2) return i;
  const int64_t L = sh->S / sh->P, h = L / 2;
  const int64_t r = i / L, loc = i % L;
  return loc < h ? r * h + loc : (2 * (int64_t)sh->P - 1 - r) * h + (loc - h);
}

/* Direct definition for one row, keys [k0, k1) only (under load-balanced shards,
 * only those at positions <= qpos).  Writes the normalised output and returns the
 * log-sum-exp of those keys (-inf if there are none). */
static double attend_range(const oracle_shape *sh, const uint16_t *qrow, const uint16_t *kbase,
                           const uint16_t *vbase, int64_t k0, int64_t k1, int64_t qpos, double *s_buf,
                           double *out) {
  const int d = sh->d;
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  if (k1 <= k0) return -INFINITY;
  /* pass 1: scores and their maximum */
  double m = -INFINITY;
  for (int64_t j = k0; j < k1; ++j) {
    if (sh->causal == 2 && position(sh, j) > qpos) { /* masked key */
      s_buf[j - k0] = -INFINITY;
      continue;
    }
    double s = sh->scale * dot_bf16(qrow, kbase + j * d, d);
    s_buf[j - k0] = s;
    if (s > m) m = s;
  }
  if (m == -INFINITY) return -INFINITY; /* every key masked */
  /* pass 2: exponentials, their sum and the weighted sum of V rows */
  double l = 0.0;
  for (int64_t j = k0; j < k1; ++j) {
    if (s_buf[j - k0] == -INFINITY) continue;
    double p = exp(s_buf[j - k0] - m);
    l += p;
    const uint16_t *vr = vbase + j * d;
    for (int c = 0; c < d; ++c) out[c] += p * bf16_to_f64(vr[c]);
  }
  for (int c = 0; c < d; ++c) out[c] /= l;
  return m + log(l);
}

static void *worker(void *arg) {
  job_t *jb = (job_t *)arg;
  const oracle_shape *sh = jb->sh;
  const int d = sh->d;
  const int g = sh->Hq / sh->Hkv;
  const int64_t S = sh->S;
  const int64_t L = S / sh->P;
  double *s_buf = (double *)malloc(sizeof(double) * (size_t)S);
  double *part_o = jb->chunked ? (double *)malloc(sizeof(double) * (size_t)d * sh->P) : NULL;
  double *part_lse = jb->chunked ? (double *)malloc(sizeof(double) * sh->P) : NULL;
  if (!s_buf || (jb->chunked && (!part_o || !part_lse))) {
    jb->err = 1;
    free(s_buf); free(part_o); free(part_lse);
    return NULL;
  }
  for (int64_t n = jb->lo; n < jb->n_rows; n += jb->stride) {
    const int64_t id = jb->rows ? jb->rows[n] : n;
    const int64_t i = id % S;
    const int64_t bh = id / S;
    const int64_t b = bh / sh->Hq, hq = bh % sh->Hq;
    const int64_t kv = hq / g;
    const uint16_t *qrow = jb->q + id * d;
    const uint16_t *kb = jb->k + (b * sh->Hkv + kv) * S * d;
    const uint16_t *vb = jb->v + (b * sh->Hkv + kv) * S * d;
    double *orow = jb->o + n * d;
    const int64_t kend = sh->causal == 2 ? S : allowed_end(sh, i);
    const int64_t qpos = position(sh, i);
    if (!jb->chunked) {
      jb->lse[n] = attend_range(sh, qrow, kb, vb, 0, kend, qpos, s_buf, orow);
      continue;
    }
    /* ring order: shard r = i / L consumes chunk (r - t) mod P at step t */
    const int64_t r = i / L;
    int np = 0;
    for (int t = 0; t < sh->P; ++t) {
      int64_t j = jb->perm ? jb->perm[t] : ((r - t) % sh->P + sh->P) % sh->P;
      int64_t k0 = j * L, k1 = (j + 1) * L;
      if (k1 > kend) k1 = kend; /* causal: keys beyond i are masked */
      if (k1 <= k0) continue;   /* fully masked chunk: skipped */
      part_lse[np] = attend_range(sh, qrow, kb, vb, k0, k1, qpos, s_buf, part_o + (size_t)np * d);
      if (part_lse[np] == -INFINITY) continue; /* every key of the chunk masked: skipped */
      ++np;
    }
    if (np == 0) {
      for (int c = 0; c < d; ++c) orow[c] = 0.0;
      jb->lse[n] = -INFINITY;
      continue;
    }
    double M = -INFINITY;
    for (int t = 0; t < np; ++t)
      if (part_lse[t] > M) M = part_lse[t];
    double sum = 0.0;
    for (int t = 0; t < np; ++t) sum += exp(part_lse[t] - M);
    const double lse = M + log(sum);
    for (int c = 0; c < d; ++c) orow[c] = 0.0;
    for (int t = 0; t < np; ++t) {
      const double w = exp(part_lse[t] - lse);
      for (int c = 0; c < d; ++c) orow[c] += w * part_o[(size_t)t * d + c];
    }
    jb->lse[n] = lse;
  }
  free(s_buf); free(part_o); free(part_lse);
  return NULL;
}

static int check_shape(const oracle_shape *sh) {
  if (!sh) return 1;
  if (sh->B < 1 || sh->Hq < 1 || sh->Hkv < 1 || sh->S < 1 || sh->P < 1 || sh->d < 1) return 1;
  if (sh->Hq % sh->Hkv) return 1;
  if (sh->S % sh->P) return 1;
  if (sh->causal < 0 || sh->causal > 2) return 1;
  if (sh->causal == 2 && (sh->S / sh->P) % 2) return 1; /* shards split in two halves */
  return 0;
}

static int run(const oracle_shape *sh, const uint16_t *q, const uint16_t *k, const uint16_t *v,
               const int64_t *rows, int64_t n_rows, const int *perm, int chunked, double *o, double *lse,
               int n_threads) {
  if (check_shape(sh) || !q || !k || !v || !o || !lse || n_rows < 0) return 1;
  const int64_t total = (int64_t)sh->B * sh->Hq * sh->S;
  if (rows) {
    for (int64_t n = 0; n < n_rows; ++n)
      if (rows[n] < 0 || rows[n] >= total) return 1;
  } else if (n_rows != total) {
    return 1;
  }
  if (perm) {
    /* must be a permutation of 0..P-1 */
    char *seen = (char *)calloc((size_t)sh->P, 1);
    if (!seen) return 1;
    for (int t = 0; t < sh->P; ++t) {
      if (perm[t] < 0 || perm[t] >= sh->P || seen[perm[t]]) { free(seen); return 1; }
      seen[perm[t]] = 1;
    }
    free(seen);
  }
  if (n_rows == 0) return 0;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 512) n_threads = 512;
  if (n_threads > n_rows) n_threads = (int)n_rows;
  job_t *jobs = (job_t *)calloc((size_t)n_threads, sizeof(job_t));
  pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
  char *started = (char *)calloc((size_t)n_threads, 1);
  if (!jobs || !th || !started) { free(jobs); free(th); free(started); return 1; }
  /* interleaved rows, so that causal rows of different lengths spread evenly */
  for (int t = 0; t < n_threads; ++t)
    jobs[t] = (job_t){sh, q, k, v, rows, t, n_rows, n_threads, perm, chunked, o, lse, 0};
  for (int t = 1; t < n_threads; ++t)
    started[t] = pthread_create(&th[t], NULL, worker, &jobs[t]) == 0;
  worker(&jobs[0]);
  for (int t = 1; t < n_threads; ++t) {
    if (started[t]) pthread_join(th[t], NULL);
    else worker(&jobs[t]);
  }
  int err = 0;
  for (int t = 0; t < n_threads; ++t) err |= jobs[t].err;
  free(jobs); free(th); free(started);
  return err;
}

int oracle_attn_fwd(const oracle_shape *sh, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    const int64_t *rows, int64_t n_rows, double *o, double *lse, int n_threads) {
  return run(sh, q, k, v, rows, n_rows, NULL, 0, o, lse, n_threads);
}

int oracle_attn_fwd_chunked(const oracle_shape *sh, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const int64_t *rows, int64_t n_rows, const int *perm, double *o, double *lse,
                            int n_threads) {
  return run(sh, q, k, v, rows, n_rows, perm, 1, o, lse, n_threads);
}
