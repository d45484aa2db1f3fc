/*
 * fp64 CPU oracle for the Ring Attention forward step (test infrastructure).
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
 * this library.  It is independent of the GPU library: no shared code,
 * headers, tables or constants.
 */
#ifndef RING_ATTN_ORACLE_H
#define RING_ATTN_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* causal: 0 none; 1 mask over contiguous shards (stored row i = position i);
 * 2 mask over load-balanced shards (shard r holds half-chunks r and 2P-1-r). */
typedef struct {
  int B, Hq, Hkv, S, P, d, causal;
  double scale;
} oracle_shape;

/* Plain definition, fp64.  q: [B][Hq][S][d], k,v: [B][Hkv][S][d], bf16 bit
 * patterns.  rows: flat ids (b*Hq + hq)*S + i, or NULL for all rows in order
 * (then n_rows must equal B*Hq*S).  o: [n_rows][d], lse: [n_rows].
 * Returns 0 on success, nonzero on a bad argument or allocation failure. */
int oracle_attn_fwd(const oracle_shape *sh, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    const int64_t *rows, int64_t n_rows, double *o, double *lse, int n_threads);

/* Ring-chunked evaluation with the exact log-sum-exp merge.  perm: NULL for
 * ring order j = (r - t) mod P, else a permutation of 0..P-1 giving the chunk
 * visiting order for every row. */
int oracle_attn_fwd_chunked(const oracle_shape *sh, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const int64_t *rows, int64_t n_rows, const int *perm, double *o, double *lse,
                            int n_threads);

#ifdef __cplusplus
}
#endif
#endif
