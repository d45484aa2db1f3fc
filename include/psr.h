/*
 * persistent_sm_ring_gb300 -- Ring Attention forward on one GB300 (sm_103a).
 *
 * C ABI of libpsr.so.  Plain pointers and sizes only; every call returns a
 * status code (PSR_OK = 0) and never throws or exits.
 *
 * The operation (mKernel pages: arxivdaily abstract; dataforcee and chathome
 * "five fused kernels" tables, Ring Attention row; pwwt.cn analysis §2.6,
 * Table 3, Ring Attention row): sequence-parallel attention in which P ring
 * ranks each hold one shard of L = S/P query rows; at ring step t the rank of
 * shard r consumes KV chunk (r - t) mod P while the next chunk is moved into
 * its receive buffer, and the per-chunk partial results are merged exactly
 * through the running max and log-sum-exp.  Here the P ranks are P shards in
 * one GPU's HBM: "staging" CTAs copy each chunk into a ring slot (three per
 * group of items that read the same chunks) with TMA and publish a readiness
 * flag (pwwt.cn §2.2 Figure 2 readiness flag; §2.5: the flag names the
 * completed payload), "compute" CTAs run the FlashAttention pass on tcgen05
 * tensor cores, and an on-GPU controller re-splits CTAs between the two roles
 * with the pwwt.cn §2.4 rule
 *     n_s* = N * (R_s*C_s) / (R_p*C_p + R_s*C_s).
 * Without a causal mask every compute item takes the same time, and the
 * adaptive target is capped at the largest split that keeps the compute
 * waves ceil(items / compute CTAs) of the split the staging work needs.
 *
 * Result: O = softmax(scale * Q K^T [+ causal mask over global positions]) V,
 * rounded to bf16, and LSE = natural-log log-sum-exp of the scaled scores per
 * query row, fp32.  Query head hq reads KV head hq / (Hq/Hkv).
 */
#ifndef PSR_H
#define PSR_H
#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PSR_API __attribute__((visibility("default")))
#else
#define PSR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------------------------------- */
#define PSR_OK 0
#define PSR_ERR_ARG 1         /* null pointer, bad value, workspace too small */
#define PSR_ERR_UNSUPPORTED 2 /* shape outside the supported set, or not an sm_103 device */
#define PSR_ERR_CUDA 3        /* a CUDA runtime call failed (launch, memset, copy) */
#define PSR_ERR_TIMEOUT 4     /* a bounded device wait expired (reported by psr_get_stats) */

/* ---- partition modes --------------------------------------------------------------------------- */
#define PSR_STATIC 0   /* n_staging CTAs stage for the whole launch, the rest compute */
#define PSR_ADAPTIVE 1 /* the on-GPU controller re-splits CTAs at task boundaries */

/* Fault-injection codes (psr_partition.fault); 0 in normal use.  They act on
 * the host-visible protocol only and never fault the GPU: a dropped flag makes
 * the consumers' bounded waits expire and the launch report PSR_ERR_TIMEOUT. */
#define PSR_FAULT_NONE 0
#define PSR_FAULT_DROP_FIRST_FLAG 1 /* the first staged chunk never publishes its readiness flag */
#define PSR_FAULT_SLOW_STAGING 2    /* every staging task sleeps ~20 us before copying */

/* Causal layouts (psr_shape.causal).  With PSR_CAUSAL_BALANCED, shard r (rows r*L .. r*L+L-1
 * of the S axis, L = S/P) holds two halves of the sequence: its rows i < L/2 are global
 * position r*L/2 + i and its rows i >= L/2 are global position (2P-1-r)*L/2 + (i - L/2).  Every
 * shard then does the same causal work at every ring step (with contiguous shards shard r does
 * r+1 of the P steps).  The caller stores Q, K, V (and receives O, LSE) in that shard order;
 * the mask is over the global positions.  This layout is not on the mKernel pages: it is the
 * usual load balancing of causal ring attention.  Requires L a multiple of 512. */
#define PSR_CAUSAL 1
#define PSR_CAUSAL_BALANCED 2

typedef struct {
  int B;        /* batch */
  int Hq;       /* query heads */
  int Hkv;      /* key/value heads; Hq % Hkv == 0 */
  int S;        /* global sequence length */
  int P;        /* ring size (number of shards); S % P == 0 */
  int d;        /* head dim: 64 or 128 */
  int causal;   /* 0: none; PSR_CAUSAL (1): mask k_pos > q_pos over global positions, shard r
                   holding positions r*L .. r*L+L-1; PSR_CAUSAL_BALANCED (2): the same mask over
                   load-balanced shards (see below) */
  float scale;  /* <= 0 selects 1/sqrt(d) */
} psr_shape;

typedef struct {
  int mode;       /* PSR_STATIC or PSR_ADAPTIVE */
  int n_staging;  /* static: staging CTA count; adaptive: initial count (<= 0: automatic) */
  int n_min;      /* adaptive clamp, lower (<= 0: 1) */
  int n_max;      /* adaptive clamp, upper (<= 0: automatic) */
  int fault;      /* PSR_FAULT_* */
  int timeout_ms; /* bound on every device wait (<= 0: 2000 ms); in the GEMM entries the waits
                     inside the tile pipeline, which only follow an upstream wait, give up after
                     4 x timeout_ms, so that the upstream wait reports the cause */
} psr_partition;

typedef struct {
  int status;                     /* PSR_OK or PSR_ERR_TIMEOUT */
  int error_site;                 /* which wait gave up (0 = none) */
  int n_cta;                      /* persistent CTAs launched */
  int n_s_initial, n_s_final;     /* controller target at start / end */
  int n_s_min, n_s_max;           /* range of the target over the launch */
  int traj_len;                   /* entries in the target trajectory log */
  unsigned long long staging_cycles, compute_cycles; /* SM cycles spent inside tasks */
  unsigned long long staging_tasks, compute_items, compute_tiles;
  unsigned long long staging_bytes;                  /* bytes written into ring slots */
  unsigned long long role_switches;
  unsigned long long idle_polls;                     /* task-boundary polls that found no work */
  /* Per-role cycle counters, filled only by a library built with PSR_TRACE=1
   * (zero otherwise): softmax threads waiting for S / computing (summed over
   * warps, lane 0 each), the two MMA-issuing threads in their issue sections /
   * the part of that spent waiting for K,V tiles, and the TMA producer waiting
   * for free stages / for readiness flags. */
  unsigned long long trace_softmax_wait, trace_softmax_busy;
  unsigned long long trace_mma_issue, trace_mma_wait_kv;
  unsigned long long trace_producer_wait_empty, trace_producer_wait_flag;
} psr_stats;

/* Bytes of device workspace psr_ring_attn_fwd needs for this shape: the
 * control block, readiness flags, consumption counters, the staging ready
 * queue, the trajectory log and the three ring slots for K and V
 * (3 x [n_groups][L][d] bf16 each).  Returns 0 for an invalid shape. */
PSR_API size_t psr_workspace_bytes(const psr_shape* shape);

/* Ring Attention forward.
 *   q:  device, bf16, [B][Hq][S][d] contiguous      (read)
 *   k,v: device, bf16, [B][Hkv][S][d] contiguous    (read)
 *   o:  device, bf16, [B][Hq][S][d] contiguous      (written)
 *   lse: device, fp32, [B][Hq][S]                   (written)
 *   workspace: device, >= psr_workspace_bytes(shape) bytes, 256-byte aligned,
 *              owned by the caller; must not be used by another launch in flight.
 *   part: partition policy (NULL = adaptive, automatic).
 *   stream: a cudaStream_t (NULL = legacy default stream).
 * Asynchronous: enqueues a flag reset and one persistent launch on `stream`
 * and returns.  The library allocates no device memory.  A device-side
 * timeout is reported by psr_get_stats, not here.
 * Supported: d in {64, 128}; S % P == 0; L = S/P a multiple of 256 (of 512 with
 * PSR_CAUSAL_BALANCED); Hq % Hkv == 0; sm_103 device.  Otherwise PSR_ERR_UNSUPPORTED. */
PSR_API int psr_ring_attn_fwd(const psr_shape* shape, const void* q, const void* k, const void* v, void* o, float* lse,
                      void* workspace, size_t workspace_bytes, const psr_partition* part, void* stream);

/* Same operation with HOST buffers: copies q, k, v (host; pinned for overlap)
 * to the caller's device buffers dq, dk, dv (same layouts and sizes as the
 * device entry's q, k, v, o, lse), runs the attention, copies O and LSE back
 * to o_host / lse_host, and returns when they are there.  One persistent
 * launch covers the whole shape; the inputs are uploaded unit by unit (a unit
 * is one batch when B > 1, else one KV head with its query heads) on an
 * internal stream that marks each unit ready in the workspace, the launch
 * dispenses its items unit by unit and each item waits (bounded by
 * part->timeout_ms) for its unit, and a second internal stream copies each
 * unit's O and LSE out as soon as all of its items are done.  So only the first
 * unit's upload and the last unit's download are exposed.  The workspace is
 * psr_workspace_bytes(shape); psr_get_stats afterwards describes the launch.
 * Returns the first failing status, or PSR_ERR_TIMEOUT if the launch reported
 * a device timeout (for instance an upload slower than the wait bound). */
PSR_API int psr_ring_attn_fwd_host(const psr_shape* shape, const void* q_host, const void* k_host, const void* v_host,
                           void* o_host, float* lse_host, void* dq, void* dk, void* dv, void* d_o, float* d_lse,
                           void* workspace, size_t workspace_bytes, const psr_partition* part, void* stream);

/* Synchronises `stream`, reads the control block of the last launch that used
 * `workspace` and fills *out.  Returns out->status (PSR_OK or
 * PSR_ERR_TIMEOUT), or PSR_ERR_ARG / PSR_ERR_CUDA. */
PSR_API int psr_get_stats(const void* workspace, psr_stats* out, void* stream);

/* Copies up to max_entries (time_us, n_s) pairs of the controller's target
 * trajectory (device workspace -> host); synchronises `stream`.  Returns the
 * number of pairs written, or a negative status. */
PSR_API int psr_get_trajectory(const void* workspace, uint32_t* out_pairs, int max_entries, void* stream);

/* The controller rule evaluated on the host, as the device evaluates it:
 * n = round(n_cta * R_s*C_s / (R_p*C_p + R_s*C_s)), clamped to
 * [max(n_min,1), min(n_max, n_cta-1)] while both roles have work; 0 when
 * R_s == 0; n_max when R_p == 0 and R_s > 0.  For tests and tooling. */
PSR_API int psr_controller_target(int n_cta, double R_s, double C_s, double R_p, double C_p, int n_min, int n_max);

/* Allocation-free variant of psr_ring_attn_fwd.  No counterpart in the
 * mKernel pages: it exists for callers that must not call cudaMalloc (a host
 * framework whose pool owns the device memory, a plug-in that may not
 * allocate, a latency-critical path that cannot afford cudaMalloc's implicit
 * synchronisation).  Same arguments and layouts as psr_ring_attn_fwd, minus the
 * workspace: the scratch is a file-scope device array of
 * PSR_NOALLOC_SCRATCH_BYTES held by every GPU that loads the library until the
 * process exits.  The library allocates nothing (no cudaMalloc, cudaFree or
 * allocating library call).
 *   - Checks in the order of psr_ring_attn_fwd, with the same status codes:
 *     null or misaligned q, k, v, o, lse -> PSR_ERR_ARG; the device; the shape
 *     (PSR_ERR_ARG / PSR_ERR_UNSUPPORTED).  Only then, a supported shape whose
 *     psr_workspace_bytes(shape) exceeds PSR_NOALLOC_SCRATCH_BYTES ->
 *     PSR_ERR_UNSUPPORTED.
 *   - The first call on a device looks up the array's device address with that
 *     device current (and looks it up again after the device's context was
 *     reset); make that first call before any stream capture.
 *   - All calls on a device share the array and each call clears its control
 *     words first; calls whose launches overlap on the GPU race on it, so order
 *     them (one stream, or events).
 *   - A device-side timeout is not reported here: read it with
 *     psr_noalloc_get_stats after the call (before the next no-alloc call). */
#define PSR_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
PSR_API int psr_ring_attn_fwd_noalloc(const psr_shape* shape, const void* q, const void* k, const void* v, void* o,
                                      float* lse, const psr_partition* part, void* stream);

/* psr_get_stats for the allocation-free entry: synchronises `stream`, reads the
 * control block of the last psr_ring_attn_fwd_noalloc launch on the current
 * device from the fixed scratch and fills *out.  Returns out->status (PSR_OK or
 * PSR_ERR_TIMEOUT), or PSR_ERR_ARG / PSR_ERR_CUDA.  Allocates nothing. */
PSR_API int psr_noalloc_get_stats(psr_stats* out, void* stream);

/* Human-readable name of a status code (static string). */
PSR_API const char* psr_status_string(int status);

/* Number of persistent CTAs a launch on the current device uses (one per SM),
 * or a negative status. */
PSR_API int psr_num_ctas(void);

/* ---- Ring Attention backward ------------------------------------------------------------------
 * The gradient of psr_ring_attn_fwd (the mKernel pages describe only the
 * forward; the backward follows the same ring and reuses the forward's LSE).
 * With P_ij = exp(scale q_i.k_j - LSE_i) over the allowed keys, D_i = dO_i.O_i,
 * dP_ij = dO_i.v_j and dS_ij = P_ij (dP_ij - D_i):
 *     dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j
 * (dK, dV summed over the query heads that share the KV head).  In the ring
 * each KV chunk travels with its dK/dV partial sums while the queries stay;
 * on one GPU a first persistent kernel gives each task one 128-row K/V tile
 * whose dK/dV accumulators stay in tensor memory while it visits the query
 * shards in ring order, and a second, query-stationary one gives each task one
 * 128-row query tile whose dQ accumulator stays in tensor memory while it
 * visits the K/V tiles (it recomputes S and dP; no atomics).  All matrix
 * products run on tcgen05 with bf16 operands (P and dS rounded to bf16) and
 * fp32 accumulation. */

/* Bytes of device workspace psr_ring_attn_bwd needs: the control block (the
 * shared prefix, read by psr_get_stats), D = rowsum(dO * O) and -LSE*log2(e)
 * ([B][Hq][S] fp32 each).  Returns 0 for an invalid or unsupported shape. */
PSR_API size_t psr_ring_attn_bwd_workspace_bytes(const psr_shape* shape);

/* Ring Attention backward.
 *   q, o, dout: device, bf16, [B][Hq][S][d]          (read; o = the forward output)
 *   k, v:       device, bf16, [B][Hkv][S][d]         (read)
 *   lse:        device, fp32, [B][Hq][S]             (read; the forward's natural-log LSE)
 *   dq:         device, bf16, [B][Hq][S][d]          (written)
 *   dk, dv:     device, bf16, [B][Hkv][S][d]         (written)
 *   workspace:  device, >= psr_ring_attn_bwd_workspace_bytes(shape), 256-byte aligned.
 *   timeout_ms: bound on every device wait (<= 0: 2000 ms); stream: a cudaStream_t.
 * All pointers 16-byte aligned.  Asynchronous: enqueues a workspace reset, the
 * D kernel and the two persistent launches (dK/dV, then dQ) on `stream`; a device
 * timeout is reported by psr_get_stats.  Supported: d in {64, 128}; causal 0, 1 or
 * PSR_CAUSAL_BALANCED; L = S/P a multiple of 128 (of 256 with PSR_CAUSAL_BALANCED);
 * Hq % Hkv == 0; sm_103 device. */
PSR_API int psr_ring_attn_bwd(const psr_shape* shape, const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv, void* workspace,
                              size_t workspace_bytes, int timeout_ms, void* stream);

/* ---- AllGather + GEMM ------------------------------------------------------------------------ */
/* The pages' second fused pattern (dataforcee / chathome "five fused kernels"
 * table, AllGather+GEMM row; pwwt.cn analysis §2.6: 128-row chunks, local
 * inputs first): every rank holds a row shard of A; while the ranks gather
 * the peers' shards, the local GEMM consumes A tiles as they arrive.  On one
 * GPU the P ranks are emulated in HBM: rank r owns rows [r*M/P, (r+1)*M/P) of
 * A and the weight slice W_r, and produces
 *     C_r = gather(A) @ W_r^T      (fp32 accumulation, bf16 result, RNE),
 * the gathered A being the shards concatenated in rank order.  Staging CTAs
 * copy peer shards into each rank's gather buffer in the workspace (pieces of
 * >= 512 KiB, each published with a readiness flag); compute CTAs work in
 * pairs (clusters of two SMs), each pair producing one 256 x 512 tile of one
 * rank with tcgen05 cta_group::2 MMAs (a rank's last tile is 256 x 256 when Ns
 * is an odd multiple of 256), reading the rank's own shard in place and a
 * peer's rows after acquiring their flags; the same controller as the Ring
 * Attention splits the pairs between the two roles (a target of n staging CTAs
 * gives ceil(n/2) staging pairs). */
typedef struct {
  int M;   /* rows of the gathered A; M/P must be a multiple of 256 */
  int K;   /* contraction; a multiple of 128 */
  int Ns;  /* output columns per rank; a multiple of 256 */
  int P;   /* ranks */
} psr_ag_shape;

/* Bytes of device workspace psr_ag_gemm needs: the control block and
 * trajectory log (the same layout as psr_ring_attn_fwd's, so psr_get_stats and
 * psr_get_trajectory read it), the readiness flags [P][P][pieces] and the P
 * gather buffers ([P][M][K] bf16).  Returns 0 for an invalid shape. */
PSR_API size_t psr_ag_gemm_workspace_bytes(const psr_ag_shape* shape);

/* AllGather + GEMM.
 *   a: device, bf16, [M][K] contiguous (rank j's shard = rows j*M/P ..)   (read)
 *   w: device, bf16, [P][Ns][K] contiguous (rank r's weight, K-major)     (read)
 *   c: device, bf16, [P][M][Ns] contiguous (rank r's output)              (written)
 *   workspace: device, >= psr_ag_gemm_workspace_bytes(shape), 256-byte aligned, caller-owned.
 *   part: partition policy (NULL = adaptive); stream: a cudaStream_t (NULL = default).
 *   A static partition takes 1 <= n_staging <= (CTAs launched) - 2, so that at
 *   least one pair computes; the launch is one CTA per SM in whole pairs.
 * Asynchronous (one flag reset and one persistent launch of clusters of two on
 * `stream`); a device timeout is reported by psr_get_stats.  PSR_ERR_UNSUPPORTED
 * for shapes outside the constraints above or a device other than sm_103. */
PSR_API int psr_ag_gemm(const psr_ag_shape* shape, const void* a, const void* w, void* c, void* workspace,
                        size_t workspace_bytes, const psr_partition* part, void* stream);

/* ---- GEMM + ReduceScatter ---------------------------------------------------------------------
 * The mKernel pages' GEMM+ReduceScatter kernel (dataforcee and chathome "five
 * fused kernels" tables, GEMM + ReduceScatter row; pwwt.cn analysis §2.6
 * Table 3: tensor parallel, compute feeds communication): rank r holds its
 * K-shard A_r of the activations and W_r of the weights and computes the
 * partial product A_r @ W_r^T; the ranks reduce-scatter the partials, so rank q
 * receives rows [q*M/P, (q+1)*M/P) of
 *     out = sum_r A_r @ W_r^T      (fp32 partials summed in rank order, bf16 result, RNE),
 * each output tile being reduced and forwarded as soon as its partials exist.
 * On one GPU the P ranks are emulated in HBM: compute pairs (clusters of two
 * SMs) each produce one 256 x 512 fp32 partial tile of one rank (256 x 256 for
 * a rank's last tile when N is an odd multiple of 256) with tcgen05
 * cta_group::2 MMAs into the workspace, and the completion of an output tile's
 * P partials enqueues it; reduce CTAs (the communication role) stream the P
 * partials through shared memory with TMA bulk copies and write the owner's
 * rows.  The same controller splits the pairs between the roles (a target of n
 * reduce CTAs gives ceil(n/2) reduce pairs); as compute feeds the reductions,
 * the adaptive launch starts with no reduce CTA (part->n_staging > 0
 * overrides). */
typedef struct {
  int M;   /* output rows (tokens); M/P must be a multiple of 256 */
  int N;   /* output columns; a multiple of 256 */
  int Ks;  /* contraction per rank (K/P); a multiple of 64 */
  int P;   /* ranks, 1..64 */
} psr_rs_shape;

/* Bytes of device workspace psr_gemm_rs needs: the control block and
 * trajectory log (the same layout as the other entries, so psr_get_stats and
 * psr_get_trajectory read it), per-tile arrival counters and the ready queue,
 * and the fp32 partial tiles ([P][M][N'] fp32, N' = N rounded up to a
 * multiple of 512).  Returns 0 for an invalid shape. */
PSR_API size_t psr_gemm_rs_workspace_bytes(const psr_rs_shape* shape);

/* GEMM + ReduceScatter.
 *   a:   device, bf16, [P][M][Ks] contiguous (rank r's activations, K-major)  (read)
 *   w:   device, bf16, [P][N][Ks] contiguous (rank r's weights, K-major)      (read)
 *   out: device, bf16, [M][N] contiguous (rows q*M/P .. belong to rank q)     (written)
 *   workspace: device, >= psr_gemm_rs_workspace_bytes(shape), 256-byte aligned, caller-owned.
 *   part: partition policy (NULL = adaptive; static needs 1 <= n_staging <= (CTAs launched) - 2
 *         reduce CTAs, so that at least one pair computes).
 *   stream: a cudaStream_t (NULL = default).
 * Asynchronous (one counter reset and one persistent launch of clusters of two
 * on `stream`); a device timeout is reported by psr_get_stats (staging_tasks counts the tile
 * reductions, staging_bytes the partial bytes they read).  PSR_ERR_UNSUPPORTED
 * for shapes outside the constraints above or a device other than sm_103. */
PSR_API int psr_gemm_rs(const psr_rs_shape* shape, const void* a, const void* w, void* out, void* workspace,
                        size_t workspace_bytes, const psr_partition* part, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PSR_H */
