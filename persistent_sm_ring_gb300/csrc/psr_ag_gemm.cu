// AllGather + GEMM as one persistent kernel on sm_103a.
//
// The mKernel pages' AllGather+GEMM kernel (dataforcee / chathome "five fused kernels"
// table, AllGather+GEMM row; pwwt.cn analysis §2.6, 128-row chunks, local inputs first):
// every rank holds a row shard of A; while the ranks gather the peers' shards, the local
// GEMM consumes A tiles as soon as they arrive.  On one GPU the P ranks are emulated in
// HBM: rank r owns rows [r*Ms, (r+1)*Ms) of A (Ms = M/P) and the weight slice W_r
// ([Ns][K], K-major), and produces C_r = gather(A) @ W_r^T.
//
//  * the CTAs work in pairs (clusters of two); a pair takes either role;
//  * a staging pair's two CTAs each copy a piece of a peer shard's rows (>= 512 KiB) into rank
//    r's gather buffer (the same row positions) with TMA bulk copies through shared memory,
//    and publish a per-piece readiness flag with a gpu-scope release once the stores are
//    complete;
//  * a compute pair produces one 256 x 512 output tile of one rank per task (the pair tile of
//    psr_gemm_tile.cuh with two accumulator halves: each CTA 128 rows x 512 columns, tcgen05
//    cta_group::2); the rank's own shard is read in place, a peer's only after each CTA has
//    acquired the piece flags that cover its 128 rows.  When Ns is an odd multiple of 256 a
//    rank's last tile is half wide: its second half is computed and not stored;
//  * each rank's tasks run in availability order: its local tiles first, then the tiles of
//    shard r+1, r+2, ... (the order in which staging delivers them); ranks run one after
//    another, so that a rank's weight slice is read from HBM once;
//  * the shared controller re-splits the pairs between the roles with the pages' rule (a
//    target of n staging CTAs gives ceil(n/2) staging pairs).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/psr.h"
#include "psr_control.cuh"
#include "psr_device.cuh"
#include "psr_gemm_tile.cuh"
#include "psr_schedule.h"

namespace psr {
namespace ag {

using namespace gemm;  // the pair tile: stages, MMA issue, accumulator read-back
constexpr int kCopyUnit = 32768;  // staging copy unit
constexpr int kNCopyBuf = kStageArea / kCopyUnit;
constexpr int kPieceMinBytes = 512 * 1024;
static_assert(kNCopyBuf <= 16, "staging barriers");

enum : uint32_t { SITE_FLAG = 1, SITE_STAGE_LOAD = 8 };

struct Geo {
  int M, K, Ns, P, Ms;
  int n_mb;          // 256-row blocks per shard
  int n_nb;          // 512-column blocks per rank (the last one half wide when Ns % 512 = 256)
  int piece_rows;    // rows per staging piece (a multiple of 128 dividing Ms)
  int n_pieces;      // pieces per shard
  long long n_items;   // compute tasks: P ranks x P shards x n_mb x n_nb
  long long n_stage;   // staging pieces: P ranks x (P-1) peers x n_pieces
};

struct Params {
  Geo g;
  const uint16_t* a;
  uint16_t* gbuf;      // [P][M][K]: rank r's gathered copy of A (peer rows only are written)
  uint16_t* c;         // [P][M][Ns]
  uint32_t* flags;     // [P][P][n_pieces]
  Ctrl* ctrl;
  uint32_t* traj;
  unsigned long long timeout_ns;
  unsigned long long n_tiles_total, n_stage_total;
  int mode, n_s_init, n_min, n_max, fault;
  uint32_t n_wave_items;  // no wave cap here (0): the tasks' waves are many and short
  int n_wave_cap;
  float c_s0, c_p0;
  float update_headroom;
};


// task index -> (rank, shard, m-block, n-block): rank by rank, shards in availability order
// jj = 0, 1, .. (shard = (rank + jj) mod P, the local one first), then W tile by W tile with the
// m-blocks that share it.  The W tiles run forward through even shards and backward through odd
// ones, so that a shard starts on the W tiles its predecessor used last, which are still in L2
// (a rank's weight slice is larger than the share of L2 it keeps).
struct Item {
  int r, j, mb, nb;
};
__device__ __host__ inline Item item_of(const Geo& g, long long idx) {
  Item it;
  it.mb = (int)(idx % g.n_mb);
  idx /= g.n_mb;
  const int nbi = (int)(idx % g.n_nb);
  idx /= g.n_nb;
  const int jj = (int)(idx % g.P);
  it.r = (int)(idx / g.P);
  it.j = (it.r + jj) % g.P;
  it.nb = (jj & 1) ? g.n_nb - 1 - nbi : nbi;
  return it;
}
// staging task index -> (rank, shard, piece), in the compute tasks' order (rank by rank, peers
// r+1, r+2, ..)
__device__ inline void stage_of(const Geo& g, long long idx, int& r, int& j, int& piece) {
  piece = (int)(idx % g.n_pieces);
  idx /= g.n_pieces;
  const int jj = 1 + (int)(idx % (g.P - 1));
  r = (int)(idx / (g.P - 1));
  j = (r + jj) % g.P;
}

// ------------------------------------------------------------------------------------------------
// Task selection (the even CTA's thread 0, for its pair)
// ------------------------------------------------------------------------------------------------
// A staging task gives each CTA of the pair its own piece (arg, arg1).  With `ahead` (called
// while the current compute task's last loads are in flight) only a compute task is claimed;
// otherwise the result is CMD_NONE and the pair decides again once those loads are issued.
__device__ void decide(const Params& p, Smem* sc, Task& t, bool& was_staging, bool ahead) {
  Ctrl* c = p.ctrl;
  const Geo& g = p.g;
  t.cmd = ahead ? CMD_NONE : CMD_EXIT;
  t.arg = -1;
  t.arg1 = -1;
  t.pad = 0;
  if (sc->abort || ld_relaxed(&c->abort)) return;
  const int n_s = current_target(p);
  const bool staging_role = 2 * (int)(blockIdx.x / 2) < n_s;
  if (staging_role != was_staging) {
    atomicAdd(&c->role_switches, 1ull);
    was_staging = staging_role;
  }
  auto claim_pieces = [&]() -> bool {
    const uint32_t k = atomicAdd(&c->init_next, 2u);
    if (k >= (uint32_t)g.n_stage) return false;
    t.cmd = CMD_COMM;
    t.arg = (int)k;
    t.arg1 = k + 1 < (uint32_t)g.n_stage ? (int)k + 1 : -1;
    return true;
  };
  const bool all_claimed = ld_relaxed(&c->init_next) >= (uint32_t)g.n_stage;
  if (staging_role && !all_claimed) {
    if (ahead) return;
    if (claim_pieces()) return;
  }
  if (staging_role && p.mode == PSR_STATIC) return;
  if (ld_relaxed(&c->item_next) < (uint32_t)g.n_items) {
    const uint32_t n = atomicAdd(&c->item_next, 1u);
    if (n < (uint32_t)g.n_items) {
      t.cmd = CMD_COMPUTE;
      t.arg = (int)n;
      return;
    }
  }
  if (ahead) return;
  // no compute left: help with staging while any piece is unclaimed
  if (p.mode == PSR_ADAPTIVE && ld_relaxed(&c->init_next) < (uint32_t)g.n_stage && claim_pieces()) return;
  t.cmd = CMD_EXIT;
}

// ------------------------------------------------------------------------------------------------
// Staging task (thread 0 of a CTA): a piece of shard j's rows -> rank r's gather buffer, same rows
// ------------------------------------------------------------------------------------------------
// The stage area is free (wait_stages_free) when it starts; every copy has completed when it
// returns.  False on timeout or abort.
__device__ bool run_staging(const Params& p, Smem* sc, uint32_t smem_base, int task, uint32_t (&phase)[16]) {
  const Geo& g = p.g;
  int r, j, piece;
  stage_of(g, task, r, j, piece);
  const size_t row0 = (size_t)j * g.Ms + (size_t)piece * g.piece_rows;
  const size_t bytes = (size_t)g.piece_rows * g.K * 2;
  const uint8_t* src = reinterpret_cast<const uint8_t*>(p.a + row0 * g.K);
  uint8_t* dst = reinterpret_cast<uint8_t*>(p.gbuf + ((size_t)r * g.M + row0) * g.K);
  uint32_t* flag = p.flags + ((size_t)r * g.P + j) * g.n_pieces + piece;
  const bool drop = (p.fault == PSR_FAULT_DROP_FIRST_FLAG) && (atomicAdd(&p.ctrl->fault_count, 1u) == 0u);
  if (p.fault == PSR_FAULT_SLOW_STAGING) nanosleep_ns(20000);
  const int n_u = (int)((bytes + kCopyUnit - 1) / kCopyUnit);
  auto unit_bytes = [&](int u) {
    const size_t rem = bytes - (size_t)u * kCopyUnit;
    return (uint32_t)(rem < (size_t)kCopyUnit ? rem : (size_t)kCopyUnit);
  };
  auto issue_load = [&](int u) {
    const int b = u % kNCopyBuf;
    mbar_expect_tx(&sc->stg[b], unit_bytes(u));
    bulk_load(smem_base + b * kCopyUnit, src + (size_t)u * kCopyUnit, unit_bytes(u), &sc->stg[b]);
  };
  const int pre = n_u < kNCopyBuf - 1 ? n_u : kNCopyBuf - 1;
  for (int u = 0; u < pre; ++u) issue_load(u);
  int issued = pre;
  bool ok = true;
  for (int u = 0; u < n_u; ++u) {
    const int b = u % kNCopyBuf;
    if (u >= issued) break;
    if (ok && !wait_bar(&sc->stg[b], phase[b] & 1u, p, sc, SITE_STAGE_LOAD)) ok = false;
    if (!ok) {
      const uint64_t t0 = globaltimer_ns();  // drain this load (bounded)
      while (!mbar_try_wait(&sc->stg[b], phase[b] & 1u) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
    phase[b]++;
    if (ok) {
      bulk_store(dst + (size_t)u * kCopyUnit, smem_base + b * kCopyUnit, unit_bytes(u));
      bulk_commit();
    }
    const int nu = u + kNCopyBuf - 1;
    if (nu < n_u && ok) {
      bulk_wait_read<1>();  // the store that used buffer nu % kNCopyBuf has read shared memory
      issue_load(nu);
      issued = nu + 1;
    }
  }
  bulk_wait<0>();  // every store of the piece has completed
  if (ok && !drop) {
    fence_proxy_async_global();
    st_release(flag, 1u);
  }
  atomicAdd(&p.ctrl->stage_bytes, (unsigned long long)bytes);
  return ok;
}

// ------------------------------------------------------------------------------------------------
// Compute task: producer (thread 0 of each CTA), epilogue warps (both CTAs)
// ------------------------------------------------------------------------------------------------
// This CTA's 128 rows of the tile's A and W.  `starved` accumulates the cycles spent waiting
// for readiness flags.  False on timeout or abort.
template <class Ahead>
__device__ bool produce_tile(const Params& p, Smem* sc, uint32_t smem_base, uint32_t rank, const Item& it,
                             const CUtensorMap* tm_a, const CUtensorMap* tm_g, const CUtensorMap* tm_w,
                             uint32_t& fills, long long& starved, Ahead&& ahead) {
  const Geo& g = p.g;
  const int srow = it.mb * kBM + (int)rank * kRows;  // this CTA's first row inside the shard
  const CUtensorMap* ma = tm_a;
  int arow = it.j * g.Ms + srow;  // rows of A (local) ...
  if (it.j != it.r) {
    // ... or of rank r's gather buffer, once the pieces covering these rows are there
    ma = tm_g;
    const int p0 = srow / g.piece_rows, p1 = (srow + kRows - 1) / g.piece_rows;
    const uint32_t* f = p.flags + ((size_t)it.r * g.P + it.j) * g.n_pieces;
    for (int pc = p0; pc <= p1; ++pc) {
      uint32_t seen = ld_acquire(f + pc);
      if (seen < 1u) {
        const long long f0 = clock64();
        const bool ok = wait_flag(f + pc, 1u, seen, p, sc, SITE_FLAG);
        starved += clock64() - f0;
        if (!ok) return false;
      }
    }
    fence_proxy_async_global();  // acquire (generic) before the async-proxy reads of the buffer
    arow = it.r * g.M + it.j * g.Ms + srow;
  }
  const int n_k = g.K / kBK;
  // W rows of half h: wrow + 256h (past the rank's Ns in a half-wide tile: the next rank's rows,
  // or the tensor map's zero fill past the last one; never stored)
  const int wrow = it.r * g.Ns + it.nb * kCols + (int)rank * kRows;
  return load_tile(p, sc, smem_base, rank, ma, arow, tm_w, wrow, n_k, fills,
                        n_k > kNStage ? n_k - kNStage : 0, ahead);
}

// Epilogue warp: its 32 rows x 128 columns of each half of the tile, accumulator -> bf16 -> C_r
// (columns at or past Ns, the second half of a half-wide tile, are not stored).
__device__ bool epilogue(const Params& p, Smem* sc, uint8_t* epi, uint32_t rank, const Item& it, uint32_t item) {
  const Geo& g = p.g;
  const int warp = threadIdx.x / 32;
  const size_t grow0 = (size_t)it.j * g.Ms + (size_t)it.mb * kBM + rank * kRows + (warp % 4) * 32;
  const int col0 = it.nb * kCols + ((warp - 4) / 4) * 128;
  uint8_t* stage = epi + (warp - 4) * kEpiWarpBytes;
  uint16_t* rows = p.c + ((size_t)it.r * g.M + grow0) * g.Ns;
  return read_acc(p, sc, rank, item, [&](int cb, const uint32_t* v) {
    const int col = col0 + (cb / 2) * kBN + (cb % 2) * 64;
    if (col >= g.Ns) return;
    uint32_t w[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) w[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
    warp_store_rows<32>(stage, w, reinterpret_cast<uint8_t*>(rows + col), (size_t)g.Ns * 2);
  });
}

__global__ void __launch_bounds__(kThreads, 1)
    ag_gemm_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_a,
                   const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_w) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Smem sc;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t smem_base = (raw + 1023u) & ~1023u;
  uint8_t* epi = smem_raw + (smem_base - raw) + kStageArea;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (!launched_as_pairs(p)) return;
  const uint32_t rank = cluster_ctarank();
  if (threadIdx.x == 0) {
    init_barriers(&sc);
    for (int b = 0; b < 16; ++b) mbar_init(&sc.stg[b], 1);
    fence_barrier_init();
    if (blockIdx.x == 0) {
      unsigned long long z = 0;
      atomicCAS(&p.ctrl->t0_ns, z, (unsigned long long)globaltimer_ns());
      p.ctrl->ns_initial = (uint32_t)p.n_s_init;
      atomicMax(&p.ctrl->ns_max, (uint32_t)p.n_s_init);
      atomicMax(&p.ctrl->ns_min_inv, 0xFFFFu - (uint32_t)p.n_s_init);
    }
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_g);
    prefetch_tmap(&tm_w);
  }
  setup_pair(&sc);

  uint32_t fills = 0;  // thread 0: the stage fills this CTA issued
  const int n_k = p.g.K / kBK;
  if (warp == 0) {
    if (lane == 0) {
      uint32_t stg_phase[16] = {};
      long long starved = 0;
      if (rank == 0) {
        // the pair's scheduler, and the even CTA's producer
        bool was_staging = false;
        unsigned long long next_offer_ns = 0;
        Task next;
        next.cmd = CMD_NONE;
        int prev_cmd = CMD_NONE, prev_pieces = 0;
        long long t_prev = 0;
        for (uint32_t k = 0;; ++k) {
          Task t = next;
          next.cmd = CMD_NONE;
          if (t.cmd == CMD_NONE) decide(p, &sc, t, was_staging, false);
          // the previous task's cost, in CTA-cycles (both CTAs of the pair)
          const long long now = clock64();
          long long busy = now - t_prev;
          if (prev_cmd == CMD_COMPUTE) {
            busy -= starved;
            atomicAdd(&p.ctrl->starve_cycles, (unsigned long long)(starved > 0 ? starved : 0));
            atomicAdd(&p.ctrl->compute_cycles, 2ull * (unsigned long long)(busy > 0 ? busy : 0));
            atomicAdd(&p.ctrl->compute_tiles, 1ull);
            atomicAdd(&p.ctrl->compute_items, 1ull);
          } else if (prev_cmd == CMD_COMM) {
            atomicAdd(&p.ctrl->stage_cycles, (unsigned long long)(busy > 0 ? busy : 0) * prev_pieces);
            atomicAdd(&p.ctrl->stage_done, (unsigned long long)prev_pieces);
          }
          controller_tick(p, next_offer_ns);
          if (!post_task(p, &sc, k, t)) { sc.abort = 1; break; }
          if (t.cmd == CMD_EXIT) break;
          prev_cmd = t.cmd;
          t_prev = clock64();
          starved = 0;
          bool ok;
          if (t.cmd == CMD_COMPUTE) {
            ok = produce_tile(p, &sc, smem_base, 0, item_of(p.g, t.arg), &tm_a, &tm_g, &tm_w, fills, starved,
                              [&] { decide(p, &sc, next, was_staging, true); });
          } else {
            prev_pieces = t.arg1 >= 0 ? 2 : 1;
            ok = wait_stages_free(p, &sc, fills) && run_staging(p, &sc, smem_base, t.arg, stg_phase);
          }
          if (!ok) { sc.abort = 1; break; }
        }
      } else {
        // the odd CTA's producer
        for (uint32_t k = 0;; ++k) {
          Task t;
          if (!take_task(p, &sc, k, t)) { sc.abort = 1; break; }
          release_task(&sc, k, 1);
          if (t.cmd == CMD_EXIT) break;
          bool ok = true;
          if (t.cmd == CMD_COMPUTE)
            ok = produce_tile(p, &sc, smem_base, 1, item_of(p.g, t.arg), &tm_a, &tm_g, &tm_w, fills, starved, [] {});
          else if (t.arg1 >= 0)
            ok = wait_stages_free(p, &sc, fills) && run_staging(p, &sc, smem_base, t.arg1, stg_phase);
          if (!ok) { sc.abort = 1; break; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // the pair's MMA issuer
      uint32_t mfills = 0, items = 0;
      for (uint32_t k = 0;; ++k) {
        Task t;
        if (!take_task(p, &sc, k, t)) { sc.abort = 1; break; }
        release_task(&sc, k, 0);
        if (t.cmd == CMD_EXIT) break;
        if (t.cmd != CMD_COMPUTE) continue;
        if (!mma_tile(p, &sc, smem_base, n_k, mfills, items)) { sc.abort = 1; break; }
        ++items;
      }
    }
  } else if (warp >= 4) {
    uint32_t items = 0;
    for (uint32_t k = 0;; ++k) {
      Task t;
      const bool ok = __all_sync(0xffffffffu, take_task(p, &sc, k, t));
      if (!ok) { sc.abort = 1; break; }
      __syncwarp();
      if (lane == 0) release_task(&sc, k, rank);
      if (t.cmd == CMD_EXIT) break;
      if (t.cmd != CMD_COMPUTE) continue;
      if (!epilogue(p, &sc, epi, rank, item_of(p.g, t.arg), items)) break;
      ++items;
    }
  }
  drain_pair(&sc, rank, fills);
}

// ------------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------------
struct Layout {
  size_t ctrl, traj, flags, gbuf, total, reset_bytes;
};

static int geometry(const psr_ag_shape* sh, Geo& g) {
  if (!sh) return PSR_ERR_ARG;
  if (sh->M < 1 || sh->K < 1 || sh->Ns < 1 || sh->P < 1) return PSR_ERR_ARG;
  if (sh->M % sh->P != 0) return PSR_ERR_UNSUPPORTED;
  g.M = sh->M; g.K = sh->K; g.Ns = sh->Ns; g.P = sh->P;
  g.Ms = sh->M / sh->P;
  if (g.Ms % kBM != 0 || g.Ns % kBN != 0 || g.K % 128 != 0) return PSR_ERR_UNSUPPORTED;
  if ((long long)g.P * g.M >= (1LL << 31) || (long long)g.P * g.Ns >= (1LL << 31)) return PSR_ERR_UNSUPPORTED;
  g.n_mb = g.Ms / kBM;
  g.n_nb = (g.Ns + kCols - 1) / kCols;
  // piece: >= 512 KiB of rows, a multiple of 128 rows dividing the shard
  const long long row_bytes = (long long)g.K * 2;
  int pr = 128;
  while ((long long)pr * row_bytes < kPieceMinBytes && pr < g.Ms) pr *= 2;
  while (g.Ms % pr != 0) pr /= 2;
  if (pr < 128) pr = 128;
  g.piece_rows = pr;
  g.n_pieces = g.Ms / pr;
  g.n_items = (long long)g.P * g.P * g.n_mb * g.n_nb;
  g.n_stage = (long long)g.P * (g.P - 1) * g.n_pieces;
  if (g.n_items >= (1LL << 31) || g.n_stage >= (1LL << 31)) return PSR_ERR_UNSUPPORTED;
  return PSR_OK;
}

static size_t au(size_t x) { return (x + 255) / 256 * 256; }

static Layout layout(const Geo& g) {
  Layout l;
  size_t off = 0;
  l.ctrl = off; off += 256;
  l.traj = off; off = au(off + (size_t)kTrajMax * 8);  // the same offsets as the attention workspace
  l.flags = off; off = au(off + (size_t)g.P * g.P * g.n_pieces * 4);
  l.reset_bytes = off;
  l.gbuf = off; off = au(off + (size_t)g.P * g.M * g.K * 2);
  l.total = off;
  return l;
}

}  // namespace ag
}  // namespace psr

using namespace psr;
using namespace psr::ag;

extern "C" {

size_t psr_ag_gemm_workspace_bytes(const psr_ag_shape* sh) {
  Geo g;
  if (geometry(sh, g) != PSR_OK) return 0;
  return layout(g).total;
}

int psr_ag_gemm(const psr_ag_shape* sh, const void* a, const void* w, void* c, void* workspace, size_t ws_bytes,
                const psr_partition* part, void* stream) {
  if (!sh || !a || !w || !c || !workspace) return PSR_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PSR_ERR_ARG;
  for (const void* ptr : {a, w, (const void*)c})
    if ((reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return PSR_ERR_ARG;
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return PSR_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return PSR_ERR_UNSUPPORTED;
  const int n_cta = pair_ctas(ag_gemm_kernel, prop.multiProcessorCount);  // whole CTA pairs
  if (n_cta < 4) return PSR_ERR_CUDA;
  Geo g;
  int rc = geometry(sh, g);
  if (rc != PSR_OK) return rc;
  const Layout L = layout(g);
  if (ws_bytes < L.total) return PSR_ERR_ARG;
  psr_partition pt;
  if (part) pt = *part;
  else { pt.mode = PSR_ADAPTIVE; pt.n_staging = 0; pt.n_min = 0; pt.n_max = 0; pt.fault = 0; pt.timeout_ms = 0; }
  if (pt.mode != PSR_STATIC && pt.mode != PSR_ADAPTIVE) return PSR_ERR_ARG;
  if (pt.fault < 0 || pt.fault > PSR_FAULT_SLOW_STAGING) return PSR_ERR_ARG;

  Params kp;
  memset(&kp, 0, sizeof(kp));
  kp.g = g;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  kp.a = static_cast<const uint16_t*>(a);
  kp.gbuf = reinterpret_cast<uint16_t*>(ws + L.gbuf);
  kp.c = static_cast<uint16_t*>(c);
  kp.flags = reinterpret_cast<uint32_t*>(ws + L.flags);
  kp.ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  kp.traj = reinterpret_cast<uint32_t*>(ws + L.traj);
  kp.timeout_ns = (unsigned long long)(pt.timeout_ms > 0 ? pt.timeout_ms : 2000) * 1000000ull;
  kp.n_tiles_total = (unsigned long long)g.n_items;
  kp.n_stage_total = (unsigned long long)g.n_stage;
  kp.mode = pt.mode;
  kp.fault = pt.fault;
  kp.update_headroom = (float)kUpdateHeadroom;
  // priors (CTA-cycles): a piece at ~50 GB/s per staging SM (no less than ~6500 cycles); a task
  // (2*256*512*K flops) at ~60 % of an SM's dense bf16 rate
  const double piece_cycles = (double)g.piece_rows * g.K * 2 / 50e9 * 1.95e9;
  kp.c_s0 = (float)(piece_cycles > 6500.0 ? piece_cycles : 6500.0);
  kp.c_p0 = (float)(2.0 * kBM * kCols * (double)g.K / (0.6 * 8192.0));
  const int hard_max = n_cta - 2;  // at least one compute pair
  int n_max = pt.n_max > 0 ? pt.n_max : n_cta / 2;
  if (n_max > hard_max) n_max = hard_max;
  int n_min = pt.n_min > 0 ? pt.n_min : 1;
  if (n_min > n_max) n_min = n_max;
  kp.n_min = n_min;
  kp.n_max = n_max;
  const bool any_staging = g.n_stage > 0;
  int n_s;
  if (pt.mode == PSR_STATIC) {
    n_s = any_staging ? pt.n_staging : 0;
    if (any_staging && (n_s < 1 || n_s > hard_max)) return PSR_ERR_ARG;
  } else {
    n_s = pt.n_staging > 0 ? pt.n_staging
                           : controller_rule(n_cta, (double)g.n_stage, kStageHeadroom * kp.c_s0, (double)g.n_items,
                                             kp.c_p0, n_min, n_max);
    if (!any_staging) n_s = 0;
    else {
      if (n_s < n_min) n_s = n_min;
      if (n_s > n_max) n_s = n_max;
    }
  }
  kp.n_s_init = n_s;

  CUtensorMap ma, mg, mw;
  if (!tmap_kmajor(&ma, a, g.M, g.K, kRows) || !tmap_kmajor(&mg, kp.gbuf, (long long)g.P * g.M, g.K, kRows) ||
      !tmap_kmajor(&mw, w, (long long)g.P * g.Ns, g.K, kRows))
    return PSR_ERR_CUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, L.reset_bytes, st) != cudaSuccess) return PSR_ERR_CUDA;
  // all pairs co-resident: compute waits on staging
  if (launch_pairs(ag_gemm_kernel, n_cta, st, kp, ma, mg, mw) != cudaSuccess) {
    cudaGetLastError();
    return PSR_ERR_CUDA;
  }
  return PSR_OK;
}

}  // extern "C"
