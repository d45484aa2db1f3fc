// GEMM + ReduceScatter as one persistent kernel on sm_103a.
//
// The mKernel pages' GEMM+ReduceScatter kernel (dataforcee / chathome "five fused kernels"
// table, GEMM + ReduceScatter row; pwwt.cn analysis §2.6 Table 3: tensor parallel, compute
// feeds communication, partial tiles reduced as they are produced, 2-32 tile chunks): rank r
// holds its K-shard A_r ([M][Ks]) of the activations and W_r ([N][Ks]) of the weights and
// computes the partial product C_r = A_r W_r^T; the ranks reduce-scatter the partials, so that
// rank q receives rows [q*M/P, (q+1)*M/P) of sum_r C_r, and each output tile is reduced and
// forwarded to its owner as soon as its partials exist.  On one GPU the P ranks are emulated
// in HBM:
//
//  * the CTAs work in pairs (clusters of two); a pair takes either role;
//  * a compute pair produces one 256 x 512 partial tile of one rank per task (the pair tile of
//    psr_gemm_tile.cuh with two accumulator halves: each CTA 128 rows x 512 columns, tcgen05
//    cta_group::2) and writes it in fp32 to that rank's partial buffer as two 256 x 256 halves;
//    when N is an odd multiple of 256 a rank's last tile is half wide (its second half is
//    computed and not stored); the epilogue warp that completes the last of an output tile's
//    P partials enqueues the tile for reduction (a gpu-scope release, like the ring's
//    readiness flags);
//  * each CTA of a reduce pair (the communication role) takes enqueued tiles, streams the P
//    partials through shared memory with TMA bulk copies (a round carries a block of rows of one
//    half from every rank), sums them in rank order (fixed, so the result does not depend on
//    timing) and writes the owner's bf16 rows;
//  * compute tasks run window by window (up to 16 x 8 output tiles, every rank's partials of
//    the window before the next window), so reductions start one window after the launch, and a
//    rank's A and W blocks of the window are read from HBM about once per window (with
//    256 x 256 tiles, windows of 8 x 8 instead of 16 x 16 read them twice as often: 6.1 GB of
//    DRAM reads per launch against 4.6);
//  * the shared controller splits the pairs between the roles with the pages' rule (a target of
//    n reduce CTAs gives ceil(n/2) reduce pairs).  Compute feeds
//    communication here, so the launch starts with no reduce CTA (pwwt.cn §2.4: the data
//    dependence decides the initial allocation) and the controller adds them as tiles complete.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "../../include/psr.h"
#include "psr_control.cuh"
#include "psr_device.cuh"
#include "psr_gemm_tile.cuh"
#include "psr_schedule.h"

namespace psr {
namespace rs {

using namespace gemm;
constexpr int kTileElems = kBM * kBN;            // fp32 elements of one half (256 x 256) of a partial tile
constexpr int kRoundBytes = kStageArea / 3;      // one reduce round: P partial row blocks
constexpr int kMaxP = kRoundBytes / (kBN * 4);   // at least one 256-column fp32 row per rank
static_assert(kRoundBytes % 1024 == 0, "reduce round");

enum : uint32_t { SITE_FLAG = 1, SITE_REDUCE_LOAD = 8, SITE_REDUCE_FREE = 9, SITE_QUEUE = 10 };

struct Geo {
  int M, N, Ks, P, Mq;
  int n_mb, n_nb;       // 256-row / 512-column output blocks (the last one half wide when N % 512 = 256)
  int wm, wn;           // task window: wm x wn output tiles
  int n_out;            // output tiles
  long long n_items;    // compute tasks: P x n_out
  int cr;               // partial rows per rank in one reduce round (a power of two dividing 256)
};

struct Params {
  Geo g;
  float* part;          // [P][n_out][2][256][256] fp32 partial tiles (two halves each)
  uint16_t* out;        // [M][N] bf16
  uint32_t* count;      // [n_out] epilogue-warp arrivals (8 per partial tile)
  uint32_t* queue;      // [n_out] tiles ready for reduction (+1), in completion order
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

// 256-column halves of output tile column nb: 2, or 1 for a half-wide last tile
__device__ __host__ inline int halves_of(const Geo& g, int nb) {
  return (nb == g.n_nb - 1 && g.N % kCols != 0) ? 1 : 2;
}

// compute task index -> (rank, m-block, n-block): window by window, rank by rank inside a
// window, W tile by W tile inside a rank (consecutive tasks share it)
struct Item {
  int r, mb, nb, o;
};
__device__ __host__ inline Item item_of(const Geo& g, long long idx) {
  const int tiles_w = g.wm * g.wn;
  const long long per_win = (long long)g.P * tiles_w;
  const int win = (int)(idx / per_win);
  const int rem = (int)(idx % per_win);
  Item it;
  it.r = rem / tiles_w;
  const int t = rem % tiles_w;
  const int n_wn = g.n_nb / g.wn;
  it.nb = (win % n_wn) * g.wn + t / g.wm;
  it.mb = (win / n_wn) * g.wm + t % g.wm;
  it.o = it.mb * g.n_nb + it.nb;
  return it;
}

// ------------------------------------------------------------------------------------------------
// Task selection (the even CTA's thread 0, for its pair)
// ------------------------------------------------------------------------------------------------
// Reduce tickets are claimed in completion order; a reduce task carries the queue positions of
// the even CTA's ticket (arg) and of the odd CTA's (arg1, or -1).  In the adaptive mode a pair
// claims a ticket only when an enqueued tile is waiting (or when no compute task is left), and
// a second one only when a second tile is waiting, so a ticket holder waits only for tiles whose
// compute tasks are running; at most n_max < N CTAs hold tickets.  With `ahead` (called while
// the current compute task's last loads are in flight) only a compute task is claimed: a ticket
// may wait for that very task.
__device__ void decide(const Params& p, Smem* sc, Task& t, bool& was_reducing, bool ahead) {
  Ctrl* c = p.ctrl;
  const Geo& g = p.g;
  t.cmd = ahead ? CMD_NONE : CMD_EXIT;
  t.arg = -1;
  t.arg1 = -1;
  t.pad = 0;
  if (sc->abort || ld_relaxed(&c->abort)) return;
  const int n_s = current_target(p);
  const bool reduce_role = 2 * (int)(blockIdx.x / 2) < n_s;
  if (reduce_role != was_reducing) {
    atomicAdd(&c->role_switches, 1ull);
    was_reducing = reduce_role;
  }
  const bool fixed = p.mode == PSR_STATIC;
  const bool compute_left = ld_relaxed(&c->item_next) < (uint32_t)g.n_items;
  auto take_tickets = [&]() -> bool {
    const uint32_t h = atomicAdd(&c->q_head, 1u);
    if (h >= (uint32_t)g.n_out) return false;
    uint32_t seen = 0;
    if (!wait_flag(p.queue + h, 1u, seen, p, sc, SITE_FLAG)) return true;  // CMD_EXIT
    t.cmd = CMD_COMM;
    t.arg = (int)h;
    if (fixed || !compute_left || ld_relaxed(&c->q_tail) > h + 1) {
      const uint32_t h1 = atomicAdd(&c->q_head, 1u);
      if (h1 < (uint32_t)g.n_out) {
        if (!wait_flag(p.queue + h1, 1u, seen, p, sc, SITE_FLAG)) {
          t.cmd = CMD_EXIT;
          return true;
        }
        t.arg1 = (int)h1;
      }
    }
    return true;
  };
  if (reduce_role) {
    const uint32_t head = ld_relaxed(&c->q_head);
    if (head < (uint32_t)g.n_out && (fixed || !compute_left || ld_relaxed(&c->q_tail) > head)) {
      if (ahead) return;
      if (take_tickets()) return;
    }
    if (fixed) return;
  }
  if (compute_left) {
    const uint32_t n = atomicAdd(&c->item_next, 1u);
    if (n < (uint32_t)g.n_items) {
      t.cmd = CMD_COMPUTE;
      t.arg = (int)n;
      return;
    }
  }
  if (ahead) return;
  // no compute task left: help with the reductions (adaptive)
  if (!fixed && ld_relaxed(&c->q_head) < (uint32_t)g.n_out && take_tickets()) return;
  t.cmd = CMD_EXIT;
}

// ------------------------------------------------------------------------------------------------
// Reduce task (one CTA): output tile o = sum over ranks of its partial tiles, rounded to bf16
// ------------------------------------------------------------------------------------------------
// Round k of the task carries rows kr*cr .. kr*cr+cr-1 of half h of every rank's partial
// (h = k / (256/cr), kr = k % (256/cr); P bulk copies of cr KiB into one third of the stage area;
// a half-wide tile has rounds of half 0 only); thread 0 issues the copies, the eight epilogue warps
// sum and store.  Three rounds are in flight; stg[s] counts a round's bytes, stg[3 + s] the
// eight consumer warps that have read it.  `rounds` is the CTA's lifetime round count, kept by
// both sides.  `h` is the ticket's queue position (its entry is already published: the
// scheduler waited for it).
//
// Producer side.  The stage area is free of MMA reads first (wait_stages_free), and the
// consumers have read the last rounds before it returns, so that later TMA fills may overwrite
// the area.  False on timeout or abort.
__device__ bool reduce_loads(const Params& p, Smem* sc, uint32_t smem_base, int h, uint32_t& rounds, uint32_t fills) {
  const Geo& g = p.g;
  const int o = (int)ld_acquire(p.queue + h) - 1;
  const int rb = kBM / g.cr;  // row blocks per half
  const int n_rounds = halves_of(g, o % g.n_nb) * rb;
  const uint32_t rank_bytes = (uint32_t)g.cr * kBN * 4;
  if (p.fault == PSR_FAULT_SLOW_STAGING) nanosleep_ns(20000);
  const uint32_t r0 = rounds;
  rounds += (uint32_t)n_rounds;
  if (!wait_stages_free(p, sc, fills)) return false;
  // the partials were written by other CTAs (generic proxy) and published with a release that
  // the acquire above observed; order those writes before the bulk copies
  fence_proxy_async_global();
  for (int k = 0; k < n_rounds; ++k) {
    const uint32_t u = r0 + (uint32_t)k;
    const uint32_t s = u % 3, use = u / 3;
    if (use > 0) {
      if (!wait_bar(&sc->stg[3 + s], (use - 1) & 1u, p, sc, SITE_REDUCE_FREE)) return false;
      fence_proxy_async_smem();  // the consumers' generic reads of the buffer before the copies into it
    }
    mbar_expect_tx(&sc->stg[s], rank_bytes * (uint32_t)g.P);
    for (int r = 0; r < g.P; ++r) {
      const float* src =
          p.part + (((size_t)r * g.n_out + o) * 2 + k / rb) * kTileElems + (size_t)(k % rb) * g.cr * kBN;
      bulk_load(smem_base + s * kRoundBytes + (uint32_t)r * rank_bytes, src, rank_bytes, &sc->stg[s]);
    }
  }
  atomicAdd(&p.ctrl->stage_bytes, (unsigned long long)rank_bytes * g.P * n_rounds);
  const uint32_t first = rounds >= 3u ? rounds - 3u : 0u;
  for (uint32_t u = first; u < rounds; ++u)
    if (!wait_bar(&sc->stg[3 + u % 3], (u / 3) & 1u, p, sc, SITE_REDUCE_FREE)) return false;
  fence_proxy_async_smem();
  return true;
}

// Consumer side (the eight epilogue warps).  False on timeout or abort.
__device__ bool reduce_sums(const Params& p, Smem* sc, const uint8_t* smem, int h, uint32_t& rounds) {
  const Geo& g = p.g;
  const int lane = threadIdx.x % 32;
  const int o = (int)ld_acquire(p.queue + h) - 1;
  const int mb = o / g.n_nb, nb = o % g.n_nb;
  const int rb = kBM / g.cr;  // row blocks per half
  const int n_rounds = halves_of(g, nb) * rb;
  const int t = threadIdx.x - 128;            // 0..255
  const int per_round = g.cr * (kBN / 4);     // float4 elements of one rank's rows in a round
  bool ok = true;
  for (int k = 0; k < n_rounds; ++k) {
    const uint32_t u = rounds + (uint32_t)k;
    const uint32_t s = u % 3, use = u / 3;
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(&sc->stg[s], use & 1u, p, sc, SITE_REDUCE_LOAD, kSlack));
    if (ok) {
      const float4* base = reinterpret_cast<const float4*>(smem + s * kRoundBytes);
      for (int e = t; e < per_round; e += 256) {
        float4 acc = base[e];
        for (int r = 1; r < g.P; ++r) {
          const float4 x = base[r * per_round + e];
          acc.x += x.x;
          acc.y += x.y;
          acc.z += x.z;
          acc.w += x.w;
        }
        const int row = (k % rb) * g.cr + e / (kBN / 4);
        const int col = nb * kCols + (k / rb) * kBN + (e % (kBN / 4)) * 4;
        uint2 v;
        v.x = pack_bf16x2(acc.x, acc.y);
        v.y = pack_bf16x2(acc.z, acc.w);
        *reinterpret_cast<uint2*>(p.out + (size_t)(mb * kBM + row) * g.N + col) = v;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sc->stg[3 + s]);  // also on abort: the issuer's waits stay bounded
  }
  rounds += (uint32_t)n_rounds;
  if (!ok) sc->abort = 1;
  return ok;
}

// ------------------------------------------------------------------------------------------------
// Compute task epilogue (each epilogue warp of both CTAs) -> fp32 partial tile
// ------------------------------------------------------------------------------------------------
// The warp's 32 rows x 128 columns of each stored half of the partial tile; then its arrival on
// the tile's count (16 warps per partial), and the last arrival of the output tile's P partials
// enqueues it.
__device__ bool epilogue(const Params& p, Smem* sc, uint8_t* epi, uint32_t rank, const Item& it, uint32_t item) {
  const Geo& g = p.g;
  const int warp = threadIdx.x / 32;
  float* tile = p.part + ((size_t)it.r * g.n_out + it.o) * 2 * kTileElems;
  const int row0 = (int)rank * kRows + (warp % 4) * 32, col0 = ((warp - 4) / 4) * 128;
  const int halves = halves_of(g, it.nb);
  uint8_t* stage = epi + (warp - 4) * kEpiWarpBytes;
  const bool ok = read_acc(p, sc, rank, item, [&](int cb, const uint32_t* v) {
    if (cb / 2 >= halves) return;
    uint8_t* rows =
        reinterpret_cast<uint8_t*>(tile + (size_t)(cb / 2) * kTileElems + (size_t)row0 * kBN + col0 + (cb % 2) * 64);
    warp_store_rows<32>(stage, v, rows, (size_t)kBN * 4);
    warp_store_rows<32>(stage, v + 32, rows + 128, (size_t)kBN * 4);
  });
  if (!ok) return false;
  // this warp's rows are written: publish them (each thread's stores before lane 0's release)
  __threadfence();
  __syncwarp();
  if ((threadIdx.x % 32) == 0) {
    const bool drop = (p.fault == PSR_FAULT_DROP_FIRST_FLAG) && (atomicAdd(&p.ctrl->fault_count, 1u) == 0u);
    if (!drop) {
      const uint32_t old = atom_add_acq_rel(p.count + it.o, 1u);
      if (old + 1u == 2u * kEpiWarps * (uint32_t)g.P) {
        const uint32_t k = atomicAdd(&p.ctrl->q_tail, 1u);
        if (k < (uint32_t)g.n_out) st_release(p.queue + k, (uint32_t)it.o + 1u);
        else raise_error(p, SITE_QUEUE);
      }
    }
  }
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_rs_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_a,
                   const __grid_constant__ CUtensorMap tm_w) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Smem sc;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t smem_base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (smem_base - raw);
  uint8_t* epi = smem + kStageArea;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (!launched_as_pairs(p)) return;
  const uint32_t rank = cluster_ctarank();
  if (threadIdx.x == 0) {
    init_barriers(&sc);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&sc.stg[s], 1);              // a reduce round's bytes have landed
      mbar_init(&sc.stg[3 + s], kEpiWarps);  // the eight consumer warps have read it
    }
    fence_barrier_init();
    if (blockIdx.x == 0) {
      unsigned long long z = 0;
      atomicCAS(&p.ctrl->t0_ns, z, (unsigned long long)globaltimer_ns());
      p.ctrl->ns_initial = (uint32_t)p.n_s_init;
      atomicMax(&p.ctrl->ns_max, (uint32_t)p.n_s_init);
      atomicMax(&p.ctrl->ns_min_inv, 0xFFFFu - (uint32_t)p.n_s_init);
    }
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_w);
  }
  setup_pair(&sc);

  const Geo& g = p.g;
  const int n_k = g.Ks / kBK;
  uint32_t fills = 0;   // thread 0: the stage fills this CTA issued
  uint32_t rounds = 0;  // thread 0 and the epilogue warps: reduce rounds of this CTA
  // This CTA's share of a compute task's loads.
  auto produce = [&](const Task& t, int ahead_at, auto&& ahead) {
    const Item it = item_of(g, t.arg);
    // W rows of half h: + 256h (past N in a half-wide tile: the next rank's rows, or the
    // tensor map's zero fill past the last one; never stored)
    return load_tile(p, &sc, smem_base, rank, &tm_a, it.r * g.M + it.mb * kBM + (int)rank * kRows, &tm_w,
                          it.r * g.N + it.nb * kCols + (int)rank * kRows, n_k, fills, ahead_at, ahead);
  };
  if (warp == 0) {
    if (lane == 0) {
      if (rank == 0) {
        // the pair's scheduler, and the even CTA's producer
        bool was_reducing = false;
        unsigned long long next_offer_ns = 0;
        Task next;
        next.cmd = CMD_NONE;
        int prev_cmd = CMD_NONE, prev_tickets = 0;
        long long t_prev = 0;
        for (uint32_t k = 0;; ++k) {
          Task t = next;
          next.cmd = CMD_NONE;
          if (t.cmd == CMD_NONE) decide(p, &sc, t, was_reducing, false);
          // the previous task's cost, in CTA-cycles (both CTAs of the pair)
          const long long now = clock64();
          const unsigned long long busy = (unsigned long long)(now > t_prev ? now - t_prev : 0);
          if (prev_cmd == CMD_COMPUTE) {
            atomicAdd(&p.ctrl->compute_cycles, 2ull * busy);
            atomicAdd(&p.ctrl->compute_tiles, 1ull);
            atomicAdd(&p.ctrl->compute_items, 1ull);
          } else if (prev_cmd == CMD_COMM) {
            atomicAdd(&p.ctrl->stage_cycles, busy * (unsigned long long)prev_tickets);
            atomicAdd(&p.ctrl->stage_done, (unsigned long long)prev_tickets);
          }
          controller_tick(p, next_offer_ns);
          if (!post_task(p, &sc, k, t)) { sc.abort = 1; break; }
          if (t.cmd == CMD_EXIT) break;
          prev_cmd = t.cmd;
          t_prev = clock64();
          bool ok;
          if (t.cmd == CMD_COMPUTE) {
            ok = produce(t, n_k > kNStage ? n_k - kNStage : 0, [&] { decide(p, &sc, next, was_reducing, true); });
          } else {
            prev_tickets = t.arg1 >= 0 ? 2 : 1;
            ok = reduce_loads(p, &sc, smem_base, t.arg, rounds, fills);
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
          if (t.cmd == CMD_COMPUTE) ok = produce(t, -1, [] {});
          else if (t.arg1 >= 0) ok = reduce_loads(p, &sc, smem_base, t.arg1, rounds, fills);
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
      if (t.cmd == CMD_COMPUTE) {
        if (!epilogue(p, &sc, epi, rank, item_of(g, t.arg), items)) break;
        ++items;
      } else {
        const int h = rank == 0 ? t.arg : t.arg1;
        if (h >= 0 && !reduce_sums(p, &sc, smem, h, rounds)) break;
      }
    }
  }
  // every bulk copy of a reduce round has landed before the CTA exits (bounded)
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t s = 0; s < 3 && s < rounds; ++s) {
      const uint32_t uses = (rounds - s + 2) / 3;
      while (!mbar_try_wait(&sc.stg[s], (uses - 1) & 1u) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  }
  drain_pair(&sc, rank, fills);
}

// ------------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------------
struct Layout {
  size_t ctrl, traj, count, queue, part, total, reset_bytes;
};

static int largest_divisor_upto(int n, int cap) {
  for (int d = cap; d > 1; --d)
    if (n % d == 0) return d;
  return 1;
}

static int geometry(const psr_rs_shape* sh, Geo& g) {
  if (!sh) return PSR_ERR_ARG;
  if (sh->M < 1 || sh->N < 1 || sh->Ks < 1 || sh->P < 1) return PSR_ERR_ARG;
  if (sh->M % sh->P != 0) return PSR_ERR_UNSUPPORTED;
  g.M = sh->M; g.N = sh->N; g.Ks = sh->Ks; g.P = sh->P;
  g.Mq = sh->M / sh->P;
  if (g.Mq % kBM != 0 || g.N % kBN != 0 || g.Ks % kBK != 0 || g.P > kMaxP) return PSR_ERR_UNSUPPORTED;
  if ((long long)g.P * g.M >= (1LL << 31) || (long long)g.P * g.N >= (1LL << 31)) return PSR_ERR_UNSUPPORTED;
  g.n_mb = g.M / kBM;
  g.n_nb = (g.N + kCols - 1) / kCols;
  g.wm = largest_divisor_upto(g.n_mb, 16);
  g.wn = largest_divisor_upto(g.n_nb, 8);
  const long long n_out = (long long)g.n_mb * g.n_nb;
  if (n_out >= (1LL << 30) || n_out * g.P >= (1LL << 31)) return PSR_ERR_UNSUPPORTED;
  g.n_out = (int)n_out;
  g.n_items = n_out * g.P;
  int cr = 1;
  while (cr * 2 * g.P * kBN * 4 <= kRoundBytes && cr * 2 <= kBM) cr *= 2;
  g.cr = cr;
  return PSR_OK;
}

static size_t au(size_t x) { return (x + 255) / 256 * 256; }

static Layout layout(const Geo& g) {
  Layout l;
  size_t off = 0;
  l.ctrl = off; off += 256;
  l.traj = off; off = au(off + (size_t)kTrajMax * 8);  // the same offsets as the other workspaces
  l.count = off; off = au(off + (size_t)g.n_out * 4);
  l.queue = off; off = au(off + (size_t)g.n_out * 4);
  l.reset_bytes = off;
  l.part = off; off = au(off + (size_t)g.P * g.n_out * 2 * kTileElems * 4);
  l.total = off;
  return l;
}

}  // namespace rs
}  // namespace psr

using namespace psr;
using namespace psr::rs;

extern "C" {

size_t psr_gemm_rs_workspace_bytes(const psr_rs_shape* sh) {
  Geo g;
  if (geometry(sh, g) != PSR_OK) return 0;
  return layout(g).total;
}

int psr_gemm_rs(const psr_rs_shape* sh, const void* a, const void* w, void* out, void* workspace, size_t ws_bytes,
                const psr_partition* part, void* stream) {
  if (!sh || !a || !w || !out || !workspace) return PSR_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PSR_ERR_ARG;
  for (const void* ptr : {a, w, (const void*)out})
    if ((reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return PSR_ERR_ARG;
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return PSR_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return PSR_ERR_UNSUPPORTED;
  const int n_cta = pair_ctas(gemm_rs_kernel, prop.multiProcessorCount);  // whole CTA pairs
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
  kp.part = reinterpret_cast<float*>(ws + L.part);
  kp.out = static_cast<uint16_t*>(out);
  kp.count = reinterpret_cast<uint32_t*>(ws + L.count);
  kp.queue = reinterpret_cast<uint32_t*>(ws + L.queue);
  kp.ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  kp.traj = reinterpret_cast<uint32_t*>(ws + L.traj);
  kp.timeout_ns = (unsigned long long)(pt.timeout_ms > 0 ? pt.timeout_ms : 2000) * 1000000ull;
  kp.n_tiles_total = (unsigned long long)g.n_items;
  kp.n_stage_total = (unsigned long long)g.n_out;
  kp.mode = pt.mode;
  kp.fault = pt.fault;
  kp.update_headroom = (float)kUpdateHeadroom;
  // priors (CTA-cycles): a reduction streams P partial tiles in and one bf16 tile out at
  // ~100 GB/s per SM; a compute task (2*256*512*Ks flops) at ~60 % of an SM's dense bf16 rate
  kp.c_s0 = (float)(((double)g.P * 2 * kTileElems * 4 + 2 * kTileElems * 2) / 100e9 * 1.95e9);
  kp.c_p0 = (float)(2.0 * kBM * kCols * (double)g.Ks / (0.6 * 8192.0));
  const int hard_max = n_cta - 2;  // at least one compute pair
  int n_max = pt.n_max > 0 ? pt.n_max : n_cta / 2;
  if (n_max > hard_max) n_max = hard_max;
  int n_min = pt.n_min > 0 ? pt.n_min : 1;
  if (n_min > n_max) n_min = n_max;
  kp.n_min = n_min;
  kp.n_max = n_max;
  int n_s;
  if (pt.mode == PSR_STATIC) {
    n_s = pt.n_staging;
    if (n_s < 1 || n_s > hard_max) return PSR_ERR_ARG;
  } else {
    // compute feeds the reductions: nothing to reduce at launch, so every CTA starts computing
    n_s = pt.n_staging > 0 ? (pt.n_staging < n_max ? pt.n_staging : n_max) : 0;
  }
  kp.n_s_init = n_s;

  CUtensorMap ma, mw;
  if (!tmap_kmajor(&ma, a, (long long)g.P * g.M, g.Ks, kRows) || !tmap_kmajor(&mw, w, (long long)g.P * g.N, g.Ks, kRows))
    return PSR_ERR_CUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, L.reset_bytes, st) != cudaSuccess) return PSR_ERR_CUDA;
  // all pairs co-resident: reductions wait on compute
  if (launch_pairs(gemm_rs_kernel, n_cta, st, kp, ma, mw) != cudaSuccess) {
    cudaGetLastError();
    return PSR_ERR_CUDA;
  }
  return PSR_OK;
}

}  // extern "C"
