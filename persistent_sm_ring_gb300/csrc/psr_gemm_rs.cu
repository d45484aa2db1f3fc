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
//  * compute CTAs produce one 256 x 256 partial tile of one rank per task on tcgen05 (the
//    shared tile of psr_gemm_tile.cuh) and write it in fp32 to that rank's partial buffer;
//    the epilogue warp that completes the last of an output tile's P partials enqueues the
//    tile for reduction (a gpu-scope release, like the ring's readiness flags);
//  * reduce CTAs (the communication role) take enqueued tiles, stream the P partials through
//    shared memory with TMA bulk copies, sum them in rank order (fixed, so the result does not
//    depend on timing) and write the owner's bf16 rows;
//  * compute tasks run window by window (up to 8 x 8 output tiles, every rank's partials of the
//    window before the next window), so reductions start one window after the launch and a
//    window's partials are still in L2 when they are reduced;
//  * the shared controller splits CTAs between the roles with the pages' rule.  Compute feeds
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
constexpr int kTileElems = kBM * kBN;            // fp32 elements of one partial tile
constexpr int kRoundBytes = kStageArea / 3;      // one reduce round: P partial row blocks
constexpr int kMaxP = kRoundBytes / (kBN * 4);   // at least one 256-column fp32 row per rank
static_assert(kRoundBytes % 1024 == 0, "reduce round");

enum : uint32_t { SITE_FLAG = 1, SITE_KV_FULL = 2, SITE_KV_EMPTY = 3, SITE_ACC = 4, SITE_REDUCE_LOAD = 8,
                  SITE_REDUCE_FREE = 9, SITE_QUEUE = 10 };
enum : int { CMD_EXIT = 0, CMD_COMPUTE = 1, CMD_REDUCE = 2 };

struct Geo {
  int M, N, Ks, P, Mq;
  int n_mb, n_nb;       // 256-row / 256-column output blocks
  int wm, wn;           // task window: wm x wn output tiles
  int n_out;            // output tiles
  long long n_items;    // compute tasks: P x n_out
  int cr;               // partial rows per rank in one reduce round (a power of two dividing 256)
};

struct Params {
  Geo g;
  float* part;          // [P][n_out][256][256] fp32 partial tiles
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
};

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
// Task selection (thread 0)
// ------------------------------------------------------------------------------------------------
// Reduce tickets are claimed in completion order.  In the adaptive mode a CTA claims one only
// when an enqueued tile is waiting (or when no compute task is left), so a ticket holder waits
// only for tiles whose compute tasks are running; at most n_max < N CTAs hold tickets.
__device__ void decide(const Params& p, Smem* sc, bool& was_reducing) {
  Ctrl* c = p.ctrl;
  const Geo& g = p.g;
  if (sc->abort || ld_relaxed(&c->abort)) { sc->cmd = CMD_EXIT; return; }
  const int n_s = current_target(p);
  const bool reduce_role = (int)blockIdx.x < n_s;
  if (reduce_role != was_reducing) {
    atomicAdd(&c->role_switches, 1ull);
    was_reducing = reduce_role;
  }
  const bool fixed = p.mode == PSR_STATIC;
  auto take_ticket = [&]() -> bool {
    const uint32_t h = atomicAdd(&c->q_head, 1u);
    if (h >= (uint32_t)g.n_out) return false;
    uint32_t seen = 0;
    if (!wait_flag(p.queue + h, 1u, seen, p, sc, SITE_FLAG)) { sc->cmd = CMD_EXIT; return true; }
    sc->cmd = CMD_REDUCE;
    sc->arg = (int)(seen - 1u);
    return true;
  };
  const bool compute_left = ld_relaxed(&c->item_next) < (uint32_t)g.n_items;
  if (reduce_role) {
    const uint32_t head = ld_relaxed(&c->q_head);
    if (head < (uint32_t)g.n_out) {
      if ((fixed || !compute_left || ld_relaxed(&c->q_tail) > head) && take_ticket()) return;
    }
    if (fixed) { sc->cmd = CMD_EXIT; return; }
  }
  if (!(fixed && reduce_role) && compute_left) {
    const uint32_t n = atomicAdd(&c->item_next, 1u);
    if (n < (uint32_t)g.n_items) { sc->cmd = CMD_COMPUTE; sc->arg = (int)n; return; }
  }
  // no compute task left: help with the reductions (adaptive)
  if (!fixed && ld_relaxed(&c->q_head) < (uint32_t)g.n_out && take_ticket()) return;
  sc->cmd = CMD_EXIT;
}

// ------------------------------------------------------------------------------------------------
// Reduce task: output tile o = sum over ranks of its partial tiles, rounded to bf16
// ------------------------------------------------------------------------------------------------
// Round k of the task carries rows k*cr .. k*cr+cr-1 of every rank's partial (P bulk copies of
// cr KiB into one third of the stage area); thread 0 issues the copies, the eight epilogue warps
// sum and store.  Three rounds are in flight; stg[s] counts a round's bytes, stg[3 + s] the
// eight consumer warps that have read it.  `rounds` is the CTA's lifetime round count.
__device__ void run_reduce(const Params& p, Smem* sc, uint32_t smem_base, const uint8_t* smem, int o,
                           uint32_t& rounds) {
  const Geo& g = p.g;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_rounds = kBM / g.cr;
  const uint32_t rank_bytes = (uint32_t)g.cr * kBN * 4;
  const int mb = o / g.n_nb, nb = o % g.n_nb;
  if (threadIdx.x == 0) {
    if (p.fault == PSR_FAULT_SLOW_STAGING) nanosleep_ns(20000);
    // the partials were written by other CTAs (generic proxy) and published with a release
    // that the ticket's acquire observed; order those writes, and this CTA's earlier generic
    // reads of the stage area, before the bulk copies
    fence_proxy_async_global();
    fence_proxy_async_smem();
    bool ok = true;
    for (int k = 0; k < n_rounds && ok; ++k) {
      const uint32_t u = rounds + (uint32_t)k;
      const uint32_t s = u % 3, use = u / 3;
      if (use > 0) {
        if (!wait_bar(&sc->stg[3 + s], (use - 1) & 1u, p, sc, SITE_REDUCE_FREE)) { ok = false; break; }
        fence_proxy_async_smem();  // the consumers' generic reads of the buffer before the copies into it
      }
      mbar_expect_tx(&sc->stg[s], rank_bytes * (uint32_t)g.P);
      for (int r = 0; r < g.P; ++r) {
        const float* src = p.part + ((size_t)r * g.n_out + o) * kTileElems + (size_t)k * g.cr * kBN;
        bulk_load(smem_base + s * kRoundBytes + (uint32_t)r * rank_bytes, src, rank_bytes, &sc->stg[s]);
      }
    }
    if (!ok) sc->abort = 1;
    atomicAdd(&p.ctrl->stage_bytes, (unsigned long long)rank_bytes * g.P * n_rounds);
  } else if (warp >= 4) {
    const int t = threadIdx.x - 128;  // 0..255
    const int per_round = g.cr * (kBN / 4);  // float4 elements of one rank's rows in a round
    bool ok = true;
    for (int k = 0; k < n_rounds; ++k) {
      const uint32_t u = rounds + (uint32_t)k;
      const uint32_t s = u % 3, use = u / 3;
      if (ok) ok = __all_sync(0xffffffffu, wait_bar(&sc->stg[s], use & 1u, p, sc, SITE_REDUCE_LOAD));
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
          const int row = k * g.cr + e / (kBN / 4), col = (e % (kBN / 4)) * 4;
          uint2 v;
          v.x = pack_bf16x2(acc.x, acc.y);
          v.y = pack_bf16x2(acc.z, acc.w);
          *reinterpret_cast<uint2*>(p.out + (size_t)(mb * kBM + row) * g.N + (size_t)nb * kBN + col) = v;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc->stg[3 + s]);  // also on abort: the issuer's waits stay bounded
    }
    if (!ok) sc->abort = 1;
  }
  rounds += (uint32_t)n_rounds;
}

// ------------------------------------------------------------------------------------------------
// Compute task: producer (TMA), MMA issuer (tcgen05), epilogue warpgroups -> fp32 partial tile
// ------------------------------------------------------------------------------------------------
__device__ void epilogue(const Params& p, Smem* sc, uint8_t* smem, const Item& it, int i, const Counters& cnt) {
  const Geo& g = p.g;
  const int warp = threadIdx.x / 32;
  float* tile = p.part + ((size_t)it.r * g.n_out + it.o) * kTileElems + (size_t)i * 128 * kBN;
  // the stage area is idle during the epilogue (every MMA of the tile has completed): 8 KiB per warp
  uint8_t* stage = smem + (warp - 4) * 8192;
  uint8_t* rows = reinterpret_cast<uint8_t*>(tile + (size_t)((warp % 4) * 32) * kBN);
  const bool ok = read_tile(p, sc, i, cnt, SITE_ACC, [&](int, int cb, const uint32_t(&v)[64]) {
    warp_store_rows<64>(stage, v, rows + cb * 256, (size_t)kBN * 4);
  });
  if (!ok) return;
  // this warp's 32 rows are written: publish them (each thread's stores before lane 0's release)
  __threadfence();
  __syncwarp();
  if ((threadIdx.x % 32) == 0) {
    const bool drop = (p.fault == PSR_FAULT_DROP_FIRST_FLAG) && (atomicAdd(&p.ctrl->fault_count, 1u) == 0u);
    if (!drop) {
      const uint32_t old = atom_add_acq_rel(p.count + it.o, 1u);
      if (old + 1u == 8u * (uint32_t)g.P) {
        const uint32_t k = atomicAdd(&p.ctrl->q_tail, 1u);
        if (k < (uint32_t)g.n_out) st_release(p.queue + k, (uint32_t)it.o + 1u);
        else raise_error(p, SITE_QUEUE);
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_rs_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_a,
                   const __grid_constant__ CUtensorMap tm_w) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ Smem sc;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t smem_base = (raw + 1023u) & ~1023u;
  const uint8_t* smem = smem_raw + (smem_base - raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kNStage; ++s) {
      mbar_init(&sc.full[s], 1);
      mbar_init(&sc.empty[s], 1);
    }
    mbar_init(&sc.acc_full, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&sc.stg[s], 1);      // a reduce round's bytes have landed
      mbar_init(&sc.stg[3 + s], 8);  // the eight consumer warps have read it
    }
    mbar_init(&sc.drain, 1);
    sc.abort = 0;
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
  if (warp == 1) {
    tmem_alloc(&sc.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  Counters cnt{0, 0};
  uint32_t rounds = 0;
  bool was_reducing = false;
  long long t_task = 0;
  const int n_k = p.g.Ks / kBK;
  while (true) {
    if (threadIdx.x == 0) {
      decide(p, &sc, was_reducing);
      t_task = clock64();
    }
    __syncthreads();
    const int cmd = sc.cmd, arg = sc.arg;
    if (cmd == CMD_EXIT) break;
    if (cmd == CMD_REDUCE) {
      run_reduce(p, &sc, smem_base, smem, arg, rounds);
    } else {
      const Item it = item_of(p.g, arg);
      if (warp == 0 && lane == 0) {
        Counters c2 = cnt;
        fence_proxy_async_smem();  // earlier generic reads of the stage area (a reduce task)
        if (!load_tile(p, &sc, smem_base, &tm_a, it.r * p.g.M + it.mb * kBM, &tm_w, it.r * p.g.N + it.nb * kBN, n_k,
                       c2, SITE_KV_EMPTY))
          sc.abort = 1;
      } else if (warp == 1 && lane == 0) {
        Counters c2 = cnt;
        mma_tile(p, &sc, smem_base, n_k, c2, SITE_KV_FULL);
      } else if (warp >= 4) {
        epilogue(p, &sc, smem_raw + (smem_base - raw), it, warp < 8 ? 0 : 1, cnt);
      }
      cnt.fills += (uint32_t)n_k;
      cnt.items++;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
      long long busy = clock64() - t_task;
      const unsigned long long dt = (unsigned long long)(busy > 0 ? busy : 0);
      if (cmd == CMD_REDUCE) {
        atomicAdd(&p.ctrl->stage_cycles, dt);
        atomicAdd(&p.ctrl->stage_done, 1ull);
      } else {
        atomicAdd(&p.ctrl->compute_cycles, dt);
        atomicAdd(&p.ctrl->compute_tiles, 1ull);
        atomicAdd(&p.ctrl->compute_items, 1ull);
      }
      const uint32_t tick = atomicAdd(&p.ctrl->ticks, 1u);
      if (p.mode == PSR_ADAPTIVE && (tick % 16u) == 0) controller_update(p);
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
  drain_and_release(&sc, cnt);
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
  g.n_nb = g.N / kBN;
  g.wm = largest_divisor_upto(g.n_mb, 8);
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
  l.part = off; off = au(off + (size_t)g.P * g.n_out * kTileElems * 4);
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
  const int n_cta = prop.multiProcessorCount;
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
  // priors (CTA-cycles): a reduction streams P partial tiles in and one bf16 tile out at
  // ~100 GB/s per SM; a compute task (2*256*256*Ks flops) at ~60 % of an SM's dense bf16 rate
  kp.c_s0 = (float)(((double)g.P * kTileElems * 4 + kTileElems * 2) / 100e9 * 1.95e9);
  kp.c_p0 = (float)(2.0 * kBM * kBN * (double)g.Ks / (0.6 * 8192.0));
  const int hard_max = n_cta - 1;
  int n_max = pt.n_max > 0 ? pt.n_max : n_cta / 2;
  if (n_max > hard_max) n_max = hard_max;
  int n_min = pt.n_min > 0 ? pt.n_min : 1;
  if (n_min > n_max) n_min = n_max;
  kp.n_min = n_min;
  kp.n_max = n_max;
  int n_s;
  if (pt.mode == PSR_STATIC) {
    n_s = pt.n_staging;
    if (n_s < 1 || n_s > n_cta - 1) return PSR_ERR_ARG;
  } else {
    // compute feeds the reductions: nothing to reduce at launch, so every CTA starts computing
    n_s = pt.n_staging > 0 ? (pt.n_staging < n_max ? pt.n_staging : n_max) : 0;
  }
  kp.n_s_init = n_s;

  CUtensorMap ma, mw;
  if (!tmap_kmajor(&ma, a, (long long)g.P * g.M, g.Ks, 128) || !tmap_kmajor(&mw, w, (long long)g.P * g.N, g.Ks, kBN))
    return PSR_ERR_CUDA;

  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_rs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (attr_err != cudaSuccess) return PSR_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, L.reset_bytes, st) != cudaSuccess) return PSR_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_cta);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: reductions wait on compute
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gemm_rs_kernel, kp, ma, mw) != cudaSuccess) {
    cudaGetLastError();
    return PSR_ERR_CUDA;
  }
  return PSR_OK;
}

}  // extern "C"
