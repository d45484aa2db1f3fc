// The 256 x 512 output tile of the persistent GEMM kernels (AllGather+GEMM and
// GEMM+ReduceScatter) on sm_103a, computed by a pair of CTAs (a cluster of two SMs) as two
// halves of 256 columns.
//
//  * each CTA of the pair loads 128 of the tile's A rows and, per half h, 128 of its W rows
//    (output columns 256*h + 128*rank ..), one 64-wide K step per stage, K-major with the
//    128-byte swizzle, into a ring of four 48 KiB stages; both CTAs' TMA loads are counted on
//    the even CTA's stage barrier;
//  * one thread of the even CTA issues tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16)
//    per half: each SM accumulates its 128 rows x 256 columns per half in fp32 tensor memory,
//    the two halves filling its 512 columns; each half is released as soon as the epilogue
//    warps hold it in registers, and the next tile's first products into it wait only for
//    that.  The tile moves 48 KiB per SM and K step, 48 B/clk at the tensor rate: a 256 x 256
//    tile (double-buffered accumulators) needs 64 B/clk, above the ~56 B/clk of TMA tile loads
//    that a GB300 SM was measured to land;
//  * the even CTA's scheduling thread hands tasks to the roles of both CTAs through a ring of
//    task slots in shared memory (the odd CTA's copy written with distributed stores), each
//    slot released by an mbarrier: no role waits for another at a task boundary;
//  * eight epilogue warps per CTA read the accumulators back with tcgen05.ld (warp w: tensor
//    memory lanes 32*(w%4) .., columns 256*h + 128*((w-4)/4) .. of half h) and hand 64-column
//    blocks to a kernel-specific store.
// Each kernel adds its own task selection, data dependencies, communication role and epilogue
// destination.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "psr_control.cuh"
#include "psr_device.cuh"

namespace psr {
namespace gemm {

constexpr int kBM = 256;    // output rows per tile (128 per CTA of the pair)
constexpr int kBN = 256;    // output columns per half (W rows; 128 loaded by each CTA)
constexpr int kHalves = 2;
constexpr int kCols = kHalves * kBN;  // output columns per tile
constexpr int kBK = 64;     // K per stage (one 128-byte swizzle atom of bf16)
constexpr int kRows = 128;  // A rows, and W rows per half, one CTA loads per tile
constexpr int kHalf = kRows * kBK * 2;                  // 16 KiB
constexpr int kStageBytes = (1 + kHalves) * kHalf;      // this CTA's A rows and W rows of one K step
constexpr int kNStage = 4;
constexpr int kStageArea = kNStage * kStageBytes;       // 192 KiB; also the scratch of the comm roles
constexpr int kEpiWarps = 8;
constexpr int kEpiWarpBytes = 4096;  // one warp's store staging: 32 rows x 128 bytes
constexpr int kEpiArea = kEpiWarps * kEpiWarpBytes;
constexpr int kSmem = 1024 + kStageArea + kEpiArea;
constexpr int kWarps = 12, kThreads = kWarps * 32;
constexpr int kSlots = 4;  // task ring
// readers of a task slot: the odd CTA's producer, the MMA issuer, the epilogue warps of both CTAs
constexpr uint32_t kTaskReaders = 2 + 2 * kEpiWarps;
// the waits inside the tile pipeline give up after kSlack timeouts: a stall there is a
// consequence of a wait upstream (a readiness flag, a queue entry), which reports first
constexpr uint32_t kSlack = 4;
static_assert(kSmem + 1024 <= 232448, "shared memory");

enum : uint32_t { SITE_FULL = 2, SITE_EMPTY = 3, SITE_ACC = 4, SITE_TASK = 12, SITE_ACC_EMPTY = 13, SITE_LAUNCH = 14 };
enum : int { CMD_NONE = -1, CMD_EXIT = 0, CMD_COMPUTE = 1, CMD_COMM = 2 };

// One task of the pair: a compute task (arg = its index) or a communication task (arg for the
// even CTA, arg1 for the odd one; -1 = nothing for that CTA).
struct Task {
  int cmd, arg, arg1, pad;
};

// Shared control state of one CTA.
struct Smem {
  uint64_t full[kNStage], empty[kNStage];  // stage loaded (both CTAs' bytes; even CTA) / read by the MMAs
  uint64_t acc_full[kHalves], acc_empty[kHalves];  // accumulator half complete / read back (even CTA)
  uint64_t task_full[kSlots], task_empty[kSlots];  // task slot written / read by every reader (even CTA)
  uint64_t stg[16];                        // the communication role's buffers (kernel-specific)
  uint64_t drain;
  Task task[kSlots];
  uint32_t tmem_base;
  uint32_t peer_fills;  // the odd CTA's stage fills, reported at the end
  volatile uint32_t abort;
};

// Thread 0 of each CTA: the pipeline's barriers (the kernel initialises stg[] itself).
__device__ __forceinline__ void init_barriers(Smem* sc) {
  for (int s = 0; s < kNStage; ++s) {
    mbar_init(&sc->full[s], 1);
    mbar_init(&sc->empty[s], 1);
  }
  for (int b = 0; b < kHalves; ++b) {
    mbar_init(&sc->acc_full[b], 1);
    mbar_init(&sc->acc_empty[b], 2 * kEpiWarps);
  }
  for (int k = 0; k < kSlots; ++k) {
    mbar_init(&sc->task_full[k], 1);
    mbar_init(&sc->task_empty[k], kTaskReaders);
  }
  mbar_init(&sc->drain, 1);
  sc->peer_fills = 0;
  sc->abort = 0;
}

// Every thread, first: the kernel runs in clusters of two CTAs.  A launch without them (which
// no caller of launch_pairs makes) raises an error and returns before any distributed
// shared-memory access or pair allocation.
template <class KP>
__device__ __forceinline__ bool launched_as_pairs(const KP& p) {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  if (n == 2u) return true;
  if (threadIdx.x == 0) raise_error(p, SITE_LAUNCH);
  return false;
}

// Every thread of both CTAs, after init_barriers: tensor memory (512 columns per CTA, the pair's
// allocation), and both CTAs' barriers visible before any remote arrival.
__device__ __forceinline__ void setup_pair(Smem* sc) {
  if (threadIdx.x / 32 == 1) {
    tmem_alloc_cg<2>(&sc->tmem_base, 512);
    tmem_relinquish_cg<2>();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
}

// ------------------------------------------------------------------------------------------------
// Task ring
// ------------------------------------------------------------------------------------------------
// Scheduling thread (even CTA): publish task k to both CTAs.  False on timeout or abort.
template <class KP>
__device__ __forceinline__ bool post_task(const KP& p, Smem* sc, uint32_t k, const Task& t) {
  const uint32_t s = k % kSlots, use = k / kSlots;
  if (use > 0 && !wait_bar<true>(&sc->task_empty[s], (use - 1) & 1u, p, sc, SITE_TASK, kSlack)) return false;
  sc->task[s] = t;
  const uint32_t remote = mapa_shared(smem_u32(&sc->task[s]), 1);
  st_shared_cluster(remote, (uint32_t)t.cmd);
  st_shared_cluster(remote + 4, (uint32_t)t.arg);
  st_shared_cluster(remote + 8, (uint32_t)t.arg1);
  mbar_arrive(&sc->task_full[s]);
  mbar_arrive_cluster(mapa_shared(smem_u32(&sc->task_full[s]), 1));  // release: orders the stores above
  return true;
}

// A reader: wait for task k and read it.  False on timeout or abort.
template <class KP>
__device__ __forceinline__ bool take_task(const KP& p, Smem* sc, uint32_t k, Task& t) {
  const uint32_t s = k % kSlots;
  if (!wait_bar<true>(&sc->task_full[s], (k / kSlots) & 1u, p, sc, SITE_TASK, kSlack)) return false;
  const volatile Task* e = &sc->task[s];
  t.cmd = e->cmd;
  t.arg = e->arg;
  t.arg1 = e->arg1;
  t.pad = 0;
  return true;
}

// A reader is done with slot k (release: its reads of the slot come first).
__device__ __forceinline__ void release_task(Smem* sc, uint32_t k, uint32_t rank) {
  const uint32_t s = k % kSlots;
  if (rank == 0) mbar_arrive(&sc->task_empty[s]);
  else mbar_arrive_cluster(mapa_shared(smem_u32(&sc->task_empty[s]), 0));
}

// ------------------------------------------------------------------------------------------------
// Producer (thread 0 of each CTA), MMA issuer (one thread of the even CTA), epilogue warps
// ------------------------------------------------------------------------------------------------
// This CTA's share of a tile's K loop: A rows arow .. arow+127 of `ma` and, for half h, W rows
// wrow + 256h .. +127 of `mw`, n_k steps of kBK (stage layout: A, then the W rows of each half).
// `ahead()` runs once, after the loads of step `ahead_at` are issued (the scheduler decides its
// next task there).  `fills` counts the stage fills this CTA has issued.  False on timeout or
// abort.
template <class KP, class Ahead>
__device__ __forceinline__ bool load_tile(const KP& p, Smem* sc, uint32_t smem_base, uint32_t rank,
                                          const CUtensorMap* ma, int arow, const CUtensorMap* mw, int wrow, int n_k,
                                          uint32_t& fills, int ahead_at, Ahead&& ahead) {
  for (int ks = 0; ks < n_k; ++ks) {
    const uint32_t c = fills;
    const uint32_t s = c % kNStage, use = c / kNStage;
    if (use > 0 && !wait_bar(&sc->empty[s], (use - 1) & 1u, p, sc, SITE_EMPTY, kSlack)) return false;
    if (rank == 0) mbar_expect_tx(&sc->full[s], 2 * kStageBytes);  // both CTAs' bytes
    const uint32_t bar = mapa_shared(smem_u32(&sc->full[s]), 0);
    const uint32_t base = smem_base + s * kStageBytes;
    tma_load_2d_pair(base, ma, ks * kBK, arow, bar);
#pragma unroll
    for (int h = 0; h < kHalves; ++h) tma_load_2d_pair(base + (1 + h) * kHalf, mw, ks * kBK, wrow + h * kBN, bar);
    fills = c + 1;
    if (ks == ahead_at) ahead();
  }
  return true;
}

// Producer, before a communication task reuses the stage area: every stage this CTA filled
// has been read by the MMAs.  False on timeout or abort.
template <class KP>
__device__ __forceinline__ bool wait_stages_free(const KP& p, Smem* sc, uint32_t fills) {
  for (uint32_t s = 0; s < (uint32_t)kNStage && s < fills; ++s) {
    const uint32_t last = s + ((fills - 1 - s) / kNStage) * kNStage;  // the stage's last fill
    if (!wait_bar(&sc->empty[s], (last / kNStage) & 1u, p, sc, SITE_EMPTY, kSlack)) return false;
  }
  return true;
}

// MMA issuer: one tile's n_k stages into both halves, each waited for (acc_empty: its previous
// tile read back) just before the first product that overwrites it; acc_full on both CTAs per
// half at the end.  `fills` counts the stages consumed.  False on timeout or abort.
template <class KP>
__device__ __forceinline__ bool mma_tile(const KP& p, Smem* sc, uint32_t smem_base, int n_k, uint32_t& fills,
                                         uint32_t item) {
  constexpr uint32_t ID = idesc_bf16_f32(2 * kRows, kBN, false);
  constexpr uint32_t kHi = sdesc_hi_sw128(1024);  // 8-row groups 1024 B apart
  auto acquire = [&](int h) -> bool {
    if (item > 0 && !wait_bar<true>(&sc->acc_empty[h], (item - 1) & 1u, p, sc, SITE_ACC_EMPTY, kSlack)) return false;
    tc_fence_after();
    return true;
  };
  if (!acquire(0)) return false;
  for (int ks = 0; ks < n_k; ++ks) {
    const uint32_t c = fills;
    const uint32_t s = c % kNStage;
    if (!wait_bar(&sc->full[s], (c / kNStage) & 1u, p, sc, SITE_FULL, kSlack)) return false;
    tc_fence_after();
    const uint32_t base = smem_base + s * kStageBytes;
    const uint32_t a_lo = sdesc_lo(base, 16);
#pragma unroll
    for (int h = 0; h < kHalves; ++h) {
      if (h > 0 && ks == 0 && !acquire(h)) return false;
      const uint32_t w_lo = sdesc_lo(base + (1 + h) * kHalf, 16);
      const uint32_t tacc = sc->tmem_base + h * kBN;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        mma_ss_cg<2>(tacc, a_lo + kk * 2, kHi, w_lo + kk * 2, kHi, ID, (ks > 0 || kk > 0) ? 1u : 0u);
    }
    mma_commit_cg<2>(&sc->empty[s], 3);
    fills = c + 1;
  }
#pragma unroll
  for (int h = 0; h < kHalves; ++h) mma_commit_cg<2>(&sc->acc_full[h], 3);
  return true;
}

// Epilogue warp: for each half of the tile it waits for the half, reads this warp's 32 rows x 128
// columns of it as two 64-column blocks, releases the half once both are in registers, and
// hands each block to store(cb, v[64]).  Block cb covers the tile's columns
// 256*(cb/2) + 128*chalf + 64*(cb%2) .. (chalf = (warp-4)/4); v holds raw fp32 bits; the thread's
// row inside the CTA's 128 is 32*(warp%4) + lane.  False on timeout or abort.
template <class KP, class Store>
__device__ __forceinline__ bool read_acc(const KP& p, Smem* sc, uint32_t rank, uint32_t item, Store&& store) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quarter = warp % 4, chalf = (warp - 4) / 4;
#pragma unroll 1
  for (int h = 0; h < kHalves; ++h) {
    const bool ok = __all_sync(0xffffffffu, wait_bar(&sc->acc_full[h], item & 1u, p, sc, SITE_ACC, kSlack));
    if (!ok) { sc->abort = 1; return false; }
    tc_fence_after();
    const uint32_t tacc = sc->tmem_base + ((uint32_t)(quarter * 32) << 16) + h * kBN + chalf * 128;
    uint32_t v[64];
    tmem_ld64(tacc, v);
    tmem_ld_wait();
    store(2 * h, v);
    tmem_ld64(tacc + 64, v);
    tmem_ld_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (rank == 0) mbar_arrive(&sc->acc_empty[h]);
      else mbar_arrive_cluster(mapa_shared(smem_u32(&sc->acc_empty[h]), 0));
    }
    store(2 * h + 1, v);
  }
  return true;
}

// Coalesced store of one block of a warp's 32 rows (the 32x32b tensor-memory load gives each
// thread one row).  Each thread hands W 32-bit words of its row; the warp writes them into its
// shared-memory staging area (32 x 4W bytes) with the 16-byte chunks XOR-swizzled by row,
// reads them back row-contiguous, and stores whole 4W-byte row segments (W/4 lanes per row
// instead of one lane per row).  Both shared-memory passes are free of bank conflicts.
// `gbase` is the byte address of the block in the warp's first row, `stride` the row pitch.
template <int W>
__device__ __forceinline__ void warp_store_rows(uint8_t* stage, const uint32_t* words, uint8_t* gbase, size_t stride) {
  constexpr int R = W / 4;     // 16-byte chunks per row segment
  constexpr int RPI = 32 / R;  // rows per read-back instruction
  const int lane = threadIdx.x % 32;
#pragma unroll
  for (int j = 0; j < R; ++j)
    *reinterpret_cast<uint4*>(stage + lane * (4 * W) + ((j ^ (lane % R)) * 16)) =
        make_uint4(words[4 * j], words[4 * j + 1], words[4 * j + 2], words[4 * j + 3]);
  __syncwarp();
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const int r = k * RPI + lane / R, c = lane % R;
    const uint4 v = *reinterpret_cast<const uint4*>(stage + r * (4 * W) + ((c ^ (r % R)) * 16));
    *reinterpret_cast<uint4*>(gbase + (size_t)r * stride + c * 16) = v;
  }
  __syncwarp();  // the staging area is reused for the next block
}

// End of the kernel (every thread of both CTAs).  `fills` is thread 0's count of the stage
// fills its CTA issued.  Every tcgen05 op has completed and every TMA load into either CTA's
// stages has landed (bounded waits) before tensor memory is released and either CTA exits.
// The loads of both CTAs count on the even CTA's barriers; after an abort the two producers
// may have issued different numbers of fills (at most one apart per stage), so the even CTA
// completes each stage's last phase itself: it arms a phase only the odd CTA loaded, and
// accounts for the odd CTA's bytes of a phase that only it loaded.
__device__ __forceinline__ void drain_pair(Smem* sc, uint32_t rank, uint32_t fills) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (warp == 1 && lane == 0 && rank == 0) {
    mma_commit_cg<2>(&sc->drain, 1);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(&sc->drain, 0)) {
      if (globaltimer_ns() - t0 > 100000000ull) break;
    }
  }
  if (threadIdx.x == 0 && rank == 1) st_shared_cluster(mapa_shared(smem_u32(&sc->peer_fills), 0), fills);
  __syncthreads();
  cluster_sync();
  if (threadIdx.x == 0 && rank == 0) {
    const uint32_t L = fills, Q = sc->peer_fills, F = L > Q ? L : Q;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t s = 0; s < (uint32_t)kNStage && s < F; ++s) {
      const uint32_t m = s + ((F - 1 - s) / kNStage) * kNStage;  // the stage's last fill by either CTA
      if (m >= L) mbar_expect_tx(&sc->full[s], kStageBytes);         // armed by no one: the odd CTA's bytes
      else if (m >= Q) mbar_complete_tx(&sc->full[s], kStageBytes);  // the odd CTA's bytes will not come
      while (!mbar_try_wait(&sc->full[s], (m / kNStage) & 1u) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the other may still signal it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_cg<2>(sc->tmem_base, 512);
}

// ------------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------------
// cuTensorMapEncodeTiled from the driver (looked up once), or null.
inline PFN_cuTensorMapEncodeTiled_v12000 encode_tiled_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Tensor map of a [rows][K] bf16 matrix (K-major): boxes of 64 columns x box_rows rows,
// 128-byte swizzle.
inline bool tmap_kmajor(CUtensorMap* m, const void* base, long long rows, int K, int box_rows) {
  const auto encode = encode_tiled_fn();
  if (!encode) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTAs of a pair kernel that can all be resident at once: whole pairs, no more than the SMs
// and the device's co-resident clusters allow (0 on error).  Computed once per kernel.
template <class Kern>
inline int pair_ctas(Kern kern, int n_sm) {
  static std::once_flag once;
  static int n_ok = 0;
  std::call_once(once, [kern, n_sm] {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_sm / 2 * 2));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int max_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    n_ok = 2 * max_clusters < n_sm / 2 * 2 ? 2 * max_clusters : n_sm / 2 * 2;
  });
  return n_ok;
}

// Launch n_cta CTAs (whole pairs, all co-resident: pair_ctas) as clusters of two.  The grid is
// no larger than the clusters the device holds at once, one CTA per SM, so every pair is resident
// from the start (the roles wait on one another, with bounded waits).
template <class Kern, class... Args>
inline cudaError_t launch_pairs(Kern kern, int n_cta, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_cta);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace gemm
}  // namespace psr
