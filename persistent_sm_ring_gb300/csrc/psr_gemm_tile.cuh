// The 256 x 256 output tile of the persistent GEMM kernels (AllGather+GEMM and
// GEMM+ReduceScatter) on sm_103a.
//
//  * a ring of kNStage shared-memory stages, each holding two 128-row A tiles and one 256-row
//    W tile of one 64-wide K step (both K-major, loaded by TMA with the 128-byte swizzle);
//  * one elected thread issues tcgen05.mma (M = 128, N = 256, K = 16) for both 128-row halves
//    of the tile, with both fp32 accumulators in tensor memory (2 x 256 columns), and commits
//    each stage back to the producer as soon as its MMAs have read it;
//  * two warpgroups read the accumulators back with tcgen05.ld, one 128-row half each (tensor
//    memory lane = tile row), in 64-column blocks handed to a kernel-specific store.
// Each kernel adds its own task selection, data dependencies and epilogue destination.
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

constexpr int kBM = 256;          // output rows per tile (two 128-row A tiles)
constexpr int kBN = 256;          // output columns per tile (one W tile)
constexpr int kBK = 64;           // K per stage (one 128-byte swizzle atom of bf16)
constexpr int kNStage = 3;        // stages of A0 | A1 | W
constexpr int kATile = 128 * kBK * 2;   // 16 KiB
constexpr int kWTile = kBN * kBK * 2;   // 32 KiB
constexpr int kStageBytes = 2 * kATile + kWTile;
constexpr int kStageArea = kNStage * kStageBytes;  // also the scratch of the copy / reduce roles
constexpr int kSmem = 1024 + kStageArea;
constexpr int kWarps = 12, kThreads = kWarps * 32;
static_assert(kSmem <= 232448 - 512, "shared memory");

// Shared control state of one CTA.
struct Smem {
  uint64_t full[kNStage], empty[kNStage];  // stage loaded (TMA bytes) / stage read by the MMAs
  uint64_t acc_full;                       // accumulators of the current tile complete
  uint64_t stg[16];                        // the other role's buffers (kernel-specific)
  uint64_t drain;
  uint32_t tmem_base;
  int cmd, arg;
  volatile uint32_t abort;
};

// Running counts over the CTA's lifetime; every role advances its own copy identically,
// so mbarrier phases agree across roles.
struct Counters {
  uint32_t fills;  // stage fills issued (producer) / consumed (issuer)
  uint32_t items;  // tiles completed (accumulator phase)
};

// Producer (one thread): the K loop of one tile, A rows arow .. arow+255 of `ma` and W rows
// wrow .. wrow+255 of `mw`, n_k steps of kBK.  False on timeout or abort.
template <class KP>
__device__ __forceinline__ bool load_tile(const KP& p, Smem* sc, uint32_t smem_base, const CUtensorMap* ma, int arow,
                                          const CUtensorMap* mw, int wrow, int n_k, Counters& cnt,
                                          uint32_t site_empty) {
  for (int ks = 0; ks < n_k; ++ks) {
    const uint32_t c = cnt.fills++;
    const uint32_t s = c % kNStage, fill = c / kNStage;
    if (fill > 0 && !wait_bar(&sc->empty[s], (fill - 1) & 1u, p, sc, site_empty)) return false;
    const uint32_t base = smem_base + s * kStageBytes;
    mbar_expect_tx(&sc->full[s], kStageBytes);
    tma_load_2d(base, ma, ks * kBK, arow, &sc->full[s]);
    tma_load_2d(base + kATile, ma, ks * kBK, arow + 128, &sc->full[s]);
    tma_load_2d(base + 2 * kATile, mw, ks * kBK, wrow, &sc->full[s]);
  }
  return true;
}

// MMA issuer (one thread): n_k stages into the two accumulators, then acc_full.
template <class KP>
__device__ __forceinline__ void mma_tile(const KP& p, Smem* sc, uint32_t smem_base, int n_k, Counters& cnt,
                                         uint32_t site_full) {
  constexpr uint32_t ID = idesc_bf16_f32(128, kBN, false);
  constexpr uint32_t kHi = sdesc_hi_sw128(1024);
  for (int ks = 0; ks < n_k; ++ks) {
    const uint32_t c = cnt.fills++;
    const uint32_t s = c % kNStage, fill = c / kNStage;
    if (!wait_bar(&sc->full[s], fill & 1u, p, sc, site_full)) { sc->abort = 1; return; }
    tc_fence_after();
    const uint32_t base = smem_base + s * kStageBytes;
    const uint32_t w_lo = sdesc_lo(base + 2 * kATile, 16);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t a_lo = sdesc_lo(base + i * kATile, 16);
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        mma_ss_w(sc->tmem_base + i * kBN, a_lo + kk * 2, kHi, w_lo + kk * 2, kHi, ID, (ks > 0 || kk > 0) ? 1u : 0u);
    }
    mma_commit(&sc->empty[s]);
  }
  mma_commit(&sc->acc_full);
}

// Epilogue warpgroup for 128-row half i of the tile: waits for the accumulators, then hands
// each 64-column block of this thread's row (row = 0..127 inside the half) to
// store(row, cb, v[64]) as raw fp32 bits.  False on timeout or abort.
template <class KP, class Store>
__device__ __forceinline__ bool read_tile(const KP& p, Smem* sc, int i, const Counters& cnt, uint32_t site_acc,
                                          Store&& store) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quarter = warp % 4;
  const int row = quarter * 32 + lane;
  const bool ok = __all_sync(0xffffffffu, wait_bar(&sc->acc_full, cnt.items & 1u, p, sc, site_acc));
  if (!ok) { sc->abort = 1; return false; }
  tc_fence_after();
  const uint32_t tacc = sc->tmem_base + ((uint32_t)(quarter * 32) << 16) + i * kBN;
#pragma unroll 1
  for (int cb = 0; cb < kBN / 64; ++cb) {
    uint32_t v[64];
    tmem_ld64(tacc + cb * 64, v);
    tmem_ld_wait();
    store(row, cb, v);
  }
  return true;
}

// Coalesced store of one 64-column block of a warp's 32 rows (the 32x32b tensor-memory load gives
// each thread one row).  Each thread hands W 32-bit words of its row (W = 64: fp32; W = 32: bf16
// pairs); the warp writes them into its shared-memory staging area (32 x 4W bytes) with the
// 16-byte chunks XOR-swizzled by row, reads them back row-contiguous, and stores whole 4W-byte row
// segments: 16 (fp32) or 8 (bf16) lanes per row instead of one lane per row.  Both shared-memory
// passes are free of bank conflicts.  `gbase` is the byte address of the block in the warp's
// first row, `stride` the row pitch in bytes.
template <int W>
__device__ __forceinline__ void warp_store_rows(uint8_t* stage, const uint32_t* words, uint8_t* gbase, size_t stride) {
  constexpr int R = W / 4;        // 16-byte chunks per row segment
  constexpr int RPI = 32 / R;     // rows per read-back instruction
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

// End of the kernel (all threads): every tcgen05 op has completed and every TMA load into
// the stages has landed (bounded waits) before tensor memory is released.
__device__ __forceinline__ void drain_and_release(Smem* sc, const Counters& cnt) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (warp == 1 && lane == 0) {
    mma_commit(&sc->drain);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(&sc->drain, 0)) {
      if (globaltimer_ns() - t0 > 100000000ull) break;
    }
  }
  if (threadIdx.x == 0) {
    bulk_wait<0>();
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t s = 0; s < (uint32_t)kNStage && s < cnt.fills; ++s) {
      const uint32_t fills = (cnt.fills - s + kNStage - 1) / kNStage;
      while (!mbar_try_wait(&sc->full[s], (fills - 1) & 1u) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(sc->tmem_base, 512);
}

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

}  // namespace gemm
}  // namespace psr
