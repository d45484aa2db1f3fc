// Ring Attention backward on sm_103a.
//
// The gradient of the forward step in psr_ring_attn.cu (the mKernel pages describe only the
// forward; the backward follows the same ring and reuses its log-sum-exp).  With the forward's
// LSE and D_i = dO_i . O_i, for each (query row i, key j) that the mask allows:
//     P_ij = exp(scale q_i.k_j - LSE_i),   dP_ij = dO_i . v_j,   dS_ij = P_ij (dP_ij - D_i),
//     dV_j += P_ij dO_i,   dK_j += scale dS_ij q_i,   dQ_i += scale dS_ij k_j.
// In the ring, each KV chunk travels around the ranks together with its dK / dV partial sums
// while every rank keeps its queries; the partials are back at the owner after P steps.  On one
// GPU two persistent kernels follow the two data flows:
//
//  * dK, dV (K/V-stationary): an item holds one 128-row K/V tile and its dK / dV accumulators
//    in tensor memory for the whole ring, visiting the query shards in ring order (its own
//    shard first, then r+1, r+2, ...); per query tile, with the key rows on the lanes:
//        S^T = K Q^T, dP^T = V dO^T (SS)  ->  P^T, dS^T in place (bf16)  ->
//        dV += P^T dO, dK += dS^T Q (TS)
//  * dQ (Q-stationary, the forward's ring order): an item holds one 128-row query tile and its
//    dQ accumulator; per K/V tile, with the query rows on the lanes:
//        S = Q K^T, dP = dO V^T (SS)  ->  dS in place (bf16)  ->  dQ += dS K (TS)
//
// dQ could also be accumulated by the first kernel with atomic adds, saving the second
// kernel's S and dP products; on GB300 those fp32 atomics (64 KiB per tile pair) ran at
// ~1.6 TB/s and bounded the whole pass (41 ms per causal B1 H32 S32768 pass, against 27.5 ms
// with the second kernel).  In each kernel one thread
// issues every MMA; tensor-core instructions of one thread run in order, so an MMA that
// overwrites columns another MMA reads is simply issued after it.  Two warpgroups share the
// elementwise work, each on half of the columns, and each writes its bf16 results over its own
// fp32 columns (the MMAs take the operand from the two column ranges), so they never wait for
// each other.
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

namespace psr {
namespace bwd {

constexpr int kRows = 128;                 // rows of a query tile and of a K/V tile
constexpr int kThreads = 384;
constexpr float kLog2e = 1.4426950408889634f;

enum : uint32_t { SITE_KV = 21, SITE_Q_FULL = 22, SITE_Q_EMPTY = 23, SITE_S = 24, SITE_DP = 25, SITE_P = 26,
                  SITE_DS = 27, SITE_ACC = 29, SITE_KV_EMPTY = 30 };

struct BParams {
  int B, Hq, Hkv, S, P, L, gqa, causal;
  int balanced;         // causal over load-balanced shards (shard r holds half-chunks r and 2P-1-r)
  int tiles_per_shard;  // L / 128
  int n_items_kv;       // B * Hkv * (S / 128)
  int n_items_q;        // B * Hq * (S / 128)
  float sl2;            // scale * log2(e)
  float scale;
  const float* nlse2;   // [B][Hq][S] -LSE * log2(e) (LSE: the forward's natural-log log-sum-exp)
  const float* ndelta;  // [B][Hq][S] -D = -rowsum(dO * O)
  uint16_t* dq;         // [B][Hq][S][d] bf16
  uint16_t* dk;         // [B][Hkv][S][d] bf16
  uint16_t* dv;
  Ctrl* ctrl;
  unsigned long long timeout_ns;
};

// Global position (in 128-row tiles) of stored tile g, and its inverse.  Contiguous shards: g
// itself.  Load-balanced shards: local tiles [0, T/2) of shard r are half-chunk r, local tiles
// [T/2, T) half-chunk 2P-1-r (T = tiles per shard); positions rise inside a tile and a shard.
__device__ __forceinline__ int tile_pos(const BParams& p, int g) {
  if (!p.balanced) return g;
  const int T = p.tiles_per_shard, h = T / 2, r = g / T, lt = g % T;
  return lt < h ? r * h + lt : (2 * p.P - 1 - r) * h + (lt - h);
}
__device__ __forceinline__ int tile_at_pos(const BParams& p, int pos) {
  if (!p.balanced) return pos;
  const int T = p.tiles_per_shard, h = T / 2, c = pos / h, o = pos % h;
  return c < p.P ? c * T + o : (2 * p.P - 1 - c) * T + h + o;
}

__host__ __device__ constexpr uint32_t idesc_ab(uint32_t M, uint32_t N, bool a_mn, bool b_mn) {
  return idesc_bf16_f32(M, N, b_mn) | ((a_mn ? 1u : 0u) << 15);
}

// Shared-memory descriptors of a [128 rows][D cols] tile stored as D/64 boxes of 16 KiB
// (128-byte swizzle): K-major use (rows = M or N, K = columns) for the 16-column step kk, and
// MN-major use (rows = K, columns = M or N) for the 16-row step kk.
__device__ __forceinline__ uint32_t kmaj_lo(uint32_t tile, int kk) {
  return sdesc_lo(tile + (kk / 4) * 16384 + (kk % 4) * 32, 16);
}
__device__ __forceinline__ uint32_t mnmaj_lo(uint32_t tile, int kk) { return sdesc_lo(tile + kk * 2048, 16384); }

// TMEM column of the bf16 A operand (P^T, dS^T or dS) for the 16-element K step kk: warpgroup w
// writes its 64 elements as 32 bf16 pairs into the low half of its own 64 fp32 columns
// [64w, 64w + 64), so neither warpgroup overwrites columns the other still reads.
__device__ __forceinline__ uint32_t bf16_col(int kk) { return (kk / 4) * 64 + (kk % 4) * 8; }

__device__ __forceinline__ void unpack_bf16x2(uint32_t v, float& lo, float& hi) {
  lo = __uint_as_float(v << 16);
  hi = __uint_as_float(v & 0xFFFF0000u);
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ================================================================================================
// dK, dV: K/V-stationary
// ================================================================================================
template <int D>
struct KvCfg {
  static constexpr int TILE = kRows * D * 2;
  static constexpr int OFF_K = 0, OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;      // + qb * TILE
  static constexpr int OFF_DO = 4 * TILE;     // + qb * TILE
  static constexpr int OFF_LD = 6 * TILE;     // + qb * 1024: -LSE*log2(e)[128] then -D[128] (fp32)
  static constexpr int SMEM = 1024 + OFF_LD + 2 * 1024;
  static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 256 + D;
  static_assert(SMEM <= 232448 - 1024, "shared memory");
};

struct KvSmem {
  uint64_t kv_full, q_full[2], q_empty[2], s_full, dp_full, p_ready, ds_ready, acc_full, drain;
  uint32_t tmem_base;
  int arg;
  volatile uint32_t abort;
};

struct KvItem {
  int b, kvh, gk;  // batch, KV head, K/V tile (global 128-row index)
};
__device__ inline KvItem kv_item_of(const BParams& p, int n) {
  KvItem it;
  it.gk = tile_at_pos(p, n / (p.B * p.Hkv));  // the earliest positions have the most causal work: first
  const int rest = n % (p.B * p.Hkv);
  it.b = rest / p.Hkv;
  it.kvh = rest % p.Hkv;
  return it;
}

// The item's (query head, query tile) pairs in ring order: shard j of the K/V tile first, then
// j+1, j+2, ... (mod P); under the causal mask only query tiles at or after the K/V tile's
// position (with contiguous shards no tile of a shard before j qualifies; with load-balanced
// shards the qualifying tiles of each half-chunk are a suffix of it, visited directly).
template <class F>
__device__ __forceinline__ void for_each_q(const BParams& p, const KvItem& it, F&& f) {
  const int j = it.gk / p.tiles_per_shard;
  const int kpos = tile_pos(p, it.gk);
  const int hh = p.tiles_per_shard / 2;
  for (int t = 0; t < p.P; ++t) {
    const int r = (j + t) % p.P;
    if (p.causal && !p.balanced && r < j) continue;
    for (int h = 0; h < p.gqa; ++h) {
      const int hq = it.kvh * p.gqa + h;
      if (p.causal && p.balanced) {
        // local tiles [0, hh) hold positions r*hh + o, tiles [hh, 2hh) positions (2P-1-r)*hh + o
        for (int half = 0; half < 2; ++half) {
          const int c = half ? 2 * p.P - 1 - r : r;
          const int o0 = kpos - c * hh > 0 ? kpos - c * hh : 0;
          for (int o = o0; o < hh; ++o)
            if (!f(hq, r * p.tiles_per_shard + half * hh + o, c * hh + o == kpos)) return;
        }
        continue;
      }
      for (int qt = 0; qt < p.tiles_per_shard; ++qt) {
        const int gq = r * p.tiles_per_shard + qt;
        const int qpos = tile_pos(p, gq);
        if (p.causal && qpos < kpos) continue;
        if (!f(hq, gq, p.causal && qpos == kpos)) return;
      }
    }
  }
}

template <int D>
__device__ void kv_producer(const BParams& p, KvSmem* sc, uint32_t sbase, const KvItem& it, const CUtensorMap* tq,
                            const CUtensorMap* tdo, const CUtensorMap* tk, const CUtensorMap* tv, uint32_t& qcnt) {
  using C = KvCfg<D>;
  const int kv_row = (it.b * p.Hkv + it.kvh) * p.S + it.gk * kRows;
  mbar_expect_tx(&sc->kv_full, 2 * C::TILE);
#pragma unroll
  for (int h = 0; h < D / 64; ++h) {
    tma_load_2d(sbase + C::OFF_K + h * 16384, tk, 64 * h, kv_row, &sc->kv_full);
    tma_load_2d(sbase + C::OFF_V + h * 16384, tv, 64 * h, kv_row, &sc->kv_full);
  }
  for_each_q(p, it, [&](int hq, int gq, bool) -> bool {
    const uint32_t qb = qcnt % 2, fill = qcnt / 2;
    if (fill > 0 && !wait_bar(&sc->q_empty[qb], (fill - 1) & 1u, p, sc, SITE_Q_EMPTY)) return false;
    const int q_row = (it.b * p.Hq + hq) * p.S + gq * kRows;
    const uint32_t ld = sbase + C::OFF_LD + qb * 1024;
    mbar_expect_tx(&sc->q_full[qb], 2 * C::TILE + 1024);
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      tma_load_2d(sbase + C::OFF_Q + qb * C::TILE + h * 16384, tq, 64 * h, q_row, &sc->q_full[qb]);
      tma_load_2d(sbase + C::OFF_DO + qb * C::TILE + h * 16384, tdo, 64 * h, q_row, &sc->q_full[qb]);
    }
    bulk_load(ld, p.nlse2 + q_row, 512, &sc->q_full[qb]);
    bulk_load(ld + 512, p.ndelta + q_row, 512, &sc->q_full[qb]);
    ++qcnt;
    return true;
  });
}

// Order per query tile j: dP^T(j), dV(j), S^T(j+1), dK(j); S^T(j+1) is issued as soon as dV(j)
// has been issued (it reads P^T(j) from the columns S^T(j+1) overwrites), so that the tensor
// core computes it while the warpgroups form dS^T(j).
template <int D>
__device__ void kv_mma(const BParams& p, KvSmem* sc, uint32_t sbase, const KvItem& it, uint32_t items, uint32_t& qcnt,
                       uint32_t& jg) {
  using C = KvCfg<D>;
  constexpr uint32_t I_SS = idesc_ab(128, 128, false, false);
  constexpr uint32_t I_TS = idesc_ab(128, D, false, true);
  constexpr uint32_t kHi = sdesc_hi_sw128(1024);
  const uint32_t tm = sc->tmem_base;
  const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  int n_pairs = 0;
  for_each_q(p, it, [&](int, int, bool) -> bool { ++n_pairs; return true; });
  if (!wait_bar(&sc->kv_full, items & 1u, p, sc, SITE_KV)) { sc->abort = 1; return; }
  auto issue_s = [&](uint32_t c) -> bool {  // S^T of the pair with load index c
    if (!wait_bar(&sc->q_full[c % 2], (c / 2) & 1u, p, sc, SITE_Q_FULL)) return false;
    tc_fence_after();
    const uint32_t sQ = sbase + C::OFF_Q + (c % 2) * C::TILE;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      mma_ss_w(tm + C::COL_S, kmaj_lo(sK, kk), kHi, kmaj_lo(sQ, kk), kHi, I_SS, kk > 0 ? 1u : 0u);
    mma_commit(&sc->s_full);
    return true;
  };
  if (!issue_s(qcnt)) { sc->abort = 1; return; }
  int i = 0;
  for_each_q(p, it, [&](int, int, bool) -> bool {
    const uint32_t qb = qcnt % 2;
    const uint32_t sQ = sbase + C::OFF_Q + qb * C::TILE, sDO = sbase + C::OFF_DO + qb * C::TILE;
    // dP^T = V dO^T (its columns held dS^T of the previous tile, read by that tile's dK MMA)
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      mma_ss_w(tm + C::COL_DP, kmaj_lo(sV, kk), kHi, kmaj_lo(sDO, kk), kHi, I_SS, kk > 0 ? 1u : 0u);
    mma_commit(&sc->dp_full);
    if (!wait_bar(&sc->p_ready, jg & 1u, p, sc, SITE_P)) return false;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < kRows / 16; ++kk)
      mma_ts_w(tm + C::COL_DV, tm + C::COL_S + bf16_col(kk), mnmaj_lo(sDO, kk), kHi, I_TS, (i == 0 && kk == 0) ? 0u : 1u);
    if (i + 1 < n_pairs && !issue_s(qcnt + 1)) return false;
    if (!wait_bar(&sc->ds_ready, jg & 1u, p, sc, SITE_DS)) return false;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < kRows / 16; ++kk)
      mma_ts_w(tm + C::COL_DK, tm + C::COL_DP + bf16_col(kk), mnmaj_lo(sQ, kk), kHi, I_TS, (i == 0 && kk == 0) ? 0u : 1u);
    mma_commit(&sc->q_empty[qb]);  // Q, dO of this tile are read (LSE, D: the warpgroups are past them)
    ++qcnt;
    ++jg;
    ++i;
    return true;
  });
  if (i != n_pairs) { sc->abort = 1; return; }
  mma_commit(&sc->acc_full);
}

// Warpgroup w (warps 4..7: w = 0, warps 8..11: w = 1): the K/V tile's rows on the lanes, query
// columns [64w, 64w + 64).
template <int D>
__device__ void kv_elementwise(const BParams& p, KvSmem* sc, const uint8_t* smem, const KvItem& it, uint32_t items,
                               uint32_t& jg) {
  using C = KvCfg<D>;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int w = warp >= 8 ? 1 : 0;
  const int quarter = warp % 4;
  const int row = quarter * 32 + lane;  // K/V row of the tile
  const uint32_t lanes = sc->tmem_base + ((uint32_t)(quarter * 32) << 16);
  bool ok = true;
  for_each_q(p, it, [&](int, int, bool diag) -> bool {
    // -LSE*log2(e) and -D of this warpgroup's 64 query columns, as fp32 pairs
    const uint64_t* nl2 = reinterpret_cast<const uint64_t*>(smem + C::OFF_LD + (jg % 2) * 1024) + 32 * w;
    const uint64_t* nd2 = nl2 + 64;
    ok = __all_sync(0xffffffffu, wait_bar(&sc->q_full[jg % 2], (jg / 2) & 1u, p, sc, SITE_Q_FULL));
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(&sc->s_full, jg & 1u, p, sc, SITE_S));
    if (!ok) return false;
    tc_fence_after();
    uint32_t pk[32];  // P^T of this row over the warpgroup's 64 query columns, bf16 pairs
    const uint64_t sl2 = f2_pack(p.sl2, p.sl2);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t s[32];
      tmem_ld32(lanes + C::COL_S + 64 * w + 32 * c, s);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        // log2-domain exponent of the pair: s * scale * log2(e) - LSE * log2(e)
        float x0, x1;
        f2_unpack(fma2(f2_pack(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), sl2, nl2[16 * c + e / 2]), x0, x1);
        pk[16 * c + e / 2] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
      }
      if (diag) {  // diagonal tile: keys after the query are masked (query column < key row)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int col = 64 * w + 32 * c + e;
          if (col + 1 < row) pk[16 * c + e / 2] = 0u;
          else if (col < row) pk[16 * c + e / 2] &= 0xFFFF0000u;
        }
      }
    }
    // P^T as bf16 pairs over the low half of this warpgroup's own S^T columns
    tmem_st16(lanes + C::COL_S + 64 * w, pk);
    tmem_st16(lanes + C::COL_S + 64 * w + 16, pk + 16);
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sc->p_ready);
    ok = __all_sync(0xffffffffu, wait_bar(&sc->dp_full, jg & 1u, p, sc, SITE_DP));
    if (!ok) return false;
    tc_fence_after();
    uint32_t ds[32];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t dp[32];
      tmem_ld32(lanes + C::COL_DP + 64 * w + 32 * c, dp);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float p0, p1, d0, d1;
        unpack_bf16x2(pk[16 * c + e / 2], p0, p1);
        // dS = P (dP - D) for the pair
        f2_unpack(mul2(f2_pack(p0, p1), add2(f2_pack(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])),
                                             nd2[16 * c + e / 2])),
                  d0, d1);
        ds[16 * c + e / 2] = pack_bf16x2(d0, d1);
      }
    }
    // dS^T as bf16 pairs over the low half of this warpgroup's own dP^T columns
    tmem_st16(lanes + C::COL_DP + 64 * w, ds);
    tmem_st16(lanes + C::COL_DP + 64 * w + 16, ds + 16);
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sc->ds_ready);
    ++jg;
    return true;
  });
  if (!ok) { sc->abort = 1; return; }
  // the item's dK and dV rows: this warpgroup's half of the columns
  ok = __all_sync(0xffffffffu, wait_bar(&sc->acc_full, items & 1u, p, sc, SITE_ACC));
  if (!ok) { sc->abort = 1; return; }
  tc_fence_after();
  const size_t out_row = ((size_t)(it.b * p.Hkv + it.kvh) * p.S + (size_t)it.gk * kRows + row) * D;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const uint32_t col = (which ? C::COL_DK : C::COL_DV) + w * (D / 2);
    const float mul = which ? p.scale : 1.0f;
    uint16_t* dst = (which ? p.dk : p.dv) + out_row + w * (D / 2);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      uint32_t v[32], o[16];
      tmem_ld32(lanes + col + 32 * c, v);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 16; ++e) o[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        reinterpret_cast<uint4*>(dst + 32 * c)[e] = make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kv_kernel(const __grid_constant__ BParams p, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ KvSmem sc;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  const uint8_t* smem = smem_raw + (sbase - raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(&sc.kv_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sc.q_full[b], 1);
      mbar_init(&sc.q_empty[b], 1);
    }
    mbar_init(&sc.s_full, 1);
    mbar_init(&sc.dp_full, 1);
    mbar_init(&sc.p_ready, 8);   // the eight warps of the two elementwise warpgroups
    mbar_init(&sc.ds_ready, 8);
    mbar_init(&sc.acc_full, 1);
    mbar_init(&sc.drain, 1);
    sc.abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_do);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(&sc.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  uint32_t items = 0, qcnt_p = 0, qcnt_m = 0, jg_m = 0, jg_e = 0;
  while (true) {
    if (threadIdx.x == 0) {
      int n = -1;
      if (!sc.abort && !ld_relaxed(&p.ctrl->abort)) {
        const uint32_t t = atomicAdd(&p.ctrl->item_next, 1u);
        if (t < (uint32_t)p.n_items_kv) n = (int)t;
      }
      sc.arg = n;
    }
    __syncthreads();
    const int n = sc.arg;
    if (n < 0) break;
    const KvItem it = kv_item_of(p, n);
    if (warp == 0 && lane == 0) {
      kv_producer<D>(p, &sc, sbase, it, &tm_q, &tm_do, &tm_k, &tm_v, qcnt_p);
    } else if (warp == 1 && lane == 0) {
      kv_mma<D>(p, &sc, sbase, it, items, qcnt_m, jg_m);
    } else if (warp >= 4) {
      kv_elementwise<D>(p, &sc, smem, it, items, jg_e);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0 && !sc.abort) atomicAdd(&p.ctrl->compute_items, 1ull);
    ++items;
    if (sc.abort) break;
  }
  // drain (bounded): every MMA has completed and every TMA load has landed
  if (warp == 1 && lane == 0) {
    mma_commit(&sc.drain);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(&sc.drain, 0) && globaltimer_ns() - t0 < 100000000ull) {
    }
  }
  if (warp == 0 && lane == 0) {
    const uint64_t t0 = globaltimer_ns();
    if (items > 0)
      while (!mbar_try_wait(&sc.kv_full, (items - 1) & 1u) && globaltimer_ns() - t0 < 100000000ull) {
      }
    for (uint32_t b = 0; b < 2 && b < qcnt_p; ++b) {
      const uint32_t fills = (qcnt_p - b + 1) / 2;
      while (!mbar_try_wait(&sc.q_full[b], (fills - 1) & 1u) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(sc.tmem_base, 512);
}

// ================================================================================================
// dQ: Q-stationary
// ================================================================================================
template <int D>
struct QCfg {
  static constexpr int TILE = kRows * D * 2;
  // K tiles in three buffers, V tiles in two: K(j) is read until dQ(j), V(j) only until dP(j),
  // and the S product of a tile is issued a tile ahead, so a third K buffer lets each K load
  // start a whole tile before it is needed
  static constexpr int KST = 3, VST = 2;
  static constexpr int OFF_Q = 0, OFF_DO = TILE;
  static constexpr int OFF_K = 2 * TILE;           // + kb * TILE
  static constexpr int OFF_V = (2 + KST) * TILE;   // + vb * TILE
  static constexpr int SMEM = 1024 + (2 + KST + VST) * TILE;
  static constexpr uint32_t COL_S = 0;        // + (tile % 2) * 128: S double-buffered
  static constexpr uint32_t COL_DP = 256, COL_DQ = 384;
  static_assert(SMEM <= 232448 - 1024, "shared memory");
};

struct QSmem {
  uint64_t qd_full, k_full[3], k_empty[3], v_full[2], v_empty[2], s_full[2], dp_full, ds_ready, acc_full, drain;
  uint32_t tmem_base;
  int arg;
  volatile uint32_t abort;
};

struct QItem {
  int b, hq, gq;  // batch, query head, query tile (global 128-row index)
};
__device__ inline QItem q_item_of(const BParams& p, int n) {
  QItem it;
  const int per = p.B * p.Hq;
  // causal: the last query positions (most keys) first
  it.gq = tile_at_pos(p, p.causal ? (p.S / kRows - 1 - n / per) : n / per);
  const int rest = n % per;
  it.b = rest / p.Hq;
  it.hq = rest % p.Hq;
  return it;
}

// The item's K/V tiles in the forward's ring order: the query shard r's own chunk first, then
// r-1, r-2, ... (mod P); under the causal mask only K/V tiles at or before the query tile's
// position (with load-balanced shards a prefix of each half-chunk, visited directly).
template <class F>
__device__ __forceinline__ void for_each_kv(const BParams& p, const QItem& it, F&& f) {
  const int r = it.gq / p.tiles_per_shard;
  const int qpos = tile_pos(p, it.gq);
  const int hh = p.tiles_per_shard / 2;
  for (int t = 0; t < p.P; ++t) {
    const int j = ((r - t) % p.P + p.P) % p.P;
    if (p.causal && !p.balanced && j > r) continue;
    if (p.causal && p.balanced) {
      for (int half = 0; half < 2; ++half) {
        const int c = half ? 2 * p.P - 1 - j : j;
        const int o1 = qpos - c * hh + 1 < hh ? qpos - c * hh + 1 : hh;  // exclusive end
        for (int o = 0; o < o1; ++o)
          if (!f(j * p.tiles_per_shard + half * hh + o, c * hh + o == qpos)) return;
      }
      continue;
    }
    for (int kt = 0; kt < p.tiles_per_shard; ++kt) {
      const int gk = j * p.tiles_per_shard + kt;
      const int kpos = tile_pos(p, gk);
      if (p.causal && kpos > qpos) continue;
      if (!f(gk, p.causal && kpos == qpos)) return;
    }
  }
}

template <int D>
__device__ void q_producer(const BParams& p, QSmem* sc, uint32_t sbase, const QItem& it, const CUtensorMap* tq,
                           const CUtensorMap* tdo, const CUtensorMap* tk, const CUtensorMap* tv, uint32_t& kcnt,
                           uint32_t& vcnt) {
  using C = QCfg<D>;
  const int q_row = (it.b * p.Hq + it.hq) * p.S + it.gq * kRows;
  mbar_expect_tx(&sc->qd_full, 2 * C::TILE);
#pragma unroll
  for (int h = 0; h < D / 64; ++h) {
    tma_load_2d(sbase + C::OFF_Q + h * 16384, tq, 64 * h, q_row, &sc->qd_full);
    tma_load_2d(sbase + C::OFF_DO + h * 16384, tdo, 64 * h, q_row, &sc->qd_full);
  }
  const int kv_base = (it.b * p.Hkv + it.hq / p.gqa) * p.S;
  for_each_kv(p, it, [&](int gk, bool) -> bool {
    // kcnt and vcnt count the K and V loads issued (equal between tiles; both kept so that the
    // end of the kernel waits for exactly the loads in flight after an abort)
    const uint32_t kb = kcnt % C::KST, kfill = kcnt / C::KST, vb = vcnt % C::VST, vfill = vcnt / C::VST;
    if (kfill > 0 && !wait_bar(&sc->k_empty[kb], (kfill - 1) & 1u, p, sc, SITE_KV_EMPTY)) return false;
    mbar_expect_tx(&sc->k_full[kb], C::TILE);
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
      tma_load_2d(sbase + C::OFF_K + kb * C::TILE + h * 16384, tk, 64 * h, kv_base + gk * kRows, &sc->k_full[kb]);
    ++kcnt;
    if (vfill > 0 && !wait_bar(&sc->v_empty[vb], (vfill - 1) & 1u, p, sc, SITE_KV_EMPTY)) return false;
    mbar_expect_tx(&sc->v_full[vb], C::TILE);
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
      tma_load_2d(sbase + C::OFF_V + vb * C::TILE + h * 16384, tv, 64 * h, kv_base + gk * kRows, &sc->v_full[vb]);
    ++vcnt;
    return true;
  });
}

// Order per K/V tile j: S(j+1) (into the other S buffer, as soon as its K has landed), dQ(j)
// (after the warpgroups have written dS(j) over dP(j)), dP(j+1).
template <int D>
__device__ void q_mma(const BParams& p, QSmem* sc, uint32_t sbase, const QItem& it, uint32_t items, uint32_t& kcnt,
                      uint32_t& jg) {
  using C = QCfg<D>;
  constexpr uint32_t I_SS = idesc_ab(128, 128, false, false);  // S, dP
  constexpr uint32_t I_TS = idesc_ab(128, D, false, true);     // dQ: A = dS in TMEM, B = K MN-major
  constexpr uint32_t kHi = sdesc_hi_sw128(1024);
  const uint32_t tm = sc->tmem_base;
  const uint32_t sQ = sbase + C::OFF_Q, sDO = sbase + C::OFF_DO;
  int n_kv = 0;
  for_each_kv(p, it, [&](int, bool) -> bool { ++n_kv; return true; });
  if (!wait_bar(&sc->qd_full, items & 1u, p, sc, SITE_Q_FULL)) { sc->abort = 1; return; }
  auto k_of = [&](uint32_t c) { return sbase + C::OFF_K + (c % C::KST) * C::TILE; };
  auto v_of = [&](uint32_t c) { return sbase + C::OFF_V + (c % C::VST) * C::TILE; };
  auto issue_s = [&](uint32_t c, uint32_t j) -> bool {  // S of K load c into S buffer j % 2
    if (!wait_bar(&sc->k_full[c % C::KST], (c / C::KST) & 1u, p, sc, SITE_KV)) return false;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      mma_ss_w(tm + C::COL_S + (j % 2) * 128, kmaj_lo(sQ, kk), kHi, kmaj_lo(k_of(c), kk), kHi, I_SS, kk > 0 ? 1u : 0u);
    mma_commit(&sc->s_full[j % 2]);
    return true;
  };
  auto issue_dp = [&](uint32_t c) -> bool {  // dP of V load c; V is then released
    if (!wait_bar(&sc->v_full[c % C::VST], (c / C::VST) & 1u, p, sc, SITE_KV)) return false;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      mma_ss_w(tm + C::COL_DP, kmaj_lo(sDO, kk), kHi, kmaj_lo(v_of(c), kk), kHi, I_SS, kk > 0 ? 1u : 0u);
    mma_commit(&sc->dp_full);
    mma_commit(&sc->v_empty[c % C::VST]);
    return true;
  };
  tc_fence_after();
  if (!issue_s(kcnt, jg) || !issue_dp(kcnt)) { sc->abort = 1; return; }
  int i = 0;
  for_each_kv(p, it, [&](int, bool) -> bool {
    if (i + 1 < n_kv && !issue_s(kcnt + 1, jg + 1)) return false;
    if (!wait_bar(&sc->ds_ready, jg & 1u, p, sc, SITE_DS)) return false;
    tc_fence_after();
    const uint32_t sK = k_of(kcnt);
#pragma unroll
    for (int kk = 0; kk < kRows / 16; ++kk)
      mma_ts_w(tm + C::COL_DQ, tm + C::COL_DP + bf16_col(kk), mnmaj_lo(sK, kk), kHi, I_TS, (i == 0 && kk == 0) ? 0u : 1u);
    mma_commit(&sc->k_empty[kcnt % C::KST]);  // K of this tile is read
    if (i + 1 < n_kv && !issue_dp(kcnt + 1)) return false;  // dP(j+1) over dS(j), after the dQ MMA has read it
    ++kcnt;
    ++jg;
    ++i;
    return true;
  });
  if (i != n_kv) { sc->abort = 1; return; }
  mma_commit(&sc->acc_full);
}

// Warpgroup w: the query tile's rows on the lanes, K/V columns [64w, 64w + 64).
template <int D>
__device__ void q_elementwise(const BParams& p, QSmem* sc, const QItem& it, uint32_t items, uint32_t& jg) {
  using C = QCfg<D>;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int w = warp >= 8 ? 1 : 0;
  const int quarter = warp % 4;
  const int row = quarter * 32 + lane;  // query row of the tile
  const uint32_t lanes = sc->tmem_base + ((uint32_t)(quarter * 32) << 16);
  const size_t qrow = (size_t)(it.b * p.Hq + it.hq) * p.S + (size_t)it.gq * kRows + row;
  const float nlse2 = p.nlse2[qrow];  // -LSE * log2(e) of this query row
  const float ndlt = p.ndelta[qrow];  // -D
  bool ok = true;
  for_each_kv(p, it, [&](int, bool diag) -> bool {
    ok = __all_sync(0xffffffffu, wait_bar(&sc->s_full[jg % 2], (jg / 2) & 1u, p, sc, SITE_S));
    if (!ok) return false;
    tc_fence_after();
    float pv[64];  // P over the warpgroup's 64 key columns
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t s[32];
      tmem_ld32(lanes + C::COL_S + (jg % 2) * 128 + 64 * w + 32 * c, s);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) pv[32 * c + e] = ex2_approx(fmaf(__uint_as_float(s[e]), p.sl2, nlse2));
      if (diag) {  // diagonal tile: keys after the query are masked (key column > query row)
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (64 * w + 32 * c + e > row) pv[32 * c + e] = 0.0f;
      }
    }
    ok = __all_sync(0xffffffffu, wait_bar(&sc->dp_full, jg & 1u, p, sc, SITE_DP));
    if (!ok) return false;
    tc_fence_after();
    uint32_t ds[32];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t dp[32];
      tmem_ld32(lanes + C::COL_DP + 64 * w + 32 * c, dp);
      tmem_ld_wait();
      const uint64_t nd2 = f2_pack(ndlt, ndlt);
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float d0, d1;
        f2_unpack(mul2(f2_pack(pv[32 * c + e], pv[32 * c + e + 1]),
                       add2(f2_pack(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), nd2)),
                  d0, d1);
        ds[16 * c + e / 2] = pack_bf16x2(d0, d1);
      }
    }
    // dS as bf16 pairs over the low half of this warpgroup's own dP columns
    tmem_st16(lanes + C::COL_DP + 64 * w, ds);
    tmem_st16(lanes + C::COL_DP + 64 * w + 16, ds + 16);
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sc->ds_ready);
    ++jg;
    return true;
  });
  if (!ok) { sc->abort = 1; return; }
  ok = __all_sync(0xffffffffu, wait_bar(&sc->acc_full, items & 1u, p, sc, SITE_ACC));
  if (!ok) { sc->abort = 1; return; }
  tc_fence_after();
  uint16_t* dst = p.dq + qrow * D + w * (D / 2);
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t v[32], o[16];
    tmem_ld32(lanes + C::COL_DQ + w * (D / 2) + 32 * c, v);
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 16; ++e)
      o[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * p.scale, __uint_as_float(v[2 * e + 1]) * p.scale);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      reinterpret_cast<uint4*>(dst + 32 * c)[e] = make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_q_kernel(const __grid_constant__ BParams p, const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ QSmem sc;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(&sc.qd_full, 1);
    for (int b = 0; b < 3; ++b) {
      mbar_init(&sc.k_full[b], 1);
      mbar_init(&sc.k_empty[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sc.v_full[b], 1);
      mbar_init(&sc.v_empty[b], 1);
      mbar_init(&sc.s_full[b], 1);
    }
    mbar_init(&sc.dp_full, 1);
    mbar_init(&sc.ds_ready, 8);
    mbar_init(&sc.acc_full, 1);
    mbar_init(&sc.drain, 1);
    sc.abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_do);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(&sc.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  uint32_t items = 0, kcnt_p = 0, kcnt_v = 0, kcnt_m = 0, jg_m = 0, jg_e = 0;
  while (true) {
    if (threadIdx.x == 0) {
      int n = -1;
      if (!sc.abort && !ld_relaxed(&p.ctrl->abort)) {
        const uint32_t t = atomicAdd(&p.ctrl->init_next, 1u);
        if (t < (uint32_t)p.n_items_q) n = (int)t;
      }
      sc.arg = n;
    }
    __syncthreads();
    const int n = sc.arg;
    if (n < 0) break;
    const QItem it = q_item_of(p, n);
    if (warp == 0 && lane == 0) {
      q_producer<D>(p, &sc, sbase, it, &tm_q, &tm_do, &tm_k, &tm_v, kcnt_p, kcnt_v);
    } else if (warp == 1 && lane == 0) {
      q_mma<D>(p, &sc, sbase, it, items, kcnt_m, jg_m);
    } else if (warp >= 4) {
      q_elementwise<D>(p, &sc, it, items, jg_e);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0 && !sc.abort) atomicAdd(&p.ctrl->compute_items, 1ull);
    ++items;
    if (sc.abort) break;
  }
  if (warp == 1 && lane == 0) {
    mma_commit(&sc.drain);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(&sc.drain, 0) && globaltimer_ns() - t0 < 100000000ull) {
    }
  }
  if (warp == 0 && lane == 0) {
    const uint64_t t0 = globaltimer_ns();
    if (items > 0)
      while (!mbar_try_wait(&sc.qd_full, (items - 1) & 1u) && globaltimer_ns() - t0 < 100000000ull) {
      }
    // every K and V load has landed (the producer issued K before V for each tile, so the
    // last fill of each buffer is the one to wait for)
    for (uint32_t b = 0; b < (uint32_t)QCfg<D>::KST && b < kcnt_p; ++b) {
      const uint32_t fills = (kcnt_p - b + QCfg<D>::KST - 1) / QCfg<D>::KST;
      while (!mbar_try_wait(&sc.k_full[b], (fills - 1) & 1u) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
    for (uint32_t b = 0; b < (uint32_t)QCfg<D>::VST && b < kcnt_v; ++b) {
      const uint32_t fills = (kcnt_v - b + QCfg<D>::VST - 1) / QCfg<D>::VST;
      while (!mbar_try_wait(&sc.v_full[b], (fills - 1) & 1u) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(sc.tmem_base, 512);
}

// -D = -rowsum(dO * O) in fp32 (one warp per row), and -LSE * log2(e)
template <int D>
__global__ void delta_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                             const float* __restrict__ lse, float* __restrict__ ndelta, float* __restrict__ nlse2,
                             long long rows) {
  const int lane = threadIdx.x % 32;
  const long long warps = (long long)gridDim.x * (blockDim.x / 32);
  for (long long r = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; r < rows; r += warps) {
    const uint16_t* a = o + r * D;
    const uint16_t* b = dout + r * D;
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      const int c = lane * (D / 32) + e;
      s += __uint_as_float((uint32_t)a[c] << 16) * __uint_as_float((uint32_t)b[c] << 16);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) {
      ndelta[r] = -s;
      nlse2[r] = -lse[r] * kLog2e;
    }
  }
}


// ------------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------------
struct BLayout {
  size_t ctrl, delta, nlse2, total;
};

static size_t au(size_t x) { return (x + 255) / 256 * 256; }

static int check_shape(const psr_shape* sh) {
  if (!sh) return PSR_ERR_ARG;
  if (sh->B < 1 || sh->Hq < 1 || sh->Hkv < 1 || sh->S < 1 || sh->P < 1) return PSR_ERR_ARG;
  if (sh->causal < 0 || sh->causal > PSR_CAUSAL_BALANCED) return PSR_ERR_ARG;
  if (!(sh->scale == sh->scale)) return PSR_ERR_ARG;
  if (sh->d != 64 && sh->d != 128) return PSR_ERR_UNSUPPORTED;
  if (sh->Hq % sh->Hkv != 0 || sh->S % sh->P != 0 || (sh->S / sh->P) % kRows != 0) return PSR_ERR_UNSUPPORTED;
  if (sh->causal == PSR_CAUSAL_BALANCED && (sh->S / sh->P) % (2 * kRows) != 0) return PSR_ERR_UNSUPPORTED;
  const long long rows = (long long)sh->B * sh->Hq * sh->S;
  if (rows >= (1LL << 31) || rows * sh->d >= (1LL << 40)) return PSR_ERR_UNSUPPORTED;
  if ((long long)sh->B * sh->Hq * (sh->S / kRows) >= (1LL << 31)) return PSR_ERR_UNSUPPORTED;
  return PSR_OK;
}

static BLayout layout(const psr_shape* sh) {
  BLayout l;
  const size_t rows = (size_t)sh->B * sh->Hq * sh->S;
  size_t off = 0;
  l.ctrl = off; off += 256;
  off = au(off + (size_t)kTrajMax * 8);  // the shared workspace prefix (stats and trajectory)
  l.delta = off; off = au(off + rows * 4);
  l.nlse2 = off; off = au(off + rows * 4);
  l.total = off;
  return l;
}

template <int D>
static cudaError_t launch_bwd(const BParams& kp, const CUtensorMap* maps, int n_cta, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(bwd_kv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, KvCfg<D>::SMEM);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(bwd_q_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, QCfg<D>::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  bwd_kv_kernel<D><<<n_cta, kThreads, KvCfg<D>::SMEM, st>>>(kp, maps[0], maps[1], maps[2], maps[3]);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_q_kernel<D><<<n_cta, kThreads, QCfg<D>::SMEM, st>>>(kp, maps[0], maps[1], maps[2], maps[3]);
  return cudaGetLastError();
}

}  // namespace bwd
}  // namespace psr

using namespace psr;
using namespace psr::bwd;

extern "C" {

size_t psr_ring_attn_bwd_workspace_bytes(const psr_shape* sh) {
  if (check_shape(sh) != PSR_OK) return 0;
  return layout(sh).total;
}

int psr_ring_attn_bwd(const psr_shape* sh, const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv, void* workspace,
                      size_t ws_bytes, int timeout_ms, void* stream) {
  int rc = check_shape(sh);
  if (rc != PSR_OK) return rc;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return PSR_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PSR_ERR_ARG;
  for (const void* ptr : {q, k, v, o, (const void*)lse, dout, (const void*)dq, (const void*)dk, (const void*)dv})
    if ((reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return PSR_ERR_ARG;
  const BLayout L = layout(sh);
  if (ws_bytes < L.total) return PSR_ERR_ARG;
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return PSR_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return PSR_ERR_UNSUPPORTED;
  const int n_cta = prop.multiProcessorCount;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  BParams kp;
  memset(&kp, 0, sizeof(kp));
  kp.B = sh->B; kp.Hq = sh->Hq; kp.Hkv = sh->Hkv; kp.S = sh->S; kp.P = sh->P;
  kp.L = sh->S / sh->P;
  kp.gqa = sh->Hq / sh->Hkv;
  kp.causal = sh->causal ? 1 : 0;
  kp.balanced = sh->causal == PSR_CAUSAL_BALANCED ? 1 : 0;
  kp.tiles_per_shard = kp.L / kRows;
  kp.n_items_kv = sh->B * sh->Hkv * (sh->S / kRows);
  kp.n_items_q = sh->B * sh->Hq * (sh->S / kRows);
  const float scale = sh->scale > 0.0f ? sh->scale : 1.0f / std::sqrt((float)sh->d);
  kp.scale = scale;
  kp.sl2 = scale * kLog2e;
  kp.nlse2 = reinterpret_cast<const float*>(ws + L.nlse2);
  kp.ndelta = reinterpret_cast<const float*>(ws + L.delta);
  kp.dq = static_cast<uint16_t*>(dq);
  kp.dk = static_cast<uint16_t*>(dk);
  kp.dv = static_cast<uint16_t*>(dv);
  kp.ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  kp.timeout_ns = (unsigned long long)(timeout_ms > 0 ? timeout_ms : 2000) * 1000000ull;

  const long long rows_q = (long long)sh->B * sh->Hq * sh->S;
  const long long rows_kv = (long long)sh->B * sh->Hkv * sh->S;
  CUtensorMap maps[4];
  using gemm::tmap_kmajor;
  if (!tmap_kmajor(&maps[0], q, rows_q, sh->d, kRows) || !tmap_kmajor(&maps[1], dout, rows_q, sh->d, kRows) ||
      !tmap_kmajor(&maps[2], k, rows_kv, sh->d, kRows) || !tmap_kmajor(&maps[3], v, rows_kv, sh->d, kRows))
    return PSR_ERR_CUDA;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, L.delta, st) != cudaSuccess) return PSR_ERR_CUDA;  // control block and log
  const int dgrid = n_cta * 8;
  if (sh->d == 128)
    delta_kernel<128><<<dgrid, 256, 0, st>>>(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), lse,
                                            reinterpret_cast<float*>(ws + L.delta),
                                            reinterpret_cast<float*>(ws + L.nlse2), rows_q);
  else
    delta_kernel<64><<<dgrid, 256, 0, st>>>(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), lse,
                                           reinterpret_cast<float*>(ws + L.delta),
                                           reinterpret_cast<float*>(ws + L.nlse2), rows_q);
  if (cudaGetLastError() != cudaSuccess) return PSR_ERR_CUDA;
  cudaError_t e = sh->d == 128 ? launch_bwd<128>(kp, maps, n_cta, st) : launch_bwd<64>(kp, maps, n_cta, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PSR_ERR_CUDA;
  }
  return PSR_OK;
}

}  // extern "C"
