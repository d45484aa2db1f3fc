// Ring Attention backward on sm_103a.
//
// The gradient of the forward step in psr_ring_attn.cu (the mKernel pages describe only the
// forward; the backward follows the same ring and reuses its log-sum-exp).  With the forward's
// LSE and D_i = dO_i . O_i, for each (query row i, key j) that the mask allows:
//     P_ij = exp(scale q_i.k_j - LSE_i),   dP_ij = dO_i . v_j,   dS_ij = P_ij (dP_ij - D_i),
//     dV_j += P_ij dO_i,   dK_j += scale dS_ij q_i,   dQ_i += scale dS_ij k_j.
// In the ring, each KV chunk travels around the ranks together with its dK / dV partial sums
// while every rank keeps its queries; the partials are back at the owner after P steps.  On one
// GPU an item holds one 128-row K/V tile and its dK / dV accumulators on chip for the whole
// ring, visiting the query shards in ring order (its own shard first, then r+1, r+2, ...), so
// nothing needs to be copied; dQ is accumulated in fp32 with vector atomic adds.
//
// Per (query tile, K/V tile) pair, with the key rows on the tensor-memory lanes:
//     S^T  = K Q^T          (tcgen05, SS)                      -> TMEM cols [0, 128)
//     dP^T = V dO^T         (tcgen05, SS)                      -> TMEM cols [128, 256)
//     P^T, dS^T             (one warpgroup, in place, bf16)    -> over S^T / over dP^T, and dS
//                                                                 into shared memory (MN-major)
//     dV  += P^T dO         (tcgen05, TS)                      -> TMEM cols [256, 256+d)
//     dK  += dS^T Q         (tcgen05, TS)                      -> TMEM cols [256+d, 256+2d)
//     dQ_t  = dS K          (tcgen05, SS)                      -> TMEM cols [128, 128+d)
//     dQ_acc += dQ_t        (one warpgroup: tcgen05.ld, red.global.add.v4.f32)
// One thread issues every MMA in that order; tensor-core instructions of one thread run in
// order, so an MMA that overwrites columns another MMA reads is simply issued after it.
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

template <int D>
struct BCfg {
  static constexpr int TILE = kRows * D * 2;  // one tile of Q, dO, K or V (bf16), D/64 boxes of 16 KiB
  static constexpr int DS_BYTES = kRows * kRows * 2;
  static constexpr int OFF_K = 0, OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;      // + qb * 2 * TILE (two buffers of Q | dO)
  static constexpr int OFF_DS = 6 * TILE;
  static constexpr int SMEM = 1024 + 6 * TILE + DS_BYTES;
  static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 256 + D;
  static_assert(SMEM <= 232448 - 1024, "shared memory");
};

enum : uint32_t { SITE_KV = 21, SITE_Q_FULL = 22, SITE_Q_EMPTY = 23, SITE_S = 24, SITE_DP = 25, SITE_P = 26,
                  SITE_DS = 27, SITE_DQ_FULL = 28, SITE_DQ_EMPTY = 29, SITE_DS_FREE = 30, SITE_ACC = 31 };

struct BParams {
  int B, Hq, Hkv, S, P, L, gqa, causal;
  int tiles_per_shard;  // L / 128
  int n_items;          // B * Hkv * (S / 128)
  float sl2;            // scale * log2(e)
  float scale;
  const float* lse;     // [B][Hq][S] natural-log LSE of the forward
  const float* delta;   // [B][Hq][S] D = rowsum(dO * O)
  float* dq_acc;        // [B][Hq][S][d] fp32 (zeroed before the launch)
  uint16_t* dk;         // [B][Hkv][S][d] bf16
  uint16_t* dv;
  Ctrl* ctrl;
  unsigned long long timeout_ns;
};

struct BSmem {
  uint64_t kv_full, q_full[2], q_empty[2], s_full, dp_full, p_ready, ds_ready, dq_full, dq_empty, ds_free, acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int arg;
  volatile uint32_t abort;
};

struct Item {
  int b, kvh, gk;  // batch, KV head, K/V tile (global 128-row index)
};
__device__ inline Item item_of(const BParams& p, int n) {
  Item it;
  it.gk = n / (p.B * p.Hkv);  // the earliest K/V tiles have the most causal work: dispensed first
  const int rest = n % (p.B * p.Hkv);
  it.b = rest / p.Hkv;
  it.kvh = rest % p.Hkv;
  return it;
}

// The item's (query head, query tile) pairs in ring order: shard j of the K/V tile first, then
// j+1, j+2, ... (mod P); under the causal mask only query tiles at or after the K/V tile.
template <class F>
__device__ __forceinline__ void for_each_pair(const BParams& p, const Item& it, F&& f) {
  const int j = it.gk / p.tiles_per_shard;
  for (int t = 0; t < p.P; ++t) {
    const int r = (j + t) % p.P;
    if (p.causal && r < j) continue;
    for (int h = 0; h < p.gqa; ++h) {
      const int hq = it.kvh * p.gqa + h;
      for (int qt = 0; qt < p.tiles_per_shard; ++qt) {
        const int gq = r * p.tiles_per_shard + qt;
        if (p.causal && gq < it.gk) continue;
        if (!f(hq, gq, p.causal && gq == it.gk)) return;
      }
    }
  }
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

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void unpack_bf16x2(uint32_t v, float& lo, float& hi) {
  lo = __uint_as_float(v << 16);
  hi = __uint_as_float(v & 0xFFFF0000u);
}

// ------------------------------------------------------------------------------------------------
// Roles
// ------------------------------------------------------------------------------------------------
template <int D>
__device__ void producer(const BParams& p, BSmem* sc, uint32_t sbase, const Item& it, const CUtensorMap* tq,
                         const CUtensorMap* tdo, const CUtensorMap* tk, const CUtensorMap* tv, uint32_t& qcnt) {
  using C = BCfg<D>;
  const int kv_row = (it.b * p.Hkv + it.kvh) * p.S + it.gk * kRows;
  mbar_expect_tx(&sc->kv_full, 2 * C::TILE);
#pragma unroll
  for (int h = 0; h < D / 64; ++h) {
    tma_load_2d(sbase + C::OFF_K + h * 16384, tk, 64 * h, kv_row, &sc->kv_full);
    tma_load_2d(sbase + C::OFF_V + h * 16384, tv, 64 * h, kv_row, &sc->kv_full);
  }
  for_each_pair(p, it, [&](int hq, int gq, bool) -> bool {
    const uint32_t qb = qcnt % 2, fill = qcnt / 2;
    if (fill > 0 && !wait_bar(&sc->q_empty[qb], (fill - 1) & 1u, p, sc, SITE_Q_EMPTY)) return false;
    const int q_row = (it.b * p.Hq + hq) * p.S + gq * kRows;
    const uint32_t qs = sbase + C::OFF_Q + qb * 2 * C::TILE;
    mbar_expect_tx(&sc->q_full[qb], 2 * C::TILE);
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      tma_load_2d(qs + h * 16384, tq, 64 * h, q_row, &sc->q_full[qb]);
      tma_load_2d(qs + C::TILE + h * 16384, tdo, 64 * h, q_row, &sc->q_full[qb]);
    }
    ++qcnt;
    return true;
  });
}

template <int D>
__device__ void mma_issuer(const BParams& p, BSmem* sc, uint32_t sbase, const Item& it, uint32_t items,
                           uint32_t& qcnt, uint32_t& jg) {
  using C = BCfg<D>;
  constexpr uint32_t I_SS = idesc_ab(128, 128, false, false);  // S^T, dP^T
  constexpr uint32_t I_TS = idesc_ab(128, D, false, true);     // dV, dK: A in TMEM, B MN-major
  constexpr uint32_t I_DQ = idesc_ab(128, D, true, true);      // dQ: A = dS MN-major, B = K MN-major
  constexpr uint32_t kHi = sdesc_hi_sw128(1024);
  const uint32_t tm = sc->tmem_base;
  if (!wait_bar(&sc->kv_full, items & 1u, p, sc, SITE_KV)) { sc->abort = 1; return; }
  tc_fence_after();
  const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sDS = sbase + C::OFF_DS;
  bool first = true;
  for_each_pair(p, it, [&](int, int, bool) -> bool {
    const uint32_t qb = qcnt % 2, ph = (qcnt / 2) & 1u;
    const uint32_t sQ = sbase + C::OFF_Q + qb * 2 * C::TILE, sDO = sQ + C::TILE;
    if (!wait_bar(&sc->q_full[qb], ph, p, sc, SITE_Q_FULL)) return false;
    tc_fence_after();
    // S^T = K Q^T (its columns held P^T of the previous pair, read by that pair's dV MMA)
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      mma_ss_w(tm + C::COL_S, kmaj_lo(sK, kk), kHi, kmaj_lo(sQ, kk), kHi, I_SS, kk > 0 ? 1u : 0u);
    mma_commit(&sc->s_full);
    // dP^T = V dO^T, once the previous pair's dQ has been read out of these columns
    if (jg > 0 && !wait_bar(&sc->dq_empty, (jg - 1) & 1u, p, sc, SITE_DQ_EMPTY)) return false;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      mma_ss_w(tm + C::COL_DP, kmaj_lo(sV, kk), kHi, kmaj_lo(sDO, kk), kHi, I_SS, kk > 0 ? 1u : 0u);
    mma_commit(&sc->dp_full);
    // dV += P^T dO
    if (!wait_bar(&sc->p_ready, jg & 1u, p, sc, SITE_P)) return false;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < kRows / 16; ++kk)
      mma_ts_w(tm + C::COL_DV, tm + C::COL_S + kk * 8, mnmaj_lo(sDO, kk), kHi, I_TS, (first && kk == 0) ? 0u : 1u);
    // dK += dS^T Q
    if (!wait_bar(&sc->ds_ready, jg & 1u, p, sc, SITE_DS)) return false;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < kRows / 16; ++kk)
      mma_ts_w(tm + C::COL_DK, tm + C::COL_DP + kk * 8, mnmaj_lo(sQ, kk), kHi, I_TS, (first && kk == 0) ? 0u : 1u);
    mma_commit(&sc->q_empty[qb]);  // Q and dO of this pair are read
    // dQ_t = dS K into the dP^T columns (after the dK MMA has read dS^T from them)
#pragma unroll
    for (int kk = 0; kk < kRows / 16; ++kk)
      mma_ss_w(tm + C::COL_DP, mnmaj_lo(sDS, kk), kHi, mnmaj_lo(sK, kk), kHi, I_DQ, kk > 0 ? 1u : 0u);
    mma_commit(&sc->dq_full);
    mma_commit(&sc->ds_free);
    first = false;
    ++qcnt;
    ++jg;
    return true;
  });
  mma_commit(&sc->acc_full);
}

// The warpgroup whose threads own the K/V tile's rows (tensor-memory lanes 0..127).
template <int D>
__device__ void softmax_wg(const BParams& p, BSmem* sc, uint8_t* smem, const Item& it, uint32_t items,
                           uint32_t& jg) {
  using C = BCfg<D>;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quarter = warp % 4;
  const int row = quarter * 32 + lane;  // K/V row of the tile
  const uint32_t lanes = sc->tmem_base + ((uint32_t)(quarter * 32) << 16);
  uint8_t* ds_row = smem + C::OFF_DS + row * 128;
  bool ok = true;
  for_each_pair(p, it, [&](int hq, int gq, bool diag) -> bool {
    const size_t qrow0 = (size_t)(it.b * p.Hq + hq) * p.S + (size_t)gq * kRows;
    ok = __all_sync(0xffffffffu, wait_bar(&sc->s_full, jg & 1u, p, sc, SITE_S));
    if (!ok) return false;
    tc_fence_after();
    uint32_t pk[64];  // P^T of this row, bf16 pairs
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t s[32];
      tmem_ld32(lanes + C::COL_S + 32 * c, s);
      tmem_ld_wait();
      const float4* l4 = reinterpret_cast<const float4*>(p.lse + qrow0 + 32 * c);
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) {
        const float4 l = __ldg(l4 + e4);
        const float lv[4] = {l.x, l.y, l.z, l.w};
        float pv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int col = 32 * c + 4 * e4 + u;  // query row of the tile
          const float x = __uint_as_float(s[4 * e4 + u]) * p.sl2 - lv[u] * kLog2e;
          pv[u] = (diag && col < row) ? 0.0f : ex2_approx(x);
        }
        pk[16 * c + 2 * e4] = pack_bf16x2(pv[0], pv[1]);
        pk[16 * c + 2 * e4 + 1] = pack_bf16x2(pv[2], pv[3]);
      }
      tmem_st16(lanes + C::COL_S + 16 * c, &pk[16 * c]);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sc->p_ready);
    ok = __all_sync(0xffffffffu, wait_bar(&sc->dp_full, jg & 1u, p, sc, SITE_DP));
    if (ok && jg > 0) ok = __all_sync(0xffffffffu, wait_bar(&sc->ds_free, (jg - 1) & 1u, p, sc, SITE_DS_FREE));
    if (!ok) return false;
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t dp[32];
      tmem_ld32(lanes + C::COL_DP + 32 * c, dp);
      tmem_ld_wait();
      const float4* d4 = reinterpret_cast<const float4*>(p.delta + qrow0 + 32 * c);
      uint32_t ds[16];
#pragma unroll
      for (int e4 = 0; e4 < 8; ++e4) {
        const float4 dd = __ldg(d4 + e4);
        float p0, p1, p2, p3;
        unpack_bf16x2(pk[16 * c + 2 * e4], p0, p1);
        unpack_bf16x2(pk[16 * c + 2 * e4 + 1], p2, p3);
        ds[2 * e4] = pack_bf16x2(p0 * (__uint_as_float(dp[4 * e4]) - dd.x), p1 * (__uint_as_float(dp[4 * e4 + 1]) - dd.y));
        ds[2 * e4 + 1] =
            pack_bf16x2(p2 * (__uint_as_float(dp[4 * e4 + 2]) - dd.z), p3 * (__uint_as_float(dp[4 * e4 + 3]) - dd.w));
      }
      // dS^T over the dP^T columns already read (columns 16c .. 16c+15 of the bf16 pairs)
      tmem_st16(lanes + C::COL_DP + 16 * c, ds);
      // dS into shared memory as the MN-major A operand of dQ = dS K: row = key, 64 queries per
      // 128-byte row of a 16 KiB box, 16-byte chunks swizzled with the row
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int chunk = (c % 2) * 4 + i;
        uint4 v;
        v.x = ds[4 * i];
        v.y = ds[4 * i + 1];
        v.z = ds[4 * i + 2];
        v.w = ds[4 * i + 3];
        *reinterpret_cast<uint4*>(ds_row + (c / 2) * 16384 + ((chunk ^ (row & 7)) * 16)) = v;
      }
    }
    tmem_st_wait();
    fence_proxy_async_smem();  // the generic dS stores before the MMA's reads
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sc->ds_ready);
    ++jg;
    return true;
  });
  if (!ok) { sc->abort = 1; return; }
  // the item's dK and dV rows
  ok = __all_sync(0xffffffffu, wait_bar(&sc->acc_full, items & 1u, p, sc, SITE_ACC));
  if (!ok) { sc->abort = 1; return; }
  tc_fence_after();
  const size_t out_row = ((size_t)(it.b * p.Hkv + it.kvh) * p.S + (size_t)it.gk * kRows + row) * D;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const uint32_t col = which ? C::COL_DK : C::COL_DV;
    const float mul = which ? p.scale : 1.0f;
    uint16_t* dst = (which ? p.dk : p.dv) + out_row;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(lanes + col + 32 * c, v);
      tmem_ld_wait();
      uint4 o[4];
      uint32_t* w = reinterpret_cast<uint32_t*>(o);
#pragma unroll
      for (int e = 0; e < 16; ++e)
        w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
#pragma unroll
      for (int e = 0; e < 4; ++e) reinterpret_cast<uint4*>(dst + 32 * c)[e] = o[e];
    }
  }
}

// The warpgroup that reads each pair's dQ_t (query rows on the lanes) and adds it to dQ_acc.
template <int D>
__device__ void dq_wg(const BParams& p, BSmem* sc, const Item& it, uint32_t& jg) {
  using C = BCfg<D>;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quarter = warp % 4;
  const int row = quarter * 32 + lane;
  const uint32_t lanes = sc->tmem_base + ((uint32_t)(quarter * 32) << 16);
  bool ok = true;
  for_each_pair(p, it, [&](int hq, int gq, bool) -> bool {
    ok = __all_sync(0xffffffffu, wait_bar(&sc->dq_full, jg & 1u, p, sc, SITE_DQ_FULL));
    if (!ok) return false;
    tc_fence_after();
    float* dst = p.dq_acc + ((size_t)(it.b * p.Hq + hq) * p.S + (size_t)gq * kRows + row) * D;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(lanes + C::COL_DP + 32 * c, v);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 8; ++e)
        red_add_v4(dst + 32 * c + 4 * e, __uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                   __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sc->dq_empty);
    ++jg;
    return true;
  });
  if (!ok) sc->abort = 1;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    ring_attn_bwd_kernel(const __grid_constant__ BParams p, const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ BSmem sc;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(&sc.kv_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sc.q_full[b], 1);
      mbar_init(&sc.q_empty[b], 1);
    }
    mbar_init(&sc.s_full, 1);
    mbar_init(&sc.dp_full, 1);
    mbar_init(&sc.p_ready, 4);   // the four warps of the softmax warpgroup
    mbar_init(&sc.ds_ready, 4);
    mbar_init(&sc.dq_full, 1);
    mbar_init(&sc.dq_empty, 4);  // the four warps of the dQ warpgroup
    mbar_init(&sc.ds_free, 1);
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

  uint32_t items = 0, qcnt_p = 0, qcnt_m = 0, jg_m = 0, jg_s = 0, jg_q = 0;
  while (true) {
    if (threadIdx.x == 0) {
      int n = -1;
      if (!sc.abort && !ld_relaxed(&p.ctrl->abort)) {
        const uint32_t t = atomicAdd(&p.ctrl->item_next, 1u);
        if (t < (uint32_t)p.n_items) n = (int)t;
      }
      sc.arg = n;
    }
    __syncthreads();
    const int n = sc.arg;
    if (n < 0) break;
    const Item it = item_of(p, n);
    if (warp == 0 && lane == 0) {
      producer<D>(p, &sc, sbase, it, &tm_q, &tm_do, &tm_k, &tm_v, qcnt_p);
    } else if (warp == 1 && lane == 0) {
      mma_issuer<D>(p, &sc, sbase, it, items, qcnt_m, jg_m);
    } else if (warp >= 4 && warp < 8) {
      softmax_wg<D>(p, &sc, smem, it, items, jg_s);
    } else if (warp >= 8) {
      dq_wg<D>(p, &sc, it, jg_q);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0 && !sc.abort) atomicAdd(&p.ctrl->compute_items, 1ull);
    ++items;
    if (sc.abort) break;
  }
  // drain (bounded): every MMA has completed and every TMA load has landed before TMEM and
  // shared memory are released
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

// D = rowsum(dO * O) in fp32, one warp per row
template <int D>
__global__ void delta_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout, float* __restrict__ delta,
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
    if (lane == 0) delta[r] = s;
  }
}

// dQ = scale * dQ_acc, rounded to bf16 (four elements per thread)
__global__ void dq_convert_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq, float scale, long long n4) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    const float4 v = acc[i];
    uint2 w;
    w.x = pack_bf16x2(v.x * scale, v.y * scale);
    w.y = pack_bf16x2(v.z * scale, v.w * scale);
    dq[i] = w;
  }
}

// ------------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------------
struct BLayout {
  size_t ctrl, delta, dq_acc, total;
};

static size_t au(size_t x) { return (x + 255) / 256 * 256; }

static int check_shape(const psr_shape* sh) {
  if (!sh) return PSR_ERR_ARG;
  if (sh->B < 1 || sh->Hq < 1 || sh->Hkv < 1 || sh->S < 1 || sh->P < 1) return PSR_ERR_ARG;
  if (sh->causal < 0 || sh->causal > PSR_CAUSAL_BALANCED) return PSR_ERR_ARG;
  if (!(sh->scale == sh->scale)) return PSR_ERR_ARG;
  if (sh->causal == PSR_CAUSAL_BALANCED) return PSR_ERR_UNSUPPORTED;
  if (sh->d != 64 && sh->d != 128) return PSR_ERR_UNSUPPORTED;
  if (sh->Hq % sh->Hkv != 0 || sh->S % sh->P != 0 || (sh->S / sh->P) % kRows != 0) return PSR_ERR_UNSUPPORTED;
  const long long rows = (long long)sh->B * sh->Hq * sh->S;
  if (rows >= (1LL << 31) || rows * sh->d >= (1LL << 40)) return PSR_ERR_UNSUPPORTED;
  if ((long long)sh->B * sh->Hkv * (sh->S / kRows) >= (1LL << 31)) return PSR_ERR_UNSUPPORTED;
  return PSR_OK;
}

static BLayout layout(const psr_shape* sh) {
  BLayout l;
  const size_t rows = (size_t)sh->B * sh->Hq * sh->S;
  size_t off = 0;
  l.ctrl = off; off += 256;
  off = au(off + (size_t)kTrajMax * 8);  // the shared workspace prefix (stats and trajectory)
  l.delta = off; off = au(off + rows * 4);
  l.dq_acc = off; off = au(off + rows * sh->d * 4);
  l.total = off;
  return l;
}

template <int D>
static cudaError_t launch_bwd(const BParams& kp, const CUtensorMap* maps, int n_cta, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(ring_attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    BCfg<D>::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  ring_attn_bwd_kernel<D><<<n_cta, kThreads, BCfg<D>::SMEM, st>>>(kp, maps[0], maps[1], maps[2], maps[3]);
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
  kp.causal = sh->causal;
  kp.tiles_per_shard = kp.L / kRows;
  kp.n_items = sh->B * sh->Hkv * (sh->S / kRows);
  const float scale = sh->scale > 0.0f ? sh->scale : 1.0f / std::sqrt((float)sh->d);
  kp.scale = scale;
  kp.sl2 = scale * kLog2e;
  kp.lse = lse;
  kp.delta = reinterpret_cast<const float*>(ws + L.delta);
  kp.dq_acc = reinterpret_cast<float*>(ws + L.dq_acc);
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
  if (cudaMemsetAsync(ws + L.dq_acc, 0, (size_t)rows_q * sh->d * 4, st) != cudaSuccess) return PSR_ERR_CUDA;
  const int dgrid = n_cta * 8;
  if (sh->d == 128)
    delta_kernel<128><<<dgrid, 256, 0, st>>>(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout),
                                            reinterpret_cast<float*>(ws + L.delta), rows_q);
  else
    delta_kernel<64><<<dgrid, 256, 0, st>>>(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout),
                                           reinterpret_cast<float*>(ws + L.delta), rows_q);
  if (cudaGetLastError() != cudaSuccess) return PSR_ERR_CUDA;
  cudaError_t e = sh->d == 128 ? launch_bwd<128>(kp, maps, n_cta, st) : launch_bwd<64>(kp, maps, n_cta, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PSR_ERR_CUDA;
  }
  dq_convert_kernel<<<n_cta * 8, 256, 0, st>>>(reinterpret_cast<const float4*>(ws + L.dq_acc),
                                               static_cast<uint2*>(dq), scale, rows_q * sh->d / 4);
  if (cudaGetLastError() != cudaSuccess) return PSR_ERR_CUDA;
  return PSR_OK;
}

}  // extern "C"
