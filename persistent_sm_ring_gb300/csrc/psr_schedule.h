// Work decomposition of the emulated ring, shared by host and device code.
//
// Ring (mKernel pages, dataforcee/chathome kernel tables, Ring Attention row;
// pwwt.cn Table 3): shard r consumes KV chunk j = (r - t) mod P at ring step
// t = 0..P-1; step 0 is its own chunk, read in place (pwwt.cn §2.6 schedule
// rule 3: local inputs first).  With a causal mask chunk j is needed by shard
// r only when j <= r, i.e. steps t = 0..r.
//
// Units of work:
//  * compute item  = the query rows one compute unit carries through all of
//                    shard r's ring steps with the accumulators resident in
//                    tensor memory, for one (b, hq): 256 rows (two 128-row
//                    tiles) for a single CTA, 512 rows (two tiles in each CTA)
//                    for a CTA pair that shares every K/V tile;
//  * group         = the items that read the same ring slot: shard r, batch b,
//                    KV head kvh (all Hq/Hkv query heads of it) and, when a
//                    group would exceed the deadlock bound, a sub-group index;
//  * staging chunk = one (group, step >= 1): chunk (r - step) mod P of K and V
//                    copied into the group's slot (step mod kRingSlots) in 128-row tiles
//                    (the pages' ring moves KV in 128-row tiles, Table 3);
//  * staging piece = a quarter of a chunk, but at least 512 KiB of K+V and at most
//                    kStagePieceMaxTiles tiles: the unit a staging CTA claims, so
//                    that several CTAs fill one chunk at once while each copy stays
//                    long enough to hide its fixed cost; readiness is published per
//                    piece as a tile count.
// Slot (s mod kRingSlots) of a group may be overwritten for step s > kRingSlots only
// when all of the group's items have loaded step s - kRingSlots: that is the ring
// buffer's back-pressure.
#pragma once
#include <cstdint>

#ifdef __CUDACC__
#define PSR_HD __host__ __device__ __forceinline__
#else
#define PSR_HD inline
#endif

namespace psr {

constexpr int kTileRows = 128;  // rows per Q tile and per KV tile
constexpr int kCtaRows = 256;   // query rows one CTA holds during an item (two tiles)
#ifndef PSR_PIECE_DIV
#define PSR_PIECE_DIV 4
#endif
constexpr int kStagePieceDiv = PSR_PIECE_DIV;  // staging piece: 1/kStagePieceDiv of a chunk ...
constexpr int kStagePieceMaxTiles = 8;         // ... of 1..8 tiles ...
#ifndef PSR_PIECE_MIN_KB
#define PSR_PIECE_MIN_KB 512
#endif
// ... and at least this many KiB of K+V.  Measured on GB300: a piece's copy costs ~6500 cycles
// even when it is a single 64 KiB tile, so 1-2 tile pieces halved the staging CTAs' rate;
// 512 KiB pieces cut the partition sweep's total time by 27 % (P = 64: 8.97 -> 5.43 ms).
constexpr int kStagePieceMinKB = PSR_PIECE_MIN_KB;
#ifndef PSR_RING_SLOTS
#define PSR_RING_SLOTS 3
#endif
// Ring slots per group.  Three rather than two: under the causal mask a group's items spend
// (qp+1)*2 tiles on the local step 0, so they reach the staged steps up to a whole step apart,
// and with two slots the items ahead wait for the one behind to release step s - 2.
constexpr int kRingSlots = PSR_RING_SLOTS;
static_assert(kRingSlots >= 2, "at least a double buffer");
PSR_HD int slot_of(int step) { return step % kRingSlots; }

struct Geometry {
  int B, Hq, Hkv, S, P, d, causal;
  int L;         // shard length S / P
  int gqa;       // Hq / Hkv
  int cg;        // CTAs per compute unit: 1, or 2 (a CTA pair)
  int item_rows; // query rows per item: 256 * cg
  int item_qt;   // 128-row query tiles per item: item_rows / 128
  int q_blocks;  // items per (b, hq, shard): L / item_rows
  int kv_tiles;  // 128-row KV tiles per chunk: L / 128
  int piece_tiles;  // tiles per staging piece
  int n_pieces;     // staging pieces per chunk
  int G;         // items sharing one (shard, b, kvh): gqa * q_blocks
  int n_sub;     // sub-groups per (shard, b, kvh)
  int Gs;        // items per group: G / n_sub
  int n_groups;  // P * B * Hkv * n_sub
  int n_items;   // n_groups * Gs
};

struct ItemCoord {
  int g;        // group index (dispense order)
  int b, hq, kvh, r, qp;
  int n_steps;  // active ring steps of shard r
};

// max_group: most items one group may hold (all of them must be able to run at once);
// cg: CTAs per compute unit (1 or 2).
PSR_HD int geometry_init(Geometry& G, int B, int Hq, int Hkv, int S, int P, int d, int causal, int max_group,
                         int cg = 1) {
  G.B = B; G.Hq = Hq; G.Hkv = Hkv; G.S = S; G.P = P; G.d = d; G.causal = causal ? 1 : 0;
  if (B < 1 || Hq < 1 || Hkv < 1 || S < 1 || P < 1 || d < 1) return 1;
  if (Hq % Hkv != 0 || S % P != 0) return 1;
  if (cg != 1 && cg != 2) return 1;
  G.cg = cg;
  G.item_rows = kCtaRows * cg;
  G.item_qt = G.item_rows / kTileRows;
  G.L = S / P;
  if (G.L % G.item_rows != 0) return 2;
  G.gqa = Hq / Hkv;
  G.q_blocks = G.L / G.item_rows;
  G.kv_tiles = G.L / kTileRows;
  {
    // 1/kStagePieceDiv of a chunk, but at least kStagePieceMinKB of K+V (a piece's copy has a
    // fixed cost of a few microseconds), at most kStagePieceMaxTiles tiles and one chunk
    const int min_tiles = (kStagePieceMinKB * 1024 + 2 * kTileRows * d * 2 - 1) / (2 * kTileRows * d * 2);
    int pt = G.kv_tiles / kStagePieceDiv;
    if (pt < min_tiles) pt = min_tiles;
    if (pt > kStagePieceMaxTiles) pt = kStagePieceMaxTiles;
    if (pt > G.kv_tiles) pt = G.kv_tiles;
    G.piece_tiles = pt < 1 ? 1 : pt;
  }
  G.n_pieces = (G.kv_tiles + G.piece_tiles - 1) / G.piece_tiles;
  G.G = G.gqa * G.q_blocks;
  // split a group into power-of-two sub-groups until it fits the bound
  G.n_sub = 1;
  while (G.G / G.n_sub > max_group && (G.G % (G.n_sub * 2)) == 0) G.n_sub *= 2;
  if (G.G / G.n_sub > max_group) return 2;
  G.Gs = G.G / G.n_sub;
  const long long ng = (long long)P * B * Hkv * G.n_sub;
  if (ng > (1 << 24)) return 2;
  G.n_groups = (int)ng;
  const long long ni = ng * G.Gs;
  if (ni > (1LL << 30)) return 2;
  G.n_items = (int)ni;
  return 0;
}

// Shard of the rr-th shard in dispense order: causal runs the longest shards first.
PSR_HD int shard_of_rank(const Geometry& G, int rr) { return G.causal ? (G.P - 1 - rr) : rr; }

PSR_HD int steps_of_shard(const Geometry& G, int r) { return G.causal ? (r + 1) : G.P; }

PSR_HD void group_coord(const Geometry& G, int g, int& r, int& b, int& kvh, int& sub) {
  sub = g % G.n_sub;
  int rest = g / G.n_sub;
  kvh = rest % G.Hkv;
  rest /= G.Hkv;
  b = rest % G.B;
  r = shard_of_rank(G, rest / G.B);
}

PSR_HD int group_steps(const Geometry& G, int g) {
  int r, b, kvh, sub;
  group_coord(G, g, r, b, kvh, sub);
  return steps_of_shard(G, r);
}

PSR_HD ItemCoord item_coord(const Geometry& G, int n) {
  ItemCoord c;
  c.g = n / G.Gs;
  int sub;
  group_coord(G, c.g, c.r, c.b, c.kvh, sub);
  const int w = sub * G.Gs + (n % G.Gs);
  c.hq = c.kvh * G.gqa + w / G.q_blocks;
  c.qp = w % G.q_blocks;
  c.n_steps = steps_of_shard(G, c.r);
  return c;
}

// KV tiles an item consumes at ring step t: under the causal mask the local
// chunk stops at the diagonal of the item's last row (tiles 0 .. (qp+1)*item_qt - 1).
PSR_HD int tiles_at_step(const Geometry& G, const ItemCoord& c, int t) {
  return (G.causal && t == 0) ? (c.qp + 1) * G.item_qt : G.kv_tiles;
}

PSR_HD long long item_tiles(const Geometry& G, const ItemCoord& c) {
  return G.causal ? (long long)(c.qp + 1) * G.item_qt + (long long)c.r * G.kv_tiles : (long long)G.P * G.kv_tiles;
}

PSR_HD long long total_tiles(const Geometry& G) {
  // per (b, hq): sum over shards and items
  long long per_bh = 0;
  if (G.causal) {
    const long long nb = G.q_blocks;
    for (int r = 0; r < G.P; ++r) per_bh += (long long)G.item_qt * nb * (nb + 1) / 2 + nb * r * G.kv_tiles;
  } else {
    per_bh = (long long)G.P * G.q_blocks * G.P * G.kv_tiles;
  }
  return per_bh * G.B * G.Hq;
}

// Staging tasks: every (group, step >= 1).  Steps 1..kRingSlots land in fresh slots
// and come from a static list in group order; later steps enter a ready queue
// when the slot they overwrite has been consumed.
PSR_HD long long total_staging_tasks(const Geometry& G) {
  long long n = 0;
  for (int rr = 0; rr < G.P; ++rr) n += steps_of_shard(G, shard_of_rank(G, rr)) - 1;
  return n * G.B * G.Hkv * G.n_sub;
}
PSR_HD long long dynamic_staging_tasks(const Geometry& G) {
  long long n = 0;
  for (int rr = 0; rr < G.P; ++rr) {
    int s = steps_of_shard(G, shard_of_rank(G, rr));
    n += s > kRingSlots + 1 ? s - (kRingSlots + 1) : 0;
  }
  return n * G.B * G.Hkv * G.n_sub;
}

// The pages' partition rule (pwwt.cn §2.4): equalise the predicted finish
// times R_s*C_s/n_s and R_p*C_p/(N - n_s) of the two roles, i.e.
//   n_s* = N * (R_s*C_s) / (R_p*C_p + R_s*C_s),
// rounded to nearest and clamped to [max(n_min,1), min(n_max, N-1)] while both
// roles have work; 0 once staging is finished; n_max when only staging remains.
PSR_HD int controller_rule(int n_cta, double R_s, double C_s, double R_p, double C_p, int n_min, int n_max) {
  if (n_cta < 2) return 0;
  if (R_s <= 0.0) return 0;
  int lo = n_min < 1 ? 1 : n_min;
  int hi = n_max > n_cta - 1 ? n_cta - 1 : n_max;
  if (hi < lo) hi = lo;
  if (R_p <= 0.0) return hi;
  const double ws = R_s * C_s, wp = R_p * C_p;
  double x = (ws + wp) > 0.0 ? (double)n_cta * ws / (wp + ws) : 0.0;
  int n = (int)(x + 0.5);
  if (n < lo) n = lo;
  if (n > hi) n = hi;
  return n;
}

}  // namespace psr
