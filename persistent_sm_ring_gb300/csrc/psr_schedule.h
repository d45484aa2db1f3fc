// Work decomposition of the emulated ring, shared by host and device code.
//
// Ring (mKernel pages, dataforcee/chathome kernel tables, Ring Attention row;
// pwwt.cn Table 3): shard r consumes KV chunk j = (r - t) mod P at ring step
// t = 0..P-1; step 0 is its own chunk, read in place (pwwt.cn §2.6 schedule
// rule 3: local inputs first).  With a causal mask chunk j is needed by shard
// r only when j <= r, i.e. steps t = 0..r.
//
// Load-balanced causal shards (causal == 2).  Shard r holds two halves of the
// sequence: local rows [0, L/2) are global positions r*L/2 + i and local rows
// [L/2, L) are (2P-1-r)*L/2 + (i - L/2).  Then every shard does the same causal
// work at every step: at t = 0 the local chunk is masked as in the contiguous
// case (positions rise with the local index inside a shard); at 1 <= t <= r
// (chunk j < r) every query row sees exactly the first half of the chunk; at
// t > r (chunk j > r) the first-half query rows see none of it and the
// second-half rows see all of it.  No tile other than a step-0 diagonal tile is
// ever partly masked.
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
  int balanced;  // causal over load-balanced shards (causal == 2 at the API)
  int L;         // shard length S / P
  int gqa;       // Hq / Hkv
  int cg;        // CTAs per compute unit: 1, or 2 (a CTA pair)
  int item_rows; // query rows per item: 256 * cg
  int item_qt;   // 128-row query tiles per item: item_rows / 128
  int q_blocks;  // items per (b, hq, shard): L / item_rows
  int kv_tiles;  // 128-row KV tiles per chunk: L / 128
  int piece_tiles;  // tiles per staging piece
  int n_pieces;     // staging pieces per chunk
  int half_pieces;  // staging pieces of the first half of a chunk
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
  G.balanced = causal == 2 ? 1 : 0;
  if (causal < 0 || causal > 2) return 1;
  if (B < 1 || Hq < 1 || Hkv < 1 || S < 1 || P < 1 || d < 1) return 1;
  if (Hq % Hkv != 0 || S % P != 0) return 1;
  if (cg != 1 && cg != 2) return 1;
  G.cg = cg;
  G.item_rows = kCtaRows * cg;
  G.item_qt = G.item_rows / kTileRows;
  G.L = S / P;
  if (G.L % G.item_rows != 0) return 2;
  if (G.balanced && G.L % (2 * G.item_rows) != 0) return 2;  // each half holds whole items
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
  G.half_pieces = (G.kv_tiles / 2 + G.piece_tiles - 1) / G.piece_tiles;
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

// The shard layout of the functions below: kBal = -1 reads G.balanced; 0 or 1 fixes it at
// compile time (the device code instantiates one kernel per layout, so that the contiguous
// kernel carries none of the balanced layout's branches).
template <int kBal = -1>
PSR_HD bool is_balanced(const Geometry& G) { return kBal < 0 ? G.balanced != 0 : kBal != 0; }

// Contiguous causal shards: shard r needs steps 0..r only, and runs longest first.
template <int kBal = -1>
PSR_HD bool skewed(const Geometry& G) { return G.causal && !is_balanced<kBal>(G); }

// Shard of the rr-th shard in dispense order: contiguous causal runs the longest shards first.
template <int kBal = -1>
PSR_HD int shard_of_rank(const Geometry& G, int rr) { return skewed<kBal>(G) ? (G.P - 1 - rr) : rr; }

template <int kBal = -1>
PSR_HD int steps_of_shard(const Geometry& G, int r) { return skewed<kBal>(G) ? (r + 1) : G.P; }

// Groups are dispensed unit by unit -- a unit is one batch (B > 1) or one KV head with its query
// heads (B = 1), the blocks in which the host-buffer entry uploads the inputs and downloads the
// results -- and inside a unit shard by shard in rank order (longest shards first under the causal
// mask), so that compute follows the upload and each unit's results are complete as early as
// possible.
template <int kBal = -1>
PSR_HD void group_coord(const Geometry& G, int g, int& r, int& b, int& kvh, int& sub) {
  sub = g % G.n_sub;
  int rest = g / G.n_sub;
  if (G.B > 1) {  // unit = batch: shard by shard, every KV head of the batch at each shard
    kvh = rest % G.Hkv;
    rest /= G.Hkv;
    r = shard_of_rank<kBal>(G, rest % G.P);
    b = rest / G.P;
  } else {  // unit = KV head
    r = shard_of_rank<kBal>(G, rest % G.P);
    kvh = rest / G.P;
    b = 0;
  }
}

// Units: the blocks of the input the host-buffer entry uploads (and of the output it downloads)
// one at a time.
PSR_HD int unit_count(const Geometry& G) { return G.B > 1 ? G.B : G.Hkv; }
PSR_HD int unit_of(const Geometry& G, int b, int kvh) { return G.B > 1 ? b : kvh; }

template <int kBal = -1>
PSR_HD int group_steps(const Geometry& G, int g) {
  int r, b, kvh, sub;
  group_coord<kBal>(G, g, r, b, kvh, sub);
  return steps_of_shard<kBal>(G, r);
}

template <int kBal = -1>
PSR_HD ItemCoord item_coord(const Geometry& G, int n) {
  ItemCoord c;
  c.g = n / G.Gs;
  int sub;
  group_coord<kBal>(G, c.g, c.r, c.b, c.kvh, sub);
  const int w = sub * G.Gs + (n % G.Gs);
  c.hq = c.kvh * G.gqa + w / G.q_blocks;
  c.qp = w % G.q_blocks;
  c.n_steps = steps_of_shard<kBal>(G, c.r);
  return c;
}

// KV tiles an item consumes at ring step t, always a prefix 0 .. n-1 of the chunk's tiles:
// under the causal mask the local chunk stops at the diagonal of the item's last row
// ((qp+1)*item_qt tiles); over balanced shards a later step gives the first half of the
// chunk (chunk below the shard), or all / none of it (chunk above: second / first half items).
PSR_HD bool second_half(const Geometry& G, const ItemCoord& c) { return 2 * c.qp >= G.q_blocks; }

template <int kBal = -1>
PSR_HD int tiles_at_step(const Geometry& G, const ItemCoord& c, int t) {
  if (!G.causal) return G.kv_tiles;
  if (t == 0) return (c.qp + 1) * G.item_qt;
  if (!is_balanced<kBal>(G)) return G.kv_tiles;
  if (t <= c.r) return G.kv_tiles / 2;
  return second_half(G, c) ? G.kv_tiles : 0;
}

template <int kBal = -1>
PSR_HD long long item_tiles(const Geometry& G, const ItemCoord& c) {
  if (!G.causal) return (long long)G.P * G.kv_tiles;
  const long long diag = (long long)(c.qp + 1) * G.item_qt;
  if (!is_balanced<kBal>(G)) return diag + (long long)c.r * G.kv_tiles;
  return diag + (long long)c.r * (G.kv_tiles / 2) + (second_half(G, c) ? (long long)(G.P - 1 - c.r) * G.kv_tiles : 0);
}

PSR_HD long long total_tiles(const Geometry& G) {
  // per (b, hq): sum over shards and items
  long long per_bh = 0;
  const long long nb = G.q_blocks;
  if (!G.causal) {
    per_bh = (long long)G.P * nb * G.P * G.kv_tiles;
  } else {
    for (int r = 0; r < G.P; ++r) {
      per_bh += (long long)G.item_qt * nb * (nb + 1) / 2;
      if (G.balanced)
        per_bh += nb * r * (G.kv_tiles / 2) + (nb / 2) * (G.P - 1 - r) * G.kv_tiles;
      else
        per_bh += nb * r * G.kv_tiles;
    }
  }
  return per_bh * G.B * G.Hq;
}

// Tiles of the chunk that staging copies for shard r's step t >= 1: the most any of the
// group's items consumes (over balanced shards, only the first half of a chunk below r).
template <int kBal = -1>
PSR_HD int stage_tiles(const Geometry& G, int r, int t) {
  return (is_balanced<kBal>(G) && t <= r) ? G.kv_tiles / 2 : G.kv_tiles;
}
// (no division: the producer inlines this into its slot-release path, and an integer division
// there slowed the compute CTAs by ~15 % on GB300)
template <int kBal = -1>
PSR_HD int stage_pieces(const Geometry& G, int r, int t) {
  return (is_balanced<kBal>(G) && t <= r) ? G.half_pieces : G.n_pieces;
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
// The same two counts in staging pieces (the units the lists hand out).
PSR_HD long long total_staging_pieces(const Geometry& G) {
  long long n = 0;
  for (int r = 0; r < G.P; ++r)
    for (int t = 1; t < steps_of_shard(G, r); ++t) n += stage_pieces(G, r, t);
  return n * G.B * G.Hkv * G.n_sub;
}
PSR_HD long long dynamic_staging_pieces(const Geometry& G) {
  long long n = 0;
  for (int r = 0; r < G.P; ++r)
    for (int t = kRingSlots + 1; t < steps_of_shard(G, r); ++t) n += stage_pieces(G, r, t);
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

// Compute waves.  When every compute item takes the same time (non-causal attention), the
// compute role finishes in ceil(U / (N - n)) waves of whole items for U items and n staging
// CTAs, so compute time is flat between wave boundaries and jumps by one item at each
// boundary.  Given the smallest split n_need that still gives staging its capacity, the
// largest split with the same number of waves is
//   N - ceil(U / w),  w = ceil(U / (N - n_need)):
// any split up to it costs the compute role nothing, one above it costs a whole item.
// Returns n_cta (no cap) when there is nothing to cap.
PSR_HD int wave_cap(int n_cta, int n_need, long long U) {
  if (U <= 0 || n_need < 0 || n_need >= n_cta) return n_cta;
  const long long nc = n_cta - n_need;
  const long long w = (U + nc - 1) / nc;
  return n_cta - (int)((U + w - 1) / w);
}

// The wave cap made to hold whole groups: the items of one group share their ring slots, and a
// slot can be refilled only once every item of the group has loaded it, so a group whose items
// straddle a wave boundary holds its first items back by up to a whole item.  Returns the largest
// split n in [n_need, cap] whose compute CTAs N - n are a multiple of the group size Gs, or cap
// when there is none.
PSR_HD int wave_cap_groups(int n_cta, int n_need, int cap, int Gs) {
  if (Gs <= 1) return cap;
  for (int n = cap; n >= n_need && n >= 0; --n)
    if ((n_cta - n) % Gs == 0) return n;
  return cap;
}

}  // namespace psr
