// Host check of the ring schedule used by the kernel (psr_schedule.h):
//  * every compute item's TMA coordinates (Q tiles, home K/V tiles, slot tiles)
//    stay inside the tensor extents the launcher encodes;
//  * every (b, hq, row) of the output is written by exactly one item;
//  * under a causal mask (contiguous or load-balanced shards), derived from the global
//    positions of the rows: the KV tiles an item reads at a step are exactly those in
//    which some key is visible to some row of the item; at a step t > 0 every tile read
//    is visible in full to every row of the item (the kernel masks step 0 only), and at
//    step 0 positions rise with the local index (the kernel masks by local index);
//  * staging copies, per (group, step), exactly the tiles the group's items read;
//  * flag / consumed indices stay below n_groups * P and the dynamic queue
//    receives exactly dynamic_staging_tasks() pushes;
//  * total_tiles(), total_staging_tasks() and the piece counts agree with direct enumeration.
// Usage: schedule_check wave   -> checks the controller's wave cap against enumeration.
//        schedule_check slices -> checks the host-buffer pipeline's slice plan.
// Usage: schedule_check B Hq Hkv S P d causal max_group [cg]   -> prints "OK ..." or "FAIL ..."
// (causal: 0, 1, or 2 = load-balanced shards; cg: CTAs per compute unit, 1 or 2; default 1)
#include <cstdio>
#include <algorithm>
#include <cstdlib>
#include <string>
#include <vector>

#include "../persistent_sm_ring_gb300/csrc/psr_schedule.h"

using namespace psr;

// Global position of local row i of shard r: contiguous shards, or load-balanced shards
// (local rows [0, L/2) are half-chunk r, rows [L/2, L) half-chunk 2P-1-r).
static long long pos_of(const Geometry& G, int r, long long i) {
  if (!G.balanced) return (long long)r * G.L + i;
  const long long h = G.L / 2;
  return i < h ? (long long)r * h + i : (long long)(2 * G.P - 1 - r) * h + (i - h);
}

#define CHECK(c, ...)                 \
  do {                                \
    if (!(c)) {                       \
      std::printf("FAIL ");           \
      std::printf(__VA_ARGS__);       \
      std::printf("\n");              \
      return 1;                       \
    }                                 \
  } while (0)

// wave_cap against its definition by enumeration: the largest split n in [n_need, N-1] whose
// compute waves ceil(U / (N - n)) equal those of n_need.
static int check_wave_cap() {
  for (int N = 2; N <= 160; N += (N < 20 ? 1 : 7))
    for (int need = 0; need < N; ++need)
      for (long long U = 1; U <= 5000; U += (U < 300 ? 1 : 37)) {
        auto waves = [&](int n) { return (U + (N - n) - 1) / (N - n); };
        int best = need;
        for (int n = need; n < N; ++n)
          if (waves(n) == waves(need)) best = n;
        const int cap = wave_cap(N, need, U);
        CHECK(cap == best, "wave_cap N=%d need=%d U=%lld: %d, enumeration %d", N, need, U, cap, best);
      }
  CHECK(wave_cap(152, 20, 0) == 152 && wave_cap(152, 152, 100) == 152, "wave_cap without a cap");
  CHECK(wave_cap(152, 21, 1024) == 24 && wave_cap(152, 41, 1024) == 49, "wave_cap examples");
  // wave_cap_groups against its definition: the largest n in [need, cap] with N - n a multiple of Gs
  for (int N = 2; N <= 160; N += 3)
    for (int need = 0; need < N; need += 2)
      for (int cap = need; cap < N; cap += 3)
        for (int Gs = 1; Gs <= 9; ++Gs) {
          int want = cap;
          for (int n = need; n <= cap; ++n)
            if ((N - n) % Gs == 0) want = n;
          const int got = wave_cap_groups(N, need, cap, Gs);
          CHECK(got == want, "wave_cap_groups N=%d need=%d cap=%d Gs=%d: %d, enumeration %d", N, need, cap, Gs, got, want);
        }
  CHECK(wave_cap_groups(152, 41, 49, 2) == 48 && wave_cap_groups(152, 21, 24, 4) == 24, "wave_cap_groups examples");
  std::printf("OK wave_cap\n");
  return 0;
}

int main(int argc, char** argv) {
  if (argc == 2 && std::string(argv[1]) == "wave") return check_wave_cap();
  if (argc != 9 && argc != 10) return 2;
  int a[9] = {0, 0, 0, 0, 0, 0, 0, 0, 1};
  for (int i = 0; i < argc - 1; ++i) a[i] = std::atoi(argv[i + 1]);
  Geometry G;
  int rc = geometry_init(G, a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7], a[8]);
  if (rc != 0) {
    std::printf("REJECT %d\n", rc);
    return 0;
  }
  const long long rows_q = (long long)G.B * G.Hq * G.S, rows_kv = (long long)G.B * G.Hkv * G.S;
  const long long rows_slot = (long long)kRingSlots * G.n_groups * G.L;
  std::vector<unsigned char> covered((size_t)rows_q / kTileRows, 0);
  std::vector<int> consumers((size_t)G.n_groups * G.P, 0);
  std::vector<int> max_read((size_t)G.n_groups * G.P, 0);  // most tiles any item of g reads at t
  if (G.causal) {
    // every 128-row tile covers 128 consecutive positions, and inside a shard positions rise
    for (int r = 0; r < G.P; ++r)
      for (long long i = 0; i + 1 < G.L; ++i) {
        CHECK(pos_of(G, r, i + 1) > pos_of(G, r, i), "positions fall inside shard %d", r);
        if ((i + 1) % kTileRows != 0) CHECK(pos_of(G, r, i + 1) == pos_of(G, r, i) + 1, "tile not contiguous");
      }
  }
  long long tiles = 0;
  // items are dispensed unit by unit, the same number per unit, and inside a unit (contiguous
  // causal shards) longest shards first
  const int n_units = unit_count(G);
  CHECK(G.n_items % n_units == 0, "items per unit");
  const int per_unit = G.n_items / n_units;
  for (int n = 0; n < G.n_items; ++n) {
    ItemCoord c = item_coord(G, n);
    CHECK(unit_of(G, c.b, c.kvh) == n / per_unit, "item %d in unit %d, dispensed as unit %d", n,
          unit_of(G, c.b, c.kvh), n / per_unit);
    if (n > 0 && (n % per_unit) != 0 && G.causal && !G.balanced) {
      const ItemCoord pc = item_coord(G, n - 1);
      CHECK(pc.r >= c.r, "item %d: shard %d after shard %d inside a unit", n, c.r, pc.r);
    }
    CHECK(c.g >= 0 && c.g < G.n_groups, "group %d", c.g);
    CHECK(c.b >= 0 && c.b < G.B && c.hq >= 0 && c.hq < G.Hq && c.r >= 0 && c.r < G.P, "coords item %d", n);
    CHECK(c.kvh == c.hq / G.gqa, "gqa mapping item %d", n);
    CHECK(c.qp >= 0 && c.qp < G.q_blocks, "qp item %d", n);
    const long long q_row = (long long)(c.b * G.Hq + c.hq) * G.S + (long long)c.r * G.L + (long long)c.qp * G.item_rows;
    for (int i = 0; i < G.item_qt; ++i) {
      const long long r0 = q_row + i * kTileRows;
      CHECK(r0 >= 0 && r0 + kTileRows <= rows_q, "q rows item %d", n);
      CHECK(r0 % kTileRows == 0, "q tile alignment");
      CHECK(covered[r0 / kTileRows] == 0, "q tile written twice (item %d)", n);
      covered[r0 / kTileRows] = 1;
    }
    long long it_tiles = 0;
    for (int t = 0; t < c.n_steps; ++t) {
      const int j = ((c.r - t) % G.P + G.P) % G.P;
      if (G.causal && !G.balanced) CHECK(j <= c.r, "causal chunk above the diagonal (item %d step %d)", n, t);
      const int n_kt = tiles_at_step(G, c, t);
      CHECK(n_kt >= (t == 0 ? 1 : 0) && n_kt <= G.kv_tiles, "tiles at step");
      if (G.causal) {
        // the tiles with a key visible to some row of the item are exactly 0 .. n_kt-1
        const long long q_lo = pos_of(G, c.r, (long long)c.qp * G.item_rows);
        long long q_hi = q_lo;
        for (int i = 0; i < G.item_qt; ++i)
          q_hi = std::max(q_hi, pos_of(G, c.r, (long long)c.qp * G.item_rows + i * kTileRows + kTileRows - 1));
        long long q_min = q_lo;
        for (int i = 0; i < G.item_qt; ++i)
          q_min = std::min(q_min, pos_of(G, c.r, (long long)c.qp * G.item_rows + i * kTileRows));
        for (int kt = 0; kt < G.kv_tiles; ++kt) {
          const long long k_lo = pos_of(G, j, (long long)kt * kTileRows);
          const long long k_hi = k_lo + kTileRows - 1;
          const bool any_visible = k_lo <= q_hi;
          CHECK(any_visible == (kt < n_kt), "item %d step %d tile %d: visible %d but read %d", n, t, kt,
                (int)any_visible, (int)(kt < n_kt));
          if (t > 0 && kt < n_kt) CHECK(k_hi <= q_min, "item %d step %d tile %d partly masked off step 0", n, t, kt);
        }
      }
      max_read[(size_t)c.g * G.P + t] = std::max(max_read[(size_t)c.g * G.P + t], n_kt);
      for (int kt = 0; kt < n_kt; ++kt) {
        if (t == 0) {
          const long long r0 = (long long)(c.b * G.Hkv + c.kvh) * G.S + (long long)j * G.L + (long long)kt * kTileRows;
          CHECK(r0 >= 0 && r0 + kTileRows <= rows_kv, "home kv rows item %d", n);
          // the home rows belong to chunk j of the item's own (b, kvh)
          CHECK(r0 / G.S == c.b * G.Hkv + c.kvh, "home kv head");
        } else {
          const long long r0 = (long long)(slot_of(t) * G.n_groups + c.g) * G.L + (long long)kt * kTileRows;
          CHECK(r0 >= 0 && r0 + kTileRows <= rows_slot, "slot rows item %d", n);
        }
        if (G.causal && t == 0) {
          // key tile kt of the local chunk vs the item's query tiles: no key tile lies
          // entirely above the diagonal of the item's last query tile
          const int q_first = c.qp * G.item_rows, key_first = kt * kTileRows;
          CHECK(key_first <= q_first + G.item_rows - kTileRows, "key tile masked for every query tile of the item");
        }
      }
      it_tiles += n_kt;
      if (t > 0) consumers[(size_t)c.g * G.P + t]++;
    }
    CHECK(it_tiles == item_tiles(G, c), "item_tiles mismatch item %d", n);
    tiles += it_tiles;
  }
  for (size_t i = 0; i < covered.size(); ++i) CHECK(covered[i] == 1, "q tile %zu never written", i);
  CHECK(tiles == total_tiles(G), "total_tiles %lld vs %lld", total_tiles(G), tiles);
  long long stage = 0, dyn = 0, pieces = 0, dyn_pieces = 0;
  for (int g = 0; g < G.n_groups; ++g) {
    const int ns = group_steps(G, g);
    for (int t = 1; t < ns; ++t) {
      CHECK(consumers[(size_t)g * G.P + t] == G.Gs, "group %d step %d consumers %d", g, t,
            consumers[(size_t)g * G.P + t]);
      ++stage;
      if (t > kRingSlots) ++dyn;
      int r_, b_, kvh_, sub_;
      group_coord(G, g, r_, b_, kvh_, sub_);
      CHECK(stage_tiles(G, r_, t) == max_read[(size_t)g * G.P + t], "group %d step %d stages %d tiles, items read %d",
            g, t, stage_tiles(G, r_, t), max_read[(size_t)g * G.P + t]);
      const int np = stage_pieces(G, r_, t);
      CHECK(np >= 1 && np <= G.n_pieces && (np - 1) * G.piece_tiles < stage_tiles(G, r_, t), "pieces of a step");
      pieces += np;
      if (t > kRingSlots) dyn_pieces += np;
      // staging source: chunk j of (b, kvh), L rows; destination slot slot_of(t) of g
      int r, b, kvh, sub;
      group_coord(G, g, r, b, kvh, sub);
      const int j = ((r - t) % G.P + G.P) % G.P;
      const long long src0 = (long long)(b * G.Hkv + kvh) * G.S + (long long)j * G.L;
      CHECK(src0 >= 0 && src0 + G.L <= rows_kv, "staging source rows");
      const long long dst0 = (long long)(slot_of(t) * G.n_groups + g) * G.L;
      CHECK(dst0 >= 0 && dst0 + G.L <= rows_slot, "staging destination rows");
    }
  }
  CHECK(stage == total_staging_tasks(G), "staging tasks %lld vs %lld", stage, total_staging_tasks(G));
  CHECK(dyn == dynamic_staging_tasks(G), "dynamic tasks %lld vs %lld", dyn, dynamic_staging_tasks(G));
  CHECK(pieces == total_staging_pieces(G), "staging pieces %lld vs %lld", pieces, total_staging_pieces(G));
  CHECK(dyn_pieces == dynamic_staging_pieces(G), "dynamic pieces %lld vs %lld", dyn_pieces,
        dynamic_staging_pieces(G));
  std::printf("OK items=%d groups=%d Gs=%d n_sub=%d tiles=%lld staging=%lld dynamic=%lld\n", G.n_items, G.n_groups,
              G.Gs, G.n_sub, tiles, stage, dyn);
  return 0;
}
