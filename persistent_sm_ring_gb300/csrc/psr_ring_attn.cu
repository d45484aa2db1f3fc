// Ring Attention forward as one persistent kernel on sm_103a.
//
// The mKernel pages (pwwt.cn analysis §2.2 Figure 2, §2.4, §2.6 Table 3;
// dataforcee/chathome kernel tables) describe a persistent kernel per GPU whose
// CTAs take specialised roles, move data at tile granularity, publish
// readiness flags that name completed payloads, and are re-split between roles
// by an on-GPU controller.  For Ring Attention the communication is a ring KV
// exchange in 128-row tiles ("TMA store KV") and the computation a local
// FlashAttention pass over the chunk received at the previous step.
//
// On one GPU the P ring ranks are P shards held in HBM:
//  * staging CTAs copy chunk (r - t) mod P of K and V into the ring slot
//    (t mod 3) of shard r with TMA bulk loads/stores through shared memory and
//    publish, per chunk, the count of completed 128-row tiles with a
//    gpu-scope release after the bulk stores have completed;
//  * compute units (one CTA, or a CTA pair when d = 128 and the shard length is a
//    multiple of 512) process query-row items across all ring steps of their
//    shard: step 0 reads the shard's own chunk in place, later steps read
//    the slot after acquiring its flag; QK^T and PV run on tcgen05 with the
//    accumulators in tensor memory (a pair runs M = 256 MMAs with each CTA
//    holding half of every K/V tile, which halves the K/V bytes each SM must
//    receive), the online softmax runs in two 128-thread warpgroups per CTA,
//    and the exact merge across chunks is the running max / sum of the online
//    softmax itself;
//  * the controller re-evaluates n_s* = N*(R_s*C_s)/(R_p*C_p + R_s*C_s) at task
//    boundaries from cycle-counter costs and remaining-work counters.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/psr.h"
#include "psr_device.cuh"
#include "psr_schedule.h"
#include "psr_control.cuh"
#include "psr_internal.h"

#ifndef PSR_TRACE
#define PSR_TRACE 0  // 1: accumulate per-role wait/compute cycles into the control block
#endif

namespace psr {

constexpr bool kTrace = PSR_TRACE != 0;
__device__ __forceinline__ long long trace_clock() { return kTrace ? clock64() : 0; }

// ------------------------------------------------------------------------------------------------
// Workspace: control block + protocol arrays + ring slots (all caller-owned device memory)
// ------------------------------------------------------------------------------------------------

struct WsLayout {
  size_t ctrl, flags, consumed, queue, io, traj, slot_k, slot_v, total, reset_bytes;
};

static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static WsLayout ws_layout(const Geometry& G) {
  WsLayout w;
  const size_t n_fc = (size_t)G.n_groups * G.P;
  size_t off = 0;
  w.ctrl = off; off += 256;
  w.traj = off; off = align_up(off + (size_t)kTrajMax * 8, 256);  // fixed offset: read without the shape
  w.flags = off; off = align_up(off + n_fc * G.n_pieces * 4, 256);  // per (group, step, piece)
  w.consumed = off; off = align_up(off + n_fc * 4, 256);
  w.queue = off; off = align_up(off + (size_t)(dynamic_staging_pieces(G) + 1) * 4, 256);
  w.io = off; off = align_up(off + (size_t)2 * unit_count(G) * 4, 256);  // per unit: inputs ready, items done
  w.reset_bytes = off;  // everything above is zeroed before each launch
  const size_t slot_elems = (size_t)kRingSlots * G.n_groups * G.L * G.d;
  w.slot_k = off; off = align_up(off + slot_elems * 2, 256);
  w.slot_v = off; off = align_up(off + slot_elems * 2, 256);
  w.total = off;
  return w;
}

// ------------------------------------------------------------------------------------------------
// Kernel parameters and per-D configuration
// ------------------------------------------------------------------------------------------------
struct KParams {
  Geometry geo;
  float scale_log2;  // scale * log2(e)
  const uint16_t* k;
  const uint16_t* v;
  uint16_t* slot_k;
  uint16_t* slot_v;
  uint16_t* o;
  float* lse;
  Ctrl* ctrl;
  uint32_t* flags;     // [n_groups][P][n_pieces]: completed tiles of each staging piece
  uint32_t* consumed;  // [n_groups][P]: items that have loaded the step's chunk
  uint32_t* queue;
  uint32_t* traj;
  unsigned long long timeout_ns;
  unsigned long long n_tiles_total;
  unsigned long long n_stage_total;  // staging pieces in the launch
  int n_dyn;          // ready-queue entries: pieces of the steps > kRingSlots
  int n_init;         // static list entries: pieces of steps 1..kRingSlots of every group
  int mode;           // PSR_STATIC / PSR_ADAPTIVE
  int n_s_init;
  int n_min, n_max;   // effective clamp
  int starve_charge;      // compute waits for staged data: moved to the staging cost (1) or kept (0)
  float update_headroom;  // staging headroom of the controller's updates
  uint32_t n_wave_items;  // items under the wave cap (0: none)
  int n_wave_cap;     // adaptive target bound while items remain unclaimed
  int fault;
  int lookahead;      // static list: groups ahead of the dispense frontier
  float c_s0, c_p0;   // prior costs (cycles per staging task / per tile) before measurements exist
  // Host-buffer entry only (nullptr otherwise): per unit (a batch, or a KV head with its query
  // heads), a word the upload stream sets once the unit's Q, K, V are in device memory, and the
  // count of the unit's items whose O and LSE are written (the download stream waits on it).
  const uint32_t* in_ready;
  uint32_t* out_done;
  int n_units;
};

// Warpgroup 0: warp 0 = TMA producer / staging / scheduler thread, warp 1 = MMA issuer (in a
// pair, the even CTA's only) and owner of the TMEM allocation, others idle.
// Warpgroups 1 and 2: softmax of the CTA's query tiles 0 and 1.
constexpr int kWarps = 12;
constexpr int kThreads = kWarps * 32;
// Registers: launched at kRegsLaunch per thread; warpgroup 0 gives registers to the softmax warpgroups.
constexpr int kRegsLaunch = 168, kRegsCtl = 72, kRegsSoftmax = 208;
static_assert(128 * kRegsCtl + 256 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split exceeds the launch");

// CG = CTAs per compute unit.  In a pair (CG = 2) each CTA holds half of every K tile
// (64 of its 128 rows) and half of every V tile (64 of its d = 128 columns): the B
// operands of the M = 256 MMAs are split along N between the two shared memories.
template <int D, int CG>
struct Cfg {
  static_assert(CG == 1 || (CG == 2 && D == 128), "CTA pairs are built for d = 128");
  static constexpr int QT = kTileRows * D * 2;  // bytes of one 128-row bf16 tile
  static constexpr int KVB = QT / CG;           // bytes of this CTA's share of one K or V tile
  static constexpr int NSTAGE = CG == 2 ? 10 : (D == 128 ? 5 : 12);
  static constexpr int NB = D == 128 ? 6 : 14;  // staging buffers of one K or V tile each
  static constexpr int SMEM = 1024 + 2 * QT + NSTAGE * KVB;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 256 + D;
  static constexpr uint32_t KBLK = (kTileRows / CG) * 128;  // bytes of one 64-column block of the K share
  static_assert(NB * QT <= 2 * QT + NSTAGE * KVB, "staging buffers must fit in the compute region");
  static_assert(NB <= 16, "staging barriers");
  // the MMA issuer acquires K_{j+1} before issuing PV(j): K_{j+1}'s stage was last used by load
  // 2j+2-NSTAGE, which must be released by MMAs already issued (V_{j-1} at the latest)
  static_assert(NSTAGE >= 3, "K/V stages");
  static_assert(SMEM <= 232448 - 512, "shared memory");
};

enum : int { CMD_EXIT = 0, CMD_COMPUTE = 1, CMD_STAGE = 2, CMD_IDLE = 3 };

// error sites
enum : uint32_t {
  SITE_NONE = 0, SITE_FLAG = 1, SITE_KV_FULL = 2, SITE_KV_EMPTY = 3, SITE_S_FULL = 4, SITE_P_FULL = 5,
  SITE_O_FULL = 6, SITE_Q_FULL = 7, SITE_STAGE_LOAD = 8, SITE_DRAIN = 9, SITE_QUEUE = 10, SITE_IDLE = 11,
  SITE_INPUT = 12
};



struct SmemCtl {
  uint64_t q_full[2];
  uint64_t kv_full[16];
  uint64_t kv_empty[16];
  uint64_t s_full[2];
  uint64_t p_full[2];     // [query tile]: P is in tensor memory (in every CTA)
  uint64_t o_full[2];
  uint64_t stg[16];
  uint64_t drain;
  uint32_t tmem_base;
  int cmd, arg;
  volatile uint32_t abort;
  uint32_t peer_held;  // pair: the odd CTA holds a ready-queue ticket (written by that CTA)
  uint32_t p_sink[4];  // pair: landing words of the odd CTA's P-ready signals (never read)
};

// Host-buffer entry: bounded wait until the unit's inputs are in device memory (the upload
// stream's write follows a system-wide fence after the copies), then order the async proxy's
// reads after it.
__device__ __forceinline__ bool wait_inputs(const KParams& p, SmemCtl* sc, int b, int kvh) {
  if (p.in_ready == nullptr) return true;
  uint32_t seen = 0;
  if (!wait_flag(p.in_ready + unit_of(p.geo, b, kvh), 1u, seen, p, sc, SITE_INPUT)) return false;
  fence_proxy_async_global();
  return true;
}



// ------------------------------------------------------------------------------------------------
// Task selection: thread 0 of a compute unit (the CTA, or the even CTA of a pair) picks the
// unit's role; a staging unit's CTAs then claim pieces each on its own.
// ------------------------------------------------------------------------------------------------
// Staging work comes from two lists, each claimed with one atomicAdd (a ticket):
//  * the static list: pieces of steps 1..kRingSlots of every group, in group order (their
//    slots are fresh); taken only while the group is within the lookahead window
//    of the compute dispense frontier;
//  * the ready queue: pieces of later steps, pushed by the compute CTA whose load
//    completed the consumption of the slot they overwrite.  A ticket names one
//    queue entry; the stager that holds it serves that entry once it has been
//    published and does static work meanwhile, so no stager ever blocks and no
//    claim ever retries.
// A task is (chunk * n_pieces + piece) with chunk = g*P + step.
struct StageTicket {
  int held = -1;     // queue entry this CTA owns, or -1
  bool done = false; // every queue entry has been handed out
};

// i0 / frontier_item: init_next and item_next as the caller last read them (its first attempt
// uses them; later attempts read again).
template <int BAL>
__device__ int claim_static_piece(const KParams& p, uint32_t i0, uint32_t frontier_item) {
  Ctrl* c = p.ctrl;
  const Geometry& G = p.geo;
  for (int attempt = 0; attempt < 8; ++attempt) {
    if (attempt > 0) {
      i0 = ld_relaxed(&c->init_next);
      frontier_item = ld_relaxed(&c->item_next);
    }
    if (i0 >= (uint32_t)p.n_init) return -1;
    const int g0 = (int)(i0 / ((uint32_t)kRingSlots * G.n_pieces));
    const int frontier = (int)(frontier_item / (uint32_t)G.Gs);
    if (g0 > frontier + p.lookahead) return -1;
    const uint32_t i = atomicAdd(&c->init_next, 1u);
    if (i >= (uint32_t)p.n_init) return -1;
    const int g = (int)(i / ((uint32_t)kRingSlots * G.n_pieces));
    const int step = 1 + (int)((i / G.n_pieces) % (uint32_t)kRingSlots);
    const int piece = (int)(i % G.n_pieces);
    int r, b, kvh, sub;
    group_coord<BAL>(G, g, r, b, kvh, sub);
    if (step < steps_of_shard<BAL>(G, r) && piece < stage_pieces<BAL>(G, r, step))
      return (g * G.P + step) * G.n_pieces + piece;
    // a shard with fewer steps, or a piece beyond the tiles the step needs: nothing to stage
    // for this entry; try the next one
  }
  return -1;
}

// sc != nullptr: a single staging CTA claiming its next piece while the current one's loads are in
// flight; it claims only while it is still a stager (the controller's target, or a held entry).
template <int BAL>
__device__ int try_claim_staging(const KParams& p, StageTicket& tk, const SmemCtl* sc = nullptr) {
  Ctrl* c = p.ctrl;
  // every word the branches below may read, loaded together: one round trip to L2 instead of
  // a chain of dependent ones (a staging task is a few microseconds, so this latency counts)
  const bool want_ticket = tk.held < 0 && !tk.done;
  const uint32_t e_held = tk.held >= 0 ? ld_relaxed(&p.queue[tk.held]) : 0u;
  const uint32_t i0 = ld_relaxed(&c->init_next);
  const uint32_t item = ld_relaxed(&c->item_next);
  const uint32_t qh = want_ticket ? ld_relaxed(&c->q_head) : 0u;
  if (sc != nullptr) {
    const uint32_t w_abort = ld_relaxed(&c->abort);
    const uint32_t w_target = p.mode == PSR_STATIC ? 0u : ld_relaxed(&c->target_ns);
    const int n_s = p.mode == PSR_STATIC ? p.n_s_init : (w_target ? (int)(w_target - 1) : p.n_s_init);
    if (sc->abort || w_abort) return -1;
    if ((int)blockIdx.x >= n_s && tk.held < 0) return -1;
  }
  if (e_held != 0) {
    fence_acq_rel_gpu();  // the entry was published with release: acquire it
    tk.held = -1;
    return (int)(e_held - 1);
  }
  const int t = claim_static_piece<BAL>(p, i0, item);
  if (t >= 0) return t;
  if (want_ticket) {
    if (qh >= (uint32_t)p.n_dyn) {
      tk.done = true;
    } else {
      const uint32_t h = atomicAdd(&c->q_head, 1u);
      if (h >= (uint32_t)p.n_dyn) {
        tk.done = true;
      } else {
        tk.held = (int)h;
        const uint32_t e = ld_acquire(&p.queue[h]);
        if (e != 0) {
          tk.held = -1;
          return (int)(e - 1);
        }
      }
    }
  }
  return -1;
}

// Role of the compute unit for its next task: CMD_STAGE (each CTA of the unit then claims a
// piece, or idles when none is claimable), CMD_COMPUTE with item `arg`, or CMD_EXIT.
// Unit u stages while u * CG < n_s (the controller's target counts CTAs).
template <int CG>
__device__ void decide(const KParams& p, SmemCtl* sc, bool& was_staging, const StageTicket& tk) {
  Ctrl* c = p.ctrl;
  // every control word the decision reads, loaded together (one round trip to L2)
  const uint32_t w_abort = ld_relaxed(&c->abort);
  const uint32_t w_target = p.mode == PSR_STATIC ? 0u : ld_relaxed(&c->target_ns);
  const uint32_t w_init = ld_relaxed(&c->init_next);
  const uint32_t w_qhead = ld_relaxed(&c->q_head);
  const uint32_t w_item = ld_relaxed(&c->item_next);
  if (sc->abort || w_abort) { sc->cmd = CMD_EXIT; return; }
  const int n_s = p.mode == PSR_STATIC ? p.n_s_init : (w_target ? (int)(w_target - 1) : p.n_s_init);
  const int unit = (int)blockIdx.x / CG;
  // a unit whose CTA owns a queue entry stages until that entry is served
  const bool held = tk.held >= 0 || (CG == 2 && sc->peer_held != 0);
  const bool staging_role = unit * CG < n_s || held;
  if (staging_role != was_staging) {
    atomicAdd(&c->role_switches, 1ull);
    was_staging = staging_role;
  }
  const bool all_claimed = !held && w_init >= (uint32_t)p.n_init && w_qhead >= (uint32_t)p.n_dyn;
  if (staging_role) {
    if (!all_claimed) { sc->cmd = CMD_STAGE; return; }
    if (p.mode == PSR_STATIC) { sc->cmd = CMD_EXIT; return; }
    // adaptive: nothing left to stage; fall through to compute
  }
  if (w_item < (uint32_t)p.geo.n_items) {
    const uint32_t n = atomicAdd(&c->item_next, 1u);
    if (n < (uint32_t)p.geo.n_items) { sc->cmd = CMD_COMPUTE; sc->arg = (int)n; return; }
  }
  // no compute left
  if (p.mode == PSR_STATIC || all_claimed) { sc->cmd = CMD_EXIT; return; }
  sc->cmd = CMD_STAGE;
}

// ------------------------------------------------------------------------------------------------
// Staging task (thread 0): chunk (r - step) mod P of K and V -> slot slot_of(step) of group g
// ------------------------------------------------------------------------------------------------
// A piece is copied as 2*n_kt units (K_kt and V_kt alternately), each a 128-row tile, through
// NB shared-memory buffers: a load waits only for the buffer's previous store to have read
// shared memory.  The piece's readiness flag (its tile count) is published
// once all of its stores have completed; when the same CTA goes on to stage another piece, that
// publication is deferred until the next piece's first loads are in flight, so that the store
// completion of one piece overlaps the loads of the next.
struct StagePending {
  uint32_t* flag = nullptr;
  uint32_t value = 0;
};

// Publish a deferred flag (thread 0 of a staging CTA; its bulk stores are the only ones pending).
__device__ __forceinline__ void publish_pending(StagePending& pend) {
  if (pend.flag == nullptr) return;
  bulk_wait<0>();              // every store of the piece has completed
  fence_proxy_async_global();  // async-proxy writes before the generic release
  st_release(pend.flag, pend.value);
  pend.flag = nullptr;
}

// tk != nullptr: once this piece's first loads are in flight, claim the next piece into *next
// (-1 if none), so that the claim's round trips to L2 overlap the copy.
template <int D, int CG, int BAL>
__device__ void run_staging(const KParams& p, SmemCtl* sc, uint32_t smem_base, int task, uint32_t (&stg_phase)[16],
                            StagePending& pend, StageTicket* tk, int* next) {
  using C = Cfg<D, CG>;
  const Geometry& G = p.geo;
  const int chunk = task / G.n_pieces, piece = task % G.n_pieces;
  const int g = chunk / G.P, step = chunk % G.P;
  int r, b, kvh, sub;
  group_coord<BAL>(G, g, r, b, kvh, sub);
  const int j = ((r - step) % G.P + G.P) % G.P;
  const size_t tile_elems = (size_t)kTileRows * D;
  const int kt0 = piece * G.piece_tiles;
  const int need = stage_tiles<BAL>(G, r, step);  // tiles of the chunk any item of the group reads
  const int n_kt = (need - kt0) < G.piece_tiles ? (need - kt0) : G.piece_tiles;
  const size_t src_off = ((size_t)(b * G.Hkv + kvh) * G.S + (size_t)j * G.L + (size_t)kt0 * kTileRows) * D;
  const size_t slot_off = (((size_t)slot_of(step) * G.n_groups + g) * (size_t)G.L + (size_t)kt0 * kTileRows) * D;
  uint32_t* flag = p.flags + (size_t)chunk * G.n_pieces + piece;
  if (!wait_inputs(p, sc, b, kvh)) {
    sc->abort = 1;
    return;
  }
  const bool drop = (p.fault == PSR_FAULT_DROP_FIRST_FLAG) && (atomicAdd(&p.ctrl->fault_count, 1u) == 0u);
  if (p.fault == PSR_FAULT_SLOW_STAGING) nanosleep_ns(20000);
  // staging "acquire": queue entries were published with release after the slot's
  // previous contents were consumed; order those async-proxy reads before our writes
  fence_proxy_async_global();

  constexpr int NB = C::NB;
  const int n_u = 2 * n_kt;  // unit u: tile u / 2 of K (u even) or V (u odd)
  auto src_of = [&](int u) { return ((u & 1) ? p.v : p.k) + src_off + (size_t)(u >> 1) * tile_elems; };
  auto dst_of = [&](int u) { return ((u & 1) ? p.slot_v : p.slot_k) + slot_off + (size_t)(u >> 1) * tile_elems; };
  auto issue_load = [&](int u) {
    const int bi = u % NB;
    mbar_expect_tx(&sc->stg[bi], C::QT);
    bulk_load(smem_base + bi * C::QT, src_of(u), C::QT, &sc->stg[bi]);
  };
  const int pre = n_u < NB - 1 ? n_u : NB - 1;
  for (int u = 0; u < pre; ++u) issue_load(u);
  int issued = pre;
  publish_pending(pend);  // the previous piece's stores complete while these loads are in flight
  if (tk != nullptr) *next = try_claim_staging<BAL>(p, *tk, sc);
  bool ok = true;
  for (int u = 0; u < n_u; ++u) {
    const int bi = u % NB;
    if (u >= issued) break;  // aborted: no more loads were issued
    if (ok && !wait_bar(&sc->stg[bi], stg_phase[bi] & 1u, p, sc, SITE_STAGE_LOAD)) ok = false;
    if (!ok) {
      // drain this load (bounded) so that no bulk copy targets shared memory after we leave
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&sc->stg[bi], stg_phase[bi] & 1u) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
    stg_phase[bi]++;
    if (ok) {
      bulk_store(dst_of(u), smem_base + bi * C::QT, C::QT);
      bulk_commit();
    }
    const int nu = u + NB - 1;
    if (nu < n_u && ok) {
      bulk_wait_read<1>();  // the store that used buffer nu % NB (unit u - 1) has read shared memory
      issue_load(nu);
      issued = nu + 1;
    }
  }
  if (ok && !drop) {
    pend.flag = flag;
    pend.value = (uint32_t)n_kt;
  } else {
    bulk_wait<0>();
  }
  atomicAdd(&p.ctrl->stage_bytes, (unsigned long long)n_kt * 2ull * C::QT);
}

// ------------------------------------------------------------------------------------------------
// Compute item: producer warp (TMA), MMA warp (tcgen05), two softmax warpgroups
// ------------------------------------------------------------------------------------------------
// Running counts over the CTA's lifetime; every thread keeps its own copy and
// advances it identically, so mbarrier phases agree across roles.
struct Counters {
  uint32_t kv;     // K/V tile loads (producer issues them, MMA consumes them)
  uint32_t items;  // items processed
  uint32_t tiles;  // KV tiles processed before the current item (S, P and O barrier phases)
};

// Tiled TMA load into this CTA's shared memory.  In a pair the completion is counted
// on the even CTA's mbarrier (bar_cl, a shared::cluster address), which therefore
// counts the bytes of both CTAs.
template <int CG>
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* tm, int x, int y, uint64_t* bar,
                                         uint32_t bar_cl) {
  if constexpr (CG == 1)
    tma_load_2d(dst, tm, x, y, bar);
  else
    tma_load_2d_pair(dst, tm, x, y, bar_cl);
}
// 128 rows x D columns as D/64 boxes of 64 columns, 16 KB apart (a Q tile, or a whole K/V tile)
template <int D, int CG>
__device__ __forceinline__ void load_rows128(const CUtensorMap* tm, uint32_t dst, int row, uint64_t* bar,
                                             uint32_t bar_cl) {
#pragma unroll
  for (int h = 0; h < D / 64; ++h) tma_load<CG>(dst + h * 16384, tm, 64 * h, row, bar, bar_cl);
}
// This CTA's share of K tile rows [row, row+128): all of it, or in a pair rows
// row + 64*rank .. +64 (the K tensor maps then have 64-row boxes), 8 KB per 64 columns.
template <int D, int CG>
__device__ __forceinline__ void load_k_share(const CUtensorMap* tm, uint32_t dst, int row, uint32_t rank,
                                             uint64_t* bar, uint32_t bar_cl) {
  if constexpr (CG == 1) {
    load_rows128<D, 1>(tm, dst, row, bar, bar_cl);
  } else {
#pragma unroll
    for (int h = 0; h < D / 64; ++h) tma_load<2>(dst + h * 8192, tm, 64 * h, row + 64 * (int)rank, bar, bar_cl);
  }
}
// This CTA's share of V tile rows [row, row+128): all of it, or in a pair the 64 columns
// 64*rank .. +64 (one box, 16 KB).
template <int D, int CG>
__device__ __forceinline__ void load_v_share(const CUtensorMap* tm, uint32_t dst, int row, uint32_t rank,
                                             uint64_t* bar, uint32_t bar_cl) {
  if constexpr (CG == 1)
    load_rows128<D, 1>(tm, dst, row, bar, bar_cl);
  else
    tma_load<2>(dst, tm, 64 * (int)rank, row, bar, bar_cl);
}

// Cycles an item spent waiting for readiness flags: all of them (not compute cost)
// and those that measure staging falling behind (charged to staging): every wait
// except during the CTA's first item, which overlaps the ring's fill at launch.
struct Starved {
  long long all = 0, late = 0;
};

// In a pair both CTAs run a producer for their own shares; only the even CTA's
// barriers count the bytes (for both) and only it sends "consumed" notifications.
template <int D, int CG, int BAL>
__device__ Starved producer(const KParams& p, SmemCtl* sc, uint32_t smem_base, const ItemCoord& it, uint32_t rank,
                              const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                              const CUtensorMap* tm_sk, const CUtensorMap* tm_sv, Counters& cnt) {
  using C = Cfg<D, CG>;
  const Geometry& G = p.geo;
  const bool leader = rank == 0;
  const uint32_t sQ = smem_base, sStage = smem_base + 2 * C::QT;
  auto bar_cl = [](uint64_t* b) -> uint32_t { return CG == 2 ? mapa_shared(smem_u32(b), 0) : 0u; };
  Starved starved;
  if (!wait_inputs(p, sc, it.b, it.kvh)) {
    sc->abort = 1;
    return starved;
  }
  // Q tiles (the barrier phase of q_full is the item count)
  const int q_row = (it.b * G.Hq + it.hq) * G.S + it.r * G.L + it.qp * G.item_rows + (int)rank * kCtaRows;
  for (int i = 0; i < 2; ++i) {
    if (leader) mbar_expect_tx(&sc->q_full[i], CG * C::QT);
    load_rows128<D, CG>(tm_q, sQ + i * C::QT, q_row + i * kTileRows, &sc->q_full[i], bar_cl(&sc->q_full[i]));
  }
  // pending "slot consumed" notifications: (step, load index of the step's last tile)
  int pend_step[4] = {0, 0, 0, 0};
  uint32_t pend_load[4] = {0, 0, 0, 0};
  int pend_n = 0;
  auto resolve_one = [&](bool blocking) -> bool {
    const uint32_t c = pend_load[0];
    const uint32_t stage = c % C::NSTAGE, par = (c / C::NSTAGE) & 1u;
    if (blocking) {
      if (!wait_bar(&sc->kv_full[stage], par, p, sc, SITE_KV_FULL)) return false;
    } else if (!mbar_test_wait(&sc->kv_full[stage], par)) {
      return false;
    }
    const int t = pend_step[0];
    fence_proxy_async_global();
    const uint32_t old = atom_add_acq_rel(p.consumed + (size_t)it.g * G.P + t, 1u);
    if (old + 1 == (uint32_t)G.Gs && t + kRingSlots < it.n_steps) {
      const uint32_t np = (uint32_t)stage_pieces<BAL>(G, it.r, t + kRingSlots);
      const uint32_t k = atomicAdd(&p.ctrl->q_tail, np);
      const uint32_t chunk = (uint32_t)(it.g * G.P + t + kRingSlots);
      if (k + np <= (uint32_t)p.n_dyn) {
        for (uint32_t pc = 0; pc < np; ++pc) st_release(p.queue + k + pc, chunk * (uint32_t)G.n_pieces + pc + 1u);
      } else {
        raise_error(p, SITE_QUEUE);
      }
    }
    for (int i = 1; i < pend_n; ++i) { pend_step[i - 1] = pend_step[i]; pend_load[i - 1] = pend_load[i]; }
    --pend_n;
    return true;
  };
  bool ok = true;
  unsigned long long tr_empty = 0;
  for (int t = 0; t < it.n_steps && ok; ++t) {
    const int j = ((it.r - t) % G.P + G.P) % G.P;
    const int n_kt = tiles_at_step<BAL>(G, it, t);
    const CUtensorMap* mk = t == 0 ? tm_k : tm_sk;
    const CUtensorMap* mv = t == 0 ? tm_v : tm_sv;
    const int row0 = t == 0 ? (it.b * G.Hkv + it.kvh) * G.S + j * G.L
                            : (slot_of(t) * G.n_groups + it.g) * G.L;
    const uint32_t* flags = p.flags + ((size_t)it.g * G.P + t) * G.n_pieces;
    uint32_t seen = 0;
    for (int kt = 0; kt < n_kt && ok; ++kt) {
      const int pc = kt / G.piece_tiles, in_pc = kt % G.piece_tiles;
      if (in_pc == 0) seen = 0;
      if (t > 0 && seen < (uint32_t)(in_pc + 1)) {
        const long long f0 = clock64();
        // The staging this wait depends on may itself wait for our own "consumed"
        // notifications: send every pending one (their loads are in flight) first.
        seen = ld_acquire(flags + pc);
        if (seen < (uint32_t)(in_pc + 1)) {
          while (ok && pend_n > 0)
            if (!resolve_one(true)) ok = false;
          if (!ok) break;
        }
        if (!wait_flag(flags + pc, (uint32_t)(in_pc + 1), seen, p, sc, SITE_FLAG)) { ok = false; break; }
        const long long waited = clock64() - f0;
        starved.all += waited;
        if (cnt.items > 0) starved.late += waited;
        fence_proxy_async_global();  // acquire (generic) before the async-proxy reads of the slot
      }
      for (int kv = 0; kv < 2; ++kv) {
        const uint32_t c = cnt.kv;
        const uint32_t stage = c % C::NSTAGE, fill = c / C::NSTAGE;
        // notifications whose stage is about to be refilled must be sent first
        while (pend_n > 0 && pend_load[0] + C::NSTAGE <= c) {
          if (!resolve_one(true)) { ok = false; break; }
        }
        if (!ok) break;
        if (pend_n > 0) resolve_one(false);
        const long long e0 = trace_clock();
        if (fill > 0 && !wait_bar(&sc->kv_empty[stage], (fill - 1) & 1u, p, sc, SITE_KV_EMPTY)) { ok = false; break; }
        tr_empty += trace_clock() - e0;
        if (leader) mbar_expect_tx(&sc->kv_full[stage], CG * C::KVB);
        const uint32_t dst = sStage + stage * C::KVB;
        if (kv == 0)
          load_k_share<D, CG>(mk, dst, row0 + kt * kTileRows, rank, &sc->kv_full[stage], bar_cl(&sc->kv_full[stage]));
        else
          load_v_share<D, CG>(mv, dst, row0 + kt * kTileRows, rank, &sc->kv_full[stage], bar_cl(&sc->kv_full[stage]));
        cnt.kv++;
      }
    }
    if (ok && t > 0 && leader) {
      if (pend_n == 4 && !resolve_one(true)) ok = false;
      pend_step[pend_n] = t;
      pend_load[pend_n] = cnt.kv - 1;
      ++pend_n;
    }
  }
  while (ok && pend_n > 0)
    if (!resolve_one(true)) ok = false;
  if (kTrace) {
    atomicAdd(&p.ctrl->tr_prod_wait_empty, tr_empty);
    atomicAdd(&p.ctrl->tr_prod_wait_flag, (unsigned long long)starved.all);
  }
  if (!ok) sc->abort = 1;
  return starved;
}

// Tensor-core issue (one thread; in a pair, the even CTA's, for both CTAs).  The tensor
// core's instruction queue is only a few MMAs deep, so the issuing thread stays busy
// for about as long as its MMAs run.  It issues for both query tiles, interleaved:
//   S0(0) S1(0) | PV0(j) S0(j+1) PV1(j) S1(j+1) | ...
// PV_i(j) reads P_i(j), which overlays S_i(j) in tensor memory, so S_i(j+1) is issued
// right behind it (tensor-core instructions of one thread run in order).
template <int D, int CG, int BAL>
__device__ void mma_issuer(const KParams& p, SmemCtl* sc, uint32_t smem_base, const ItemCoord& it, Counters& cnt) {
  using C = Cfg<D, CG>;
  const Geometry& G = p.geo;
  constexpr uint32_t M = kTileRows * CG;  // query rows per MMA: the pair's two tiles i stacked
  constexpr uint32_t IQK = idesc_bf16_f32(M, 128, false);
  constexpr uint32_t IPV = idesc_bf16_f32(M, D, true);
  constexpr uint32_t kHi = sdesc_hi_sw128(1024);  // 8-row (K-major) / 8-key (V, MN-major) groups 1024 B apart
  const uint32_t sStage = smem_base + 2 * C::QT;
  auto stage_of = [](uint32_t c) { return c % C::NSTAGE; };
  auto par_of = [](uint32_t c) { return (c / C::NSTAGE) & 1u; };
  auto issue_s = [&](int i, uint32_t kstage) {
    const uint32_t q_lo = sdesc_lo(smem_base + i * C::QT, 16);
    const uint32_t b_lo = sdesc_lo(sStage + kstage * C::KVB, 16);
    const uint32_t tS = sc->tmem_base + (i ? C::COL_S1 : C::COL_S0);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t a_off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
      const uint32_t b_off = ((kk / 4) * C::KBLK + (kk % 4) * 32) >> 4;
      mma_ss_cg<CG>(tS, q_lo + a_off, kHi, b_lo + b_off, kHi, IQK, kk > 0 ? 1u : 0u);
    }
    mma_commit_cg<CG>(&sc->s_full[i]);
    // a commit tracks every earlier MMA of this thread: one per K/V stage, after the second tile's
    // reads, releases the stage for both
    if (i == 1) mma_commit_cg<CG>(&sc->kv_empty[kstage]);
  };
  // PV_i(j): the K = 16 steps over the 128 keys of P_i(j)
  // O_i is only waited for at the end of the item (the rescale of a tile waits for that tile's S,
  // whose commit also tracks the previous PV_i), so only the item's last PV commits o_full
  auto issue_pv = [&](int i, uint32_t vstage, bool first, bool last, uint32_t parity) -> bool {
    // V share MN-major: 64-column halves 16 KB apart (a pair's CTA holds one half)
    const uint32_t b_lo = sdesc_lo(sStage + vstage * C::KVB, 16384);
    const uint32_t tS = sc->tmem_base + (i ? C::COL_S1 : C::COL_S0);
    const uint32_t tO = sc->tmem_base + (i ? C::COL_O1 : C::COL_O0);
    if (!wait_bar<CG == 2>(&sc->p_full[i], parity, p, sc, SITE_P_FULL)) return false;
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ts_cg<CG>(tO, tS + kk * 8, b_lo + kk * (2048 >> 4), kHi, IPV, (first && kk == 0) ? 0u : 1u);
    if (last) mma_commit_cg<CG>(&sc->o_full[i]);
    if (i == 1) mma_commit_cg<CG>(&sc->kv_empty[vstage]);
    return true;
  };
  const uint32_t n = (uint32_t)item_tiles<BAL>(G, it);
  uint32_t ck = cnt.kv;  // load index of K_0 of this item (the producer loads K_j, V_j alternately)
  cnt.kv += 2u * n;
  unsigned long long tr_issue = 0, tr_kv = 0;
  for (int i = 0; i < 2; ++i)
    if (!wait_bar(&sc->q_full[i], cnt.items & 1u, p, sc, SITE_Q_FULL)) { sc->abort = 1; return; }
  if (!wait_bar(&sc->kv_full[stage_of(ck)], par_of(ck), p, sc, SITE_KV_FULL)) { sc->abort = 1; return; }
  tc_fence_after();
  for (int i = 0; i < 2; ++i) issue_s(i, stage_of(ck));
  // K_{j+1} is acquired together with V_j, before the first block of the step: a wait between the
  // PV and QK^T halves of a block would let the tensor core's short queue run dry (measured on
  // GB300: each pause of the issuing thread costs the pipeline's refill on top of the wait).
  for (uint32_t jt = 0; jt < n; ++jt, ck += 2) {
    const uint32_t cv = ck + 1, cn = ck + 2;  // V_j, K_{j+1}
    const bool more = jt + 1 < n;
    const long long a0 = trace_clock();
    if (!wait_bar(&sc->kv_full[stage_of(cv)], par_of(cv), p, sc, SITE_KV_FULL)) { sc->abort = 1; return; }
    if (more && !wait_bar(&sc->kv_full[stage_of(cn)], par_of(cn), p, sc, SITE_KV_FULL)) { sc->abort = 1; return; }
    tr_kv += trace_clock() - a0;
    for (int i = 0; i < 2; ++i) {
      const long long a2 = trace_clock();
      if (!issue_pv(i, stage_of(cv), jt == 0, !more, (cnt.tiles + jt) & 1u)) { sc->abort = 1; return; }
      if (more) issue_s(i, stage_of(cn));
      tr_issue += trace_clock() - a2;
    }
  }
  if (kTrace) {
    atomicAdd(&p.ctrl->tr_mma_issue, tr_issue);
    atomicAdd(&p.ctrl->tr_mma_wait_kv, tr_kv);
  }
}

// Row maximum of 128 scores with three-input max (depth 5).
__device__ __forceinline__ float row_max128(const float (&s)[128]) {
  float v[43];
#pragma unroll
  for (int i = 0; i < 42; ++i) v[i] = fmax3(s[3 * i], s[3 * i + 1], s[3 * i + 2]);
  v[42] = fmaxf(s[126], s[127]);
  float w[15];
#pragma unroll
  for (int i = 0; i < 14; ++i) w[i] = fmax3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  w[14] = v[42];
  const float x0 = fmax3(w[0], w[1], w[2]), x1 = fmax3(w[3], w[4], w[5]), x2 = fmax3(w[6], w[7], w[8]);
  const float x3 = fmax3(w[9], w[10], w[11]), x4 = fmax3(w[12], w[13], w[14]);
  return fmaxf(fmax3(x0, x1, x2), fmaxf(x3, x4));
}

// p = 2^(s*sl2 - m) for scores [32*B0, 32*B1) of a row, written as bf16 pairs into TMEM
// columns [16*B0, 16*B1) at tP (16 columns at a time, so few packed values are live);
// the fp32 sums of p accumulate in acc.
template <int B0, int B1>
__device__ __forceinline__ void exp_blocks(const float (&s)[128], float sl2, float m, uint32_t tP, uint64_t (&acc)[4]) {
  const uint64_t scale2 = f2_pack(sl2, sl2), negm2 = f2_pack(-m, -m);
#pragma unroll
  for (int blk = B0; blk < B1; ++blk) {
    uint32_t pk[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int e = blk * 16 + q;
      const uint64_t x = fma2(f2_pack(s[2 * e], s[2 * e + 1]), scale2, negm2);
      float x0, x1;
      f2_unpack(x, x0, x1);
      const float y0 = ex2_approx(x0), y1 = ex2_approx(x1);
      acc[e & 3] = add2(acc[e & 3], f2_pack(y0, y1));
      pk[q] = pack_bf16x2(y0, y1);
    }
    tmem_st16(tP + blk * 16, pk);
  }
}
__device__ __forceinline__ float acc_sum(const uint64_t (&acc)[4]) {
  float a0, a1, b0, b1, c0, c1, d0, d1;
  f2_unpack(acc[0], a0, a1);
  f2_unpack(acc[1], b0, b1);
  f2_unpack(acc[2], c0, c1);
  f2_unpack(acc[3], d0, d1);
  return ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
}

// One softmax warpgroup per 128-row query tile i of the CTA (in a pair, CTA `rank`
// holds query tiles 2*rank and 2*rank + 1 of the item).
template <int D, int CG, int BAL>
__device__ void softmax_wg(const KParams& p, SmemCtl* sc, const ItemCoord& it, int i, uint32_t rank, Counters& cnt) {
  using C = Cfg<D, CG>;
  const Geometry& G = p.geo;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quarter = warp % 4;
  const int row = quarter * 32 + lane;  // TMEM lane = tile row
  const int tile = it.qp * G.item_qt + 2 * (int)rank + i;  // query tile within the shard
  const int q_local = tile * kTileRows + row;               // position within the shard
  // P ready: one arrival per warp; in a pair the odd CTA's warps signal the even CTA's
  // barrier with a 4-byte st.async each (16 bytes that its warp 0 expects)
  const uint32_t p_full_cl = CG == 2 ? mapa_shared(smem_u32(&sc->p_full[i]), 0) : 0u;
  const uint32_t p_sink_cl = CG == 2 ? mapa_shared(smem_u32(&sc->p_sink[quarter]), 0) : 0u;
  auto publish = [&]() {
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (CG == 1 || rank == 0) {
        if (CG == 2 && quarter == 0) mbar_expect_tx(&sc->p_full[i], 16);
        else mbar_arrive(&sc->p_full[i]);
      } else {
        st_async_signal(p_sink_cl, 1u, p_full_cl);
      }
    }
  };
  const uint32_t lane_base = sc->tmem_base + ((uint32_t)(quarter * 32) << 16);
  const uint32_t tS = lane_base + (i ? C::COL_S1 : C::COL_S0);
  const uint32_t tO = lane_base + (i ? C::COL_O1 : C::COL_O0);
  const float sl2 = p.scale_log2;
  float m_run = -INFINITY;  // running max in the log2-scaled domain
  float l_run = 0.0f;
  uint32_t jglob = 0;
  bool ok = true;
  unsigned long long tr_wait = 0, tr_busy = 0;
  for (int t = 0; t < it.n_steps && ok; ++t) {
    const int n_kt = tiles_at_step<BAL>(G, it, t);
    for (int kt = 0; kt < n_kt; ++kt, ++jglob) {
      const long long c0 = trace_clock();
      // tcgen05.ld/st below are warp-collective: every lane must take the same path
      ok = __all_sync(0xffffffffu, wait_bar(&sc->s_full[i], (cnt.tiles + jglob) & 1u, p, sc, SITE_S_FULL));
      if (!ok) break;
      const long long c1 = trace_clock();
      tr_wait += c1 - c0;
      tc_fence_after();
      float s[128];
      {
        uint32_t r[128];
        tmem_ld64(tS, r);
        tmem_ld64(tS + 64, r + 64);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 128; ++e) s[e] = __uint_as_float(r[e]);
      }
      // causal mask on the shard's own chunk: key position kt*128 + c > q_local.  Only key
      // tiles from this query tile's diagonal on (up to the item's last diagonal) can hold
      // masked keys; the test is per tile so that it is the same for every lane of the warp.
      const bool diag = G.causal && t == 0 && kt >= tile;
      if (diag) {
        const int lim = q_local - kt * kTileRows;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > lim) s[c] = -INFINITY;
      }
      const float m_tile = row_max128(s) * sl2;
      // raise the running max only when it grows by more than 2^8 (values below stay in range)
      const bool need = (jglob == 0) || (m_tile > m_run + 8.0f);
      const float m_new = need ? fmaxf(m_run, m_tile) : m_run;
      if (jglob > 0 && __any_sync(0xffffffffu, need)) {
        const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
        // PV_i of the previous tile has completed: the commit this tile's S was waited on tracks it
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tO + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          tmem_st32(tO + c * 32, r);
          tmem_st_wait();
        }
        l_run *= alpha;
      }
      m_run = m_new;
      const float m_use = m_run == -INFINITY ? 0.0f : m_run;
      uint64_t acc[4] = {0, 0, 0, 0};
      exp_blocks<0, 4>(s, sl2, m_use, tS, acc);
      publish();
      l_run += acc_sum(acc);
      tr_busy += trace_clock() - c1;
    }
  }
  if (kTrace && lane == 0) {
    atomicAdd(&p.ctrl->tr_softmax_wait, tr_wait);
    atomicAdd(&p.ctrl->tr_softmax_busy, tr_busy);
  }
  ok = __all_sync(0xffffffffu, ok);
  if (ok) {
    // epilogue: O / l -> bf16, LSE = (m + log2 l) * ln 2
    ok = __all_sync(0xffffffffu, wait_bar(&sc->o_full[i], cnt.items & 1u, p, sc, SITE_O_FULL));  // one phase per item
  }
  if (ok) {
    tc_fence_after();
    const float inv_l = 1.0f / l_run;
    const size_t row_id = (size_t)(it.b * G.Hq + it.hq) * G.S + (size_t)it.r * G.L + q_local;
    uint16_t* orow = p.o + row_id * D;
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      uint32_t r[64];
      tmem_ld64(tO + c * 64, r);
      tmem_ld_wait();
      uint4 v4[8];
      uint32_t* w = reinterpret_cast<uint32_t*>(v4);
#pragma unroll
      for (int e = 0; e < 32; ++e)
        w[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv_l, __uint_as_float(r[2 * e + 1]) * inv_l);
      uint4* dst = reinterpret_cast<uint4*>(orow + c * 64);
#pragma unroll
      for (int e = 0; e < 8; ++e) dst[e] = v4[e];
    }
    p.lse[row_id] = (m_run + log2f(l_run)) * 0.69314718055994530942f;
  } else {
    sc->abort = 1;
  }
}

// ------------------------------------------------------------------------------------------------
// The persistent kernel
// ------------------------------------------------------------------------------------------------
// Task boundary: every thread of the compute unit (the CTA, or both CTAs of a pair).
template <int CG>
__device__ __forceinline__ void unit_sync() {
  if constexpr (CG == 1)
    __syncthreads();
  else
    cluster_sync();
}
// The unit's command, written by thread 0 of the unit's first CTA before unit_sync().
template <int CG>
__device__ __forceinline__ void read_cmd(SmemCtl& sc, uint32_t rank, int& cmd, int& arg) {
  if (CG == 1 || rank == 0) {
    cmd = sc.cmd;
    arg = sc.arg;
  } else {
    cmd = (int)ld_shared_cluster(mapa_shared(smem_u32(&sc.cmd), 0));
    arg = (int)ld_shared_cluster(mapa_shared(smem_u32(&sc.arg), 0));
  }
}

template <int D, int CG, int BAL>
__global__ void __launch_bounds__(kThreads, 1)
    ring_attn_kernel(const __grid_constant__ KParams p, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_sk, const __grid_constant__ CUtensorMap tm_sv) {
  using C = Cfg<D, CG>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ SmemCtl sc;
  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sc.q_full[i], 1);
      mbar_init(&sc.s_full[i], 1);
      // one arrival per softmax warp of tile i (in a pair, the even CTA's four warps, the
      // first with the 16 bytes the odd CTA's warps send)
      mbar_init(&sc.p_full[i], 4);
      mbar_init(&sc.o_full[i], 1);
    }
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&sc.kv_full[s], 1);
      mbar_init(&sc.kv_empty[s], 1);  // committed once per fill, after both query tiles' reads
    }
    for (int s = 0; s < C::NB; ++s) mbar_init(&sc.stg[s], 1);
    mbar_init(&sc.drain, 1);
    sc.abort = 0;
    sc.peer_held = 0;
    fence_barrier_init();
    if (blockIdx.x == 0) {
      unsigned long long z = 0;
      atomicCAS(&p.ctrl->t0_ns, z, (unsigned long long)globaltimer_ns());
      p.ctrl->ns_initial = (uint32_t)p.n_s_init;
      atomicMax(&p.ctrl->ns_max, (uint32_t)p.n_s_init);
      atomicMax(&p.ctrl->ns_min_inv, 0xFFFFu - (uint32_t)p.n_s_init);
    }
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_sk);
    prefetch_tmap(&tm_sv);
  }
  if (warp == 1) {
    tmem_alloc_cg<CG>(&sc.tmem_base, C::TMEM_COLS);
    tmem_relinquish_cg<CG>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // the other CTA's barriers exist before any remote arrival
  tc_fence_after();
  // Each warpgroup role runs its own loop under its own register budget; the two
  // loops meet at the same unit barriers at every task boundary.
  Counters cnt{0, 0, 0};
  if (warp < 4) {
    regs_dec<kRegsCtl>();
    uint32_t stg_phase[16] = {};
    StagePending pend;  // thread 0: flag of the last staged piece, not yet published
    bool was_staging = false;
    StageTicket ticket;
    long long t_task = 0;
    Starved starved;
    uint64_t idle_since = 0;  // first idle poll of the current idle stretch (0 = not idle)
    unsigned long long next_offer_ns = 0;  // thread 0: next time this CTA may offer a controller evaluation
    while (true) {
      if (threadIdx.x == 0) {
        if (rank == 0) decide<CG>(p, &sc, was_staging, ticket);
        t_task = clock64();
      }
      unit_sync<CG>();
      int cmd, arg;
      read_cmd<CG>(sc, rank, cmd, arg);
      if (cmd == CMD_EXIT) break;
      int done_kind = cmd;  // thread 0: CMD_COMPUTE (accounted at the boundary below) or CMD_IDLE
      // a deferred publication waits only while this CTA goes straight on to another piece
      if (threadIdx.x == 0 && cmd != CMD_STAGE) publish_pending(pend);
      if (cmd == CMD_STAGE) {
        if (threadIdx.x == 0) {
          int task = try_claim_staging<BAL>(p, ticket);
          if (task >= 0) {
            // Consecutive pieces without returning to the task boundary (the CTA's other threads
            // wait there): a single CTA claims its next piece while the current one's loads are in
            // flight, and every piece is accounted for the controller as it ends.
            while (task >= 0) {
              int next = -1;
              run_staging<D, CG, BAL>(p, &sc, smem_base, task, stg_phase, pend, CG == 1 ? &ticket : nullptr, &next);
              const long long now = clock64();
              atomicAdd(&p.ctrl->stage_cycles, (unsigned long long)(now - t_task));
              atomicAdd(&p.ctrl->stage_done, 1ull);
              t_task = now;
              controller_tick(p, next_offer_ns);
              task = next;
            }
            done_kind = CMD_IDLE;  // accounted piece by piece above
            idle_since = 0;
          } else {
            publish_pending(pend);
            done_kind = CMD_IDLE;
            atomicAdd(&p.ctrl->idle_polls, 1ull);
            // a CTA that finds no claimable work for longer than the wait bound reports it
            const uint64_t now = globaltimer_ns();
            if (idle_since == 0) idle_since = now;
            else if (now - idle_since > p.timeout_ns) raise_error(p, SITE_IDLE);
            nanosleep_ns(500);
          }
          // the pair's role decision needs to know whether this CTA still holds a ticket
          if constexpr (CG == 2)
            if (rank == 1) st_shared_cluster(mapa_shared(smem_u32(&sc.peer_held), 0), ticket.held >= 0 ? 1u : 0u);
        }
      } else if (cmd == CMD_COMPUTE) {
        const ItemCoord it = item_coord<BAL>(p.geo, arg);
        if (warp == 0 && lane == 0)
          starved = producer<D, CG, BAL>(p, &sc, smem_base, it, rank, &tm_q, &tm_k, &tm_v, &tm_sk, &tm_sv, cnt);
        else if (warp == 1 && lane == 0 && rank == 0)
          mma_issuer<D, CG, BAL>(p, &sc, smem_base, it, cnt);
        cnt.items++;
        cnt.tiles += (uint32_t)item_tiles<BAL>(p.geo, it);
        if (threadIdx.x == 0) idle_since = 0;
      }
      tc_fence_before();
      unit_sync<CG>();
      tc_fence_after();
      if (threadIdx.x == 0 && done_kind != CMD_IDLE) {
        long long busy = clock64() - t_task;
        if (done_kind == CMD_COMPUTE && p.starve_charge) {
          busy -= starved.all;  // compute cost excludes waiting for staged data ...
          atomicAdd(&p.ctrl->starve_cycles, (unsigned long long)(starved.late > 0 ? starved.late : 0));  // ... charged to staging
        }
        const unsigned long long dt = (unsigned long long)(busy > 0 ? busy : 0);
        // cycles from every CTA of the unit (the cost of a tile in CTA-cycles); tiles and items once
        atomicAdd(&p.ctrl->compute_cycles, dt);
        if (rank == 0) {
          const ItemCoord it = item_coord<BAL>(p.geo, arg);
          atomicAdd(&p.ctrl->compute_tiles, (unsigned long long)item_tiles<BAL>(p.geo, it));
          atomicAdd(&p.ctrl->compute_items, 1ull);
          // the item's O and LSE rows (stored by the softmax warps before the unit barrier) are
          // released at system scope to the download stream
          if (p.out_done != nullptr && !sc.abort) red_add_release_sys(p.out_done + unit_of(p.geo, it.b, it.kvh), 1u);
        }
        controller_tick(p, next_offer_ns);
      }
    }
    // drain: every tcgen05 op issued by this CTA has completed before TMEM is released
    if (warp == 1 && lane == 0 && rank == 0) {
      mma_commit_cg<CG>(&sc.drain, 1);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&sc.drain, 0)) {
        if (globaltimer_ns() - t0 > 100000000ull) break;
      }
    }
    if (threadIdx.x == 0) {
      // a launch that gave up releases every unit's completion word, so that a download stream
      // waiting on one of them never waits for items that will not finish
      if (p.out_done != nullptr && (sc.abort || ld_relaxed(&p.ctrl->abort)))
        for (int u = 0; u < p.n_units; ++u) st_release_sys(p.out_done + u, 0x40000000u);
      publish_pending(pend);
      bulk_wait<0>();
      // every TMA load of a compute item has landed (normally already true); a pair's
      // loads are all counted on the even CTA's barriers
      if (rank == 0) {
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t s = 0; s < (uint32_t)C::NSTAGE && s < cnt.kv; ++s) {
          const uint32_t fills = (cnt.kv - s + C::NSTAGE - 1) / C::NSTAGE;  // loads that used stage s
          while (!mbar_try_wait(&sc.kv_full[s], (fills - 1) & 1u) && globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else {
    regs_inc<kRegsSoftmax>();
    while (true) {
      unit_sync<CG>();
      int cmd, arg;
      read_cmd<CG>(sc, rank, cmd, arg);
      if (cmd == CMD_EXIT) break;
      if (cmd == CMD_COMPUTE) {
        const ItemCoord it = item_coord<BAL>(p.geo, arg);
        softmax_wg<D, CG, BAL>(p, &sc, it, warp < 8 ? 0 : 1, rank, cnt);
        cnt.items++;
        cnt.tiles += (uint32_t)item_tiles<BAL>(p.geo, it);
      }
      tc_fence_before();
      unit_sync<CG>();
      tc_fence_after();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // neither CTA leaves while the other may still signal it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_cg<CG>(sc.tmem_base, C::TMEM_COLS);
}

// ------------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------------
struct DeviceInfo {
  int device = -1, n_sm = 0, cc_major = 0, cc_minor = 0;
};

static bool device_info(DeviceInfo& di) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  static std::mutex mu;
  static DeviceInfo cache[64];
  std::lock_guard<std::mutex> lk(mu);
  if (dev >= 0 && dev < 64 && cache[dev].device == dev) { di = cache[dev]; return true; }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return false;
  di.device = dev;
  di.n_sm = prop.multiProcessorCount;
  di.cc_major = prop.major;
  di.cc_minor = prop.minor;
  if (dev >= 0 && dev < 64) cache[dev] = di;
  return true;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// [rows][d] bf16, box = 64 columns x box_rows rows, 128-byte swizzle
static bool make_tmap(CUtensorMap* m, const void* base, long long rows, int d, int box_rows = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int max_group_items(int n_units) {
  // the compute units must be able to hold a whole group at once; leave room for
  // at least a quarter of the units to stage
  int m = n_units - n_units / 4 - 1;
  return m < 1 ? 1 : m;
}

#ifndef PSR_PAIRS
#define PSR_PAIRS 0
#endif
// CTAs per compute unit for a shape.  Built with PSR_PAIRS=1: CTA pairs for d = 128 when a
// shard holds whole 512-row items (a pair halves the K/V bytes each SM receives per flop).
// Off by default: measured on GB300 the pair kernel computes ~4 % slower per SM (the softmax
// of both CTAs gates every PV), and two staging CTAs of one pair copy at ~30 GB/s each
// against ~50 GB/s for single CTAs, so the single-CTA kernel is faster at every split.
static int units_cg(const psr_shape* sh, int n_cta) {
  // a pair item holds 2 * kCtaRows query rows; balanced shards need whole items in each half
  const int rows = (sh->causal == 2 ? 2 : 1) * 2 * kCtaRows;
  return (PSR_PAIRS && sh->d == 128 && sh->P > 0 && sh->S % sh->P == 0 && (sh->S / sh->P) % rows == 0 && n_cta >= 4)
             ? 2
             : 1;
}

static int shape_geometry(const psr_shape* sh, Geometry& G, int n_cta) {
  if (!sh) return PSR_ERR_ARG;
  if (sh->B < 1 || sh->Hq < 1 || sh->Hkv < 1 || sh->S < 1 || sh->P < 1) return PSR_ERR_ARG;
  if (sh->Hq % sh->Hkv != 0 || sh->S % sh->P != 0) return PSR_ERR_UNSUPPORTED;
  if (sh->d != 64 && sh->d != 128) return PSR_ERR_UNSUPPORTED;
  if (sh->causal < 0 || sh->causal > PSR_CAUSAL_BALANCED) return PSR_ERR_ARG;
  if (!(sh->scale == sh->scale)) return PSR_ERR_ARG;  // NaN
  const long long rows_q = (long long)sh->B * sh->Hq * sh->S;
  if (rows_q >= (1LL << 31) || rows_q * sh->d >= (1LL << 40)) return PSR_ERR_UNSUPPORTED;
  const int cg = units_cg(sh, n_cta);
  const int rc =
      geometry_init(G, sh->B, sh->Hq, sh->Hkv, sh->S, sh->P, sh->d, sh->causal, max_group_items(n_cta / cg), cg);
  if (rc == 1) return PSR_ERR_ARG;
  if (rc != 0) return PSR_ERR_UNSUPPORTED;
  if ((long long)kRingSlots * G.n_groups * G.L >= (1LL << 31)) return PSR_ERR_UNSUPPORTED;  // slot rows index with int32
  return PSR_OK;
}

template <int D, int CG, int BAL>
static cudaError_t launch(const KParams& kp, const CUtensorMap* maps, int n_cta, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  auto kern = ring_attn_kernel<D, CG, BAL>;
  std::call_once(once, [kern] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, CG>::SMEM);
    if (attr_err != cudaSuccess) return;
    // the warpgroup register split must fit inside what the launch allocates, or the
    // increasing warpgroups would wait forever: refuse to launch otherwise
    cudaFuncAttributes fa;
    attr_err = cudaFuncGetAttributes(&fa, kern);
    if (attr_err == cudaSuccess && fa.numRegs * kThreads < 128 * kRegsCtl + 256 * kRegsSoftmax)
      attr_err = cudaErrorInvalidConfiguration;
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_cta);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<D, CG>::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: they wait on each other
  attr[na].val.cooperative = 1;
  ++na;
  if (CG == 2) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
    // every pair must be resident at once
    int max_clusters = 0;
    cfg.attrs = attr + 1;
    cfg.numAttrs = 1;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (max_clusters * 2 < n_cta) return cudaErrorCooperativeLaunchTooLarge;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, kp, maps[0], maps[1], maps[2], maps[3], maps[4]);
  if (e != cudaSuccess && CG == 2) {
    // cooperative launch of clusters unavailable: the occupancy check above still
    // guarantees that all pairs fit on the device at once
    cudaGetLastError();
    cfg.attrs = attr + 1;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, kp, maps[0], maps[1], maps[2], maps[3], maps[4]);
  }
  return e;
}

// Streams of the host-buffer entry point, one set per device and process (created on first use,
// never freed); calls on one device serialise on a mutex.  err_host is pinned host memory that
// receives the launch's error word.
struct HostPipe {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev_start = nullptr;
  uint32_t* err_host = nullptr;
  std::mutex mu;
};

static HostPipe* host_pipe() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  static HostPipe pipes[64];
  static std::mutex init_mu;
  std::lock_guard<std::mutex> lk(init_mu);
  HostPipe& hp = pipes[dev];
  if (hp.err_host) return &hp;
  bool ok = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp.ev_start, cudaEventDisableTiming) == cudaSuccess;
  void* pinned = nullptr;
  ok = ok && cudaHostAlloc(&pinned, sizeof(uint32_t), cudaHostAllocDefault) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return nullptr;
  }
  hp.err_host = static_cast<uint32_t*>(pinned);
  return &hp;
}

// The driver's stream memory operations: a stream writes a word once its earlier copies have
// completed (with a system-wide fence before the write), or waits until a word reaches a value.
struct StreamMemOps {
  PFN_cuStreamWriteValue32_v11070 write = nullptr;
  PFN_cuStreamWaitValue32_v11070 wait = nullptr;
};

static const StreamMemOps& stream_mem_ops() {
  static StreamMemOps ops;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &f, 11070, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      ops.write = reinterpret_cast<PFN_cuStreamWriteValue32_v11070>(f);
    if (cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &f, 11070, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      ops.wait = reinterpret_cast<PFN_cuStreamWaitValue32_v11070>(f);
  });
  return ops;
}

}  // namespace psr

using namespace psr;

extern "C" {

const char* psr_status_string(int s) {
  switch (s) {
    case PSR_OK: return "ok";
    case PSR_ERR_ARG: return "invalid argument";
    case PSR_ERR_UNSUPPORTED: return "unsupported shape or device";
    case PSR_ERR_CUDA: return "CUDA runtime error";
    case PSR_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int psr_controller_target(int n_cta, double R_s, double C_s, double R_p, double C_p, int n_min, int n_max) {
  return controller_rule(n_cta, R_s, C_s, R_p, C_p, n_min, n_max);
}

int psr_num_ctas(void) {
  DeviceInfo di;
  if (!device_info(di)) return -PSR_ERR_CUDA;
  return di.n_sm;
}

static int ncta_for_sizing() {
  DeviceInfo di;
  if (device_info(di) && di.n_sm > 0) return di.n_sm;
  return 152;  // sizing without a device: the GB300's SM count
}

size_t psr_workspace_bytes(const psr_shape* sh) {
  Geometry G;
  if (shape_geometry(sh, G, ncta_for_sizing()) != PSR_OK) return 0;
  return ws_layout(G).total;
}

// The forward's argument checks short of the workspace, in the order the entry points apply
// them: null or misaligned tensors (PSR_ERR_ARG), the device (PSR_ERR_CUDA / PSR_ERR_UNSUPPORTED),
// then the shape (PSR_ERR_ARG / PSR_ERR_UNSUPPORTED).
static int fwd_prepare(const psr_shape* sh, const void* q, const void* k, const void* v, const void* o,
                       const void* lse, DeviceInfo& di, Geometry& G) {
  if (!sh || !q || !k || !v || !o || !lse) return PSR_ERR_ARG;
  for (const void* ptr : {q, k, v, o, lse})
    if ((reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return PSR_ERR_ARG;
  if (!device_info(di)) return PSR_ERR_CUDA;
  if (di.cc_major != 10 || di.cc_minor != 3) return PSR_ERR_UNSUPPORTED;
  return shape_geometry(sh, G, di.n_sm);
}

int psr_internal_fwd_check(const psr_shape* sh, const void* q, const void* k, const void* v, const void* o,
                           const void* lse, size_t* ws_need) {
  DeviceInfo di;
  Geometry G;
  const int rc = fwd_prepare(sh, q, k, v, o, lse, di, G);
  if (rc == PSR_OK && ws_need) *ws_need = ws_layout(G).total;
  return rc;
}

// Everything a forward launch needs, checked and encoded on the host (no CUDA work enqueued).
struct FwdLaunch {
  KParams kp;
  CUtensorMap tmaps[5];
  int n_cta = 0, cg = 1, d = 0;
  bool bal = false;
  uint8_t* ws = nullptr;
  WsLayout L;
};

static int fwd_setup(const psr_shape* sh, const void* q, const void* k, const void* v, void* o, float* lse,
                     void* workspace, size_t ws_bytes, const psr_partition* part, FwdLaunch& F) {
  if (!workspace) return PSR_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PSR_ERR_ARG;
  DeviceInfo di;
  Geometry G;
  int rc = fwd_prepare(sh, q, k, v, o, lse, di, G);
  if (rc != PSR_OK) return rc;
  const int cg = G.cg;
  const int n_cta = di.n_sm / cg * cg;  // whole pairs
  const int n_cunits = n_cta / cg;  // compute units (CTAs, or CTA pairs)
  const WsLayout L = ws_layout(G);
  if (ws_bytes < L.total) return PSR_ERR_ARG;
  KParams& kp = F.kp;

  psr_partition pt;
  if (part) pt = *part;
  else { pt.mode = PSR_ADAPTIVE; pt.n_staging = 0; pt.n_min = 0; pt.n_max = 0; pt.fault = 0; pt.timeout_ms = 0; }
  if (pt.mode != PSR_STATIC && pt.mode != PSR_ADAPTIVE) return PSR_ERR_ARG;
  if (pt.fault < 0 || pt.fault > PSR_FAULT_SLOW_STAGING) return PSR_ERR_ARG;

  memset(&kp, 0, sizeof(kp));
  kp.geo = G;
  kp.n_units = unit_count(G);
  const double scale = sh->scale > 0.0f ? (double)sh->scale : 1.0 / std::sqrt((double)sh->d);
  kp.scale_log2 = (float)(scale * 1.4426950408889634);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  kp.k = static_cast<const uint16_t*>(k);
  kp.v = static_cast<const uint16_t*>(v);
  kp.slot_k = reinterpret_cast<uint16_t*>(ws + L.slot_k);
  kp.slot_v = reinterpret_cast<uint16_t*>(ws + L.slot_v);
  kp.o = static_cast<uint16_t*>(o);
  kp.lse = lse;
  kp.ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  kp.flags = reinterpret_cast<uint32_t*>(ws + L.flags);
  kp.consumed = reinterpret_cast<uint32_t*>(ws + L.consumed);
  kp.queue = reinterpret_cast<uint32_t*>(ws + L.queue);
  kp.traj = reinterpret_cast<uint32_t*>(ws + L.traj);
  kp.timeout_ns = (unsigned long long)(pt.timeout_ms > 0 ? pt.timeout_ms : 2000) * 1000000ull;
  kp.n_tiles_total = (unsigned long long)total_tiles(G);
  kp.n_stage_total = (unsigned long long)total_staging_pieces(G);
  kp.n_dyn = (int)dynamic_staging_pieces(G);
  kp.n_init = kRingSlots * G.n_groups * G.n_pieces;
  kp.mode = pt.mode;
  kp.fault = pt.fault;
  // clamps (in CTAs; a unit stages while unit * cg < n_s): at least one stager while
  // staging remains; enough compute units to hold a group
  const int hard_max = n_cta - cg * (G.Gs + 1) < 1 ? 1 : n_cta - cg * (G.Gs + 1);
  // default upper clamp: at most half of the CTAs stage (a compute item's ring steps are
  // sequential, so compute throughput needs items in flight as well as staged data)
  int n_max = pt.n_max > 0 ? pt.n_max : (n_cta / 2 < hard_max ? n_cta / 2 : hard_max);
  if (n_max > hard_max) n_max = hard_max;
  int n_min = pt.n_min > 0 ? pt.n_min : 1;
  if (n_min > n_max) n_min = n_max;
  kp.n_min = n_min;
  kp.n_max = n_max;
  const bool any_staging = kp.n_stage_total > 0;
  // costs before any measurement (CTA-cycles), from GB300 measurements: a staging piece moves
  // 2*piece_rows*d*2 bytes at ~50 GB/s per SM (32 KB tile copies; ~33 GB/s for d = 64's 16 KB
  // ones) and takes no less than ~6500 cycles (its loads, stores and their completion do not
  // overlap with another piece's); a compute tile (a CTA's two query tiles against one KV tile:
  // QK^T and PV, 2 * 2*128*128*d flops) at ~60 % of an SM's dense bf16 rate (8192 flop/clk),
  // but no less than the ~2800 cycles two 128x128 softmax tiles take whatever d is
  const double piece_bytes = 2.0 * G.piece_tiles * kTileRows * G.d * 2.0;
  const double copy_cycles = piece_bytes / (G.d >= 128 ? 50e9 : 33e9) * 1.95e9;
  kp.c_s0 = (float)(copy_cycles > 6500.0 ? copy_cycles : 6500.0);
  const double mma_cycles = 2.0 * 2.0 * 2.0 * 128.0 * 128.0 * G.d / (0.6 * 8192.0);
  kp.c_p0 = (float)(cg * (mma_cycles > 2800.0 ? mma_cycles : 2800.0));
  // ring steps shorter than kWaveMinTiles tiles: items bound by their steps' latency (the
  // controller keeps their waits for staged data in the compute cost, with less headroom)
  const bool short_steps = G.kv_tiles < kWaveMinTiles;
  const double stage_headroom = short_steps ? kShortStepHeadroom : kStageHeadroom;
  int n_s;
  if (pt.mode == PSR_STATIC) {
    n_s = pt.n_staging;
    if (!any_staging) n_s = 0;
    else if (n_s < 1 || n_s > n_cta - 1) return PSR_ERR_ARG;
    // a group could never be fully resident
    if (any_staging && n_cunits - (n_s + cg - 1) / cg < G.Gs) return PSR_ERR_ARG;
  } else {
    // initial split: the rule on the prior costs with the staging cost raised by the headroom.  At launch every
    // active group needs its first staged steps at once, and later a group's staging can run
    // only a step or two ahead of its compute, so the stagers need capacity above the average
    // rate (measured best static splits for P = 4..16 sit 1.2-3x above the balanced split); the
    // measured costs and starvation then move the target.
    n_s = pt.n_staging > 0 ? pt.n_staging
                           : controller_rule(n_cta, (double)kp.n_stage_total, stage_headroom * kp.c_s0,
                                             (double)kp.n_tiles_total, kp.c_p0, n_min, n_max);
    if (!any_staging) n_s = 0;
    else {
      if (n_s < n_min) n_s = n_min;
      if (n_s > n_max) n_s = n_max;
    }
    // Equal-length items (no causal mask, single CTAs), staging paced by compute (steps
    // beyond the static list) and ring steps of at least kWaveMinTiles KV tiles: cap the
    // target at the largest split with the compute waves of the rule's split at the wave
    // margin, for the initial split and for every update while items remain unclaimed.  The
    // compute CTAs of the first wave fix the wave structure of the launch, so the cap has to
    // hold from the start.  With shorter steps an item's time is bound by the latency of its
    // ring steps and grows as staging capacity shrinks, so item time is not a constant and
    // the cap is not applied.
    if (any_staging && !G.causal && cg == 1 && kp.n_dyn > 0 && pt.n_staging <= 0 && G.kv_tiles >= kWaveMinTiles) {
      const int n_need = controller_rule(n_cta, (double)kp.n_stage_total, kWaveMargin * kp.c_s0,
                                         (double)kp.n_tiles_total, kp.c_p0, n_min, n_max);
      const int cap = wave_cap_groups(n_cta, n_need, wave_cap(n_cta, n_need, G.n_items), G.Gs);
      if (cap < n_max) {
        kp.n_wave_items = (uint32_t)G.n_items;
        kp.n_wave_cap = cap < n_min ? n_min : cap;
        if (n_s > kp.n_wave_cap) n_s = kp.n_wave_cap;
      }
    }
  }
  kp.n_s_init = n_s;
  kp.starve_charge = short_steps ? 0 : 1;
  kp.update_headroom = (float)(short_steps ? kShortStepHeadroom : kUpdateHeadroom);
  kp.lookahead = n_cunits / G.Gs + 2;

  CUtensorMap* maps = F.tmaps;
  const long long rows_q = (long long)G.B * G.Hq * G.S, rows_kv = (long long)G.B * G.Hkv * G.S;
  const long long rows_slot = (long long)kRingSlots * G.n_groups * G.L;
  // K maps: a pair's CTA loads 64 of every 128 K rows
  const int k_box = kTileRows / cg;
  if (!make_tmap(&maps[0], q, rows_q, G.d) || !make_tmap(&maps[1], k, rows_kv, G.d, k_box) ||
      !make_tmap(&maps[2], v, rows_kv, G.d) || !make_tmap(&maps[3], kp.slot_k, rows_slot, G.d, k_box) ||
      !make_tmap(&maps[4], kp.slot_v, rows_slot, G.d))
    return PSR_ERR_CUDA;
  F.n_cta = n_cta;
  F.cg = cg;
  F.d = G.d;
  F.bal = G.balanced != 0;
  F.ws = ws;
  F.L = L;
  return PSR_OK;
}

// The persistent launch itself (one kernel per d, compute unit and shard layout; CTA-pair kernels
// only in a library built with pairs).  The control words must have been cleared before it.
static int fwd_enqueue(const FwdLaunch& F, cudaStream_t st) {
  cudaError_t e;
#if PSR_PAIRS
  if (F.cg == 2)
    e = F.bal ? launch<128, 2, 1>(F.kp, F.tmaps, F.n_cta, st) : launch<128, 2, 0>(F.kp, F.tmaps, F.n_cta, st);
  else
#endif
  if (F.d == 128)
    e = F.bal ? launch<128, 1, 1>(F.kp, F.tmaps, F.n_cta, st) : launch<128, 1, 0>(F.kp, F.tmaps, F.n_cta, st);
  else
    e = F.bal ? launch<64, 1, 1>(F.kp, F.tmaps, F.n_cta, st) : launch<64, 1, 0>(F.kp, F.tmaps, F.n_cta, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PSR_ERR_CUDA;
  }
  return PSR_OK;
}

int psr_ring_attn_fwd(const psr_shape* sh, const void* q, const void* k, const void* v, void* o, float* lse,
                      void* workspace, size_t ws_bytes, const psr_partition* part, void* stream) {
  FwdLaunch F;
  const int rc = fwd_setup(sh, q, k, v, o, lse, workspace, ws_bytes, part, F);
  if (rc != PSR_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(F.ws, 0, F.L.reset_bytes, st) != cudaSuccess) return PSR_ERR_CUDA;
  return fwd_enqueue(F, st);
}

int psr_ring_attn_fwd_host(const psr_shape* sh, const void* q_host, const void* k_host, const void* v_host,
                           void* o_host, float* lse_host, void* dq, void* dk, void* dv, void* d_o, float* d_lse,
                           void* workspace, size_t ws_bytes, const psr_partition* part, void* stream) {
  if (!sh || !q_host || !k_host || !v_host || !o_host || !lse_host) return PSR_ERR_ARG;
  // the launch over the device buffers (checks the shape, the device pointers and the workspace)
  FwdLaunch F;
  int rc = fwd_setup(sh, dq, dk, dv, d_o, d_lse, workspace, ws_bytes, part, F);
  if (rc != PSR_OK) return rc;
  const StreamMemOps& mem_ops = stream_mem_ops();
  if (!mem_ops.write || !mem_ops.wait) return PSR_ERR_UNSUPPORTED;
  const Geometry& G = F.kp.geo;
  // Units: one batch (B > 1), or one KV head with its query heads (B = 1).  Each unit's Q, K, V is
  // one contiguous block of each tensor, and so is its O and LSE.
  const int n_units = unit_count(G);
  const size_t row_b = (size_t)G.S * G.d * 2;  // bytes of one head's rows of Q, K, V or O
  const size_t q_u = (size_t)(G.B > 1 ? G.Hq : G.gqa) * row_b;
  const size_t kv_u = (size_t)(G.B > 1 ? G.Hkv : 1) * row_b;
  const size_t l_u = (size_t)(G.B > 1 ? G.Hq : G.gqa) * G.S * 4;
  const uint32_t items_per_unit = (uint32_t)(G.n_items / n_units);
  uint32_t* in_ready = reinterpret_cast<uint32_t*>(F.ws + F.L.io);
  uint32_t* out_done = in_ready + n_units;
  F.kp.in_ready = in_ready;
  F.kp.out_done = out_done;

  HostPipe* hp = host_pipe();
  if (!hp) return PSR_ERR_CUDA;
  std::lock_guard<std::mutex> lk(hp->mu);  // the pipeline's streams and error word are per device
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Every failure after the first enqueue ends here: copies already queued still read the caller's
  // host buffers (or write o_host / lse_host), so they are drained before returning.  A launch
  // that gave up releases every unit's completion word, so the download stream's waits end too.
  auto fail = [&](int status) {
    cudaStreamSynchronize(hp->h2d);
    cudaStreamSynchronize(st);
    cudaStreamSynchronize(hp->d2h);
    cudaGetLastError();
    return status;
  };
  // control words (and the units' words) cleared on the caller's stream; the uploads start after
  // that and after any work already queued there
  if (cudaMemsetAsync(F.ws, 0, F.L.reset_bytes, st) != cudaSuccess) return PSR_ERR_CUDA;
  if (cudaEventRecord(hp->ev_start, st) != cudaSuccess || cudaStreamWaitEvent(hp->h2d, hp->ev_start, 0) != cudaSuccess)
    return fail(PSR_ERR_CUDA);
  // one launch for the whole shape: its items wait (bounded) for their unit's inputs
  rc = fwd_enqueue(F, st);
  if (rc != PSR_OK) return fail(rc);
  // Backstop behind the launch on the same stream: once the kernel has finished, every unit's
  // completion word is set far above its item count (bytes 0x40: 0x40404040), so the download
  // stream's waits end even if a launch that gave up had not released them.  After a normal
  // launch the words are already complete and the copies read finished results either way.
  if (cudaMemsetAsync(out_done, 0x40, (size_t)n_units * 4, st) != cudaSuccess) return fail(PSR_ERR_CUDA);
  for (int u = 0; u < n_units; ++u) {
    const size_t qo = (size_t)u * q_u, ko = (size_t)u * kv_u;
    if (cudaMemcpyAsync(static_cast<uint8_t*>(dq) + qo, static_cast<const uint8_t*>(q_host) + qo, q_u,
                        cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<uint8_t*>(dk) + ko, static_cast<const uint8_t*>(k_host) + ko, kv_u,
                        cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<uint8_t*>(dv) + ko, static_cast<const uint8_t*>(v_host) + ko, kv_u,
                        cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess ||
        mem_ops.write(reinterpret_cast<CUstream>(hp->h2d), reinterpret_cast<CUdeviceptr>(in_ready + u), 1u,
                      CU_STREAM_WRITE_VALUE_DEFAULT) != CUDA_SUCCESS)
      return fail(PSR_ERR_CUDA);
  }
  // each unit's results are copied out as soon as all of its items are done
  for (int u = 0; u < n_units; ++u) {
    const size_t qo = (size_t)u * q_u, lo = (size_t)u * l_u;
    if (mem_ops.wait(reinterpret_cast<CUstream>(hp->d2h), reinterpret_cast<CUdeviceptr>(out_done + u),
                     items_per_unit, CU_STREAM_WAIT_VALUE_GEQ) != CUDA_SUCCESS ||
        cudaMemcpyAsync(static_cast<uint8_t*>(o_host) + qo, static_cast<const uint8_t*>(d_o) + qo, q_u,
                        cudaMemcpyDeviceToHost, hp->d2h) != cudaSuccess ||
        cudaMemcpyAsync(reinterpret_cast<uint8_t*>(lse_host) + lo, reinterpret_cast<const uint8_t*>(d_lse) + lo, l_u,
                        cudaMemcpyDeviceToHost, hp->d2h) != cudaSuccess)
      return fail(PSR_ERR_CUDA);
  }
  // the launch's error word, once it has finished
  if (cudaMemcpyAsync(hp->err_host, F.ws + offsetof(Ctrl, error), 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return fail(PSR_ERR_CUDA);
  if (cudaStreamSynchronize(hp->d2h) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess ||
      cudaStreamSynchronize(hp->h2d) != cudaSuccess)
    return fail(PSR_ERR_CUDA);
  return *hp->err_host != 0 ? PSR_ERR_TIMEOUT : PSR_OK;
}

int psr_get_stats(const void* workspace, psr_stats* out, void* stream) {
  if (!workspace || !out) return PSR_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return PSR_ERR_CUDA;
  Ctrl c;
  if (cudaMemcpy(&c, workspace, sizeof(Ctrl), cudaMemcpyDeviceToHost) != cudaSuccess) return PSR_ERR_CUDA;
  memset(out, 0, sizeof(*out));
  out->status = c.error ? PSR_ERR_TIMEOUT : PSR_OK;
  out->error_site = (int)c.error;
  out->n_cta = psr_num_ctas();
  out->n_s_final = c.target_ns ? (int)c.target_ns - 1 : -1;
  out->n_s_min = (int)(0xFFFFu - c.ns_min_inv);
  out->n_s_max = (int)c.ns_max;
  out->traj_len = (int)(c.traj_len < (uint32_t)kTrajMax ? c.traj_len : kTrajMax);
  out->staging_cycles = c.stage_cycles;
  out->compute_cycles = c.compute_cycles;
  out->staging_tasks = c.stage_done;
  out->compute_items = c.compute_items;
  out->compute_tiles = c.compute_tiles;
  out->staging_bytes = c.stage_bytes;
  out->role_switches = c.role_switches;
  out->idle_polls = c.idle_polls;
  out->trace_softmax_wait = c.tr_softmax_wait;
  out->trace_softmax_busy = c.tr_softmax_busy;
  out->trace_mma_issue = c.tr_mma_issue;
  out->trace_mma_wait_kv = c.tr_mma_wait_kv;
  out->trace_producer_wait_empty = c.tr_prod_wait_empty;
  out->trace_producer_wait_flag = c.tr_prod_wait_flag;
  out->n_s_initial = (int)c.ns_initial;
  if (out->n_s_final < 0) out->n_s_final = out->n_s_initial;
  return out->status;
}

int psr_get_trajectory(const void* workspace, uint32_t* out_pairs, int max_entries, void* stream) {
  if (!workspace || (!out_pairs && max_entries > 0) || max_entries < 0) return -PSR_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return -PSR_ERR_CUDA;
  Ctrl c;
  if (cudaMemcpy(&c, workspace, sizeof(Ctrl), cudaMemcpyDeviceToHost) != cudaSuccess) return -PSR_ERR_CUDA;
  int n = (int)(c.traj_len < (uint32_t)kTrajMax ? c.traj_len : kTrajMax);
  if (n > max_entries) n = max_entries;
  if (n > 0 && cudaMemcpy(out_pairs, static_cast<const uint8_t*>(workspace) + 256, (size_t)n * 8,
                          cudaMemcpyDeviceToHost) != cudaSuccess)
    return -PSR_ERR_CUDA;
  return n;
}

}  // extern "C"
