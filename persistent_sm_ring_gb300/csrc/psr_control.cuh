// Control block, partition controller and bounded waits shared by the persistent kernels
// (Ring Attention, AllGather+GEMM).  A kernel's parameter struct provides: ctrl, traj,
// timeout_ns, mode, n_s_init, n_stage_total, n_tiles_total, c_s0, c_p0, n_min, n_max,
// n_wave_items, n_wave_cap, update_headroom; its shared control struct provides a volatile
// `abort` word.
#pragma once
#include <cstdint>

#include "../../include/psr.h"
#include "psr_device.cuh"
#include "psr_schedule.h"

namespace psr {

constexpr int kTrajMax = 4096;

struct Ctrl {
  uint32_t item_next;     // compute items dispensed
  uint32_t init_next;     // static staging list: next piece to hand out (steps 1..kRingSlots of every group)
  uint32_t q_head;        // ready queue: next ticket
  uint32_t q_tail;        // ready queue: next entry to fill
  uint32_t target_ns;     // controller target + 1 (0 = not yet set)
  uint32_t error;         // first error site (0 = none)
  uint32_t abort;         // set on any error: every CTA drains and exits
  uint32_t ticks;         // completed tasks (controller period counter)
  uint32_t traj_len;
  uint32_t ns_min_inv, ns_max;  // 0xFFFF - min target, max target
  uint32_t ns_initial;
  uint32_t fault_count;
  uint32_t pad0[3];
  unsigned long long t0_ns;  // launch start (first CTA)
  unsigned long long last_eval_ns;  // last controller evaluation
  unsigned long long stage_cycles, compute_cycles;
  unsigned long long stage_done, compute_items, compute_tiles;
  unsigned long long stage_bytes;
  unsigned long long role_switches, idle_polls;
  unsigned long long starve_cycles;  // compute cycles spent waiting for staged ring steps (after a CTA's first item)
  // tracing build only (cycles summed over threads that record them)
  unsigned long long tr_softmax_wait, tr_softmax_busy, tr_mma_issue, tr_mma_wait_kv, tr_prod_wait_empty,
      tr_prod_wait_flag;
};
static_assert(sizeof(Ctrl) <= 256, "control block");

template <class KP>
__device__ __forceinline__ void raise_error(const KP& p, uint32_t site) {
  atomicCAS(&p.ctrl->error, 0u, site);
  st_release(&p.ctrl->abort, 1u);
}

// Bounded mbarrier wait: false on timeout or abort.  CL: the acquire also covers
// arrivals released by the other CTA of a pair.  `slack` multiplies the timeout, so that a
// wait downstream of another (a pipeline stage waiting for its producer) gives the root
// cause the first chance to be reported.
template <bool CL = false, class KP, class SC>
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const KP& p, SC* sc, uint32_t site,
                                         uint32_t slack = 1) {
  auto poll = [&]() { return CL ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (poll()) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (true) {
    if (poll()) return true;
    if ((++it & 15u) == 0) {
      if (sc->abort) return false;
      if (ld_relaxed(&p.ctrl->abort)) { sc->abort = 1; return false; }
      if (globaltimer_ns() - t0 > p.timeout_ns * slack) { raise_error(p, site); sc->abort = 1; return false; }
    }
  }
}

// Bounded wait until *flag >= want (gpu-scope acquire).
template <class KP, class SC>
__device__ __forceinline__ bool wait_flag(const uint32_t* flag, uint32_t want, uint32_t& seen, const KP& p, SC* sc,
                                          uint32_t site) {
  seen = ld_acquire(flag);
  if (seen >= want) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (true) {
    nanosleep_ns(64);
    seen = ld_acquire(flag);
    if (seen >= want) return true;
    if ((++it & 15u) == 0) {
      if (sc->abort) return false;
      if (ld_relaxed(&p.ctrl->abort)) { sc->abort = 1; return false; }
      if (globaltimer_ns() - t0 > p.timeout_ns) { raise_error(p, site); sc->abort = 1; return false; }
    }
  }
}

// ------------------------------------------------------------------------------------------------
// Controller (one thread, at task boundaries)
// ------------------------------------------------------------------------------------------------
template <class KP>
__device__ int current_target(const KP& p) {
  if (p.mode == PSR_STATIC) return p.n_s_init;
  const uint32_t t = ld_relaxed(&p.ctrl->target_ns);
  return t ? (int)(t - 1) : p.n_s_init;
}

constexpr unsigned long long kCtrlMinIntervalNs = 20000;  // re-evaluate at most every 20 us
#ifndef PSR_STAGE_HEADROOM
#define PSR_STAGE_HEADROOM 150
#endif
#ifndef PSR_STARVE_WEIGHT
#define PSR_STARVE_WEIGHT 50
#endif
// Staging capacity kept above the rule's balanced split (initial split and updates), and the
// share of compute cycles starved of staged data that is charged to staging.  Chosen on
// GB300 over the partition sweep and the headline (medians of 3 runs; alternatives: 2x
// initial only with full starvation charge, sweep geomean 1.025 / worst 1.14; 1.5x without
// starvation charge, 1.015 / 1.11; this setting 1.011 / 1.12, headline 1.016 / 1.012).
constexpr double kStageHeadroom = PSR_STAGE_HEADROOM / 100.0;
constexpr double kStarveWeight = PSR_STARVE_WEIGHT / 100.0;
#ifndef PSR_UPDATE_HEADROOM
#define PSR_UPDATE_HEADROOM 150
#endif
constexpr double kUpdateHeadroom = PSR_UPDATE_HEADROOM / 100.0;  // staging headroom in the updates

#ifndef PSR_WAVE_MARGIN
#define PSR_WAVE_MARGIN 110
#endif
// Staging capacity (over the balanced split) that the wave cap keeps: the cap is the largest
// split with the compute waves of the rule's split at this headroom.
constexpr double kWaveMargin = PSR_WAVE_MARGIN / 100.0;
#ifndef PSR_WAVE_MIN_TILES
#define PSR_WAVE_MIN_TILES 4
#endif
// Shortest ring step (KV tiles) for which the wave cap is applied.  Measured on GB300 (partition
// sweep, P = 32: 4-tile steps): once the staging tasks' control path stopped waiting on chains of
// L2 round trips, compute items there were no longer bound by step latency, the static optimum sat
// at the compute-wave boundary (48 of 152 stagers: the largest split with 10 waves), and the
// adaptive target without the cap rose to 72-75 (1.10-1.16x the best static time).  Two-tile steps
// (P = 64) are left out: there the cap does not bind under the default upper clamp anyway.
constexpr int kWaveMinTiles = PSR_WAVE_MIN_TILES;

#ifndef PSR_SHORT_STEP_HEADROOM
#define PSR_SHORT_STEP_HEADROOM 120
#endif
// Staging headroom, initial split and updates, on ring steps shorter than kWaveMinTiles KV tiles.
// There a compute item is bound by the latency of its ring steps: the time it waits for staged
// data is part of what it costs (it is not moved to the staging cost), and with that cost the
// rule needs little headroom.  Measured on GB300 (partition sweep, P = 64: 2-tile steps): with the
// waits moved to staging and 1.5x headroom the d = 64 point sat at the upper clamp, 1.04-1.07x the
// best static split (64 stagers); with the waits kept in the compute cost, 1.0x headroom fit d = 64
// (0.99x) but let d = 128 fall below its optimum (the clamp, 76: 1.11x), 1.2x held both within 1.04x.
constexpr double kShortStepHeadroom = PSR_SHORT_STEP_HEADROOM / 100.0;

// The initial split stands until this fraction of the compute tiles is done: it covers the
// ring's fill, when every active group needs its first staged steps at once and measured
// costs are still dominated by start-up.
constexpr double kCtrlHold = 0.1;

template <class KP>
__device__ void controller_update(const KP& p) {
  Ctrl* c = p.ctrl;
  {
    const unsigned long long now = globaltimer_ns();
    const unsigned long long last = ld_relaxed64(&c->last_eval_ns);
    if (now - last < kCtrlMinIntervalNs) return;
    if (atomicCAS(&c->last_eval_ns, last, now) != last) return;  // another CTA evaluates now
  }
  const unsigned long long sd = atomicAdd(&c->stage_done, 0ull);
  const unsigned long long td = atomicAdd(&c->compute_tiles, 0ull);
  const unsigned long long scy = atomicAdd(&c->stage_cycles, 0ull);
  const unsigned long long ccy = atomicAdd(&c->compute_cycles, 0ull);
  const double R_s = (double)(p.n_stage_total > sd ? p.n_stage_total - sd : 0);
  const double R_p = (double)(p.n_tiles_total > td ? p.n_tiles_total - td : 0);
  if ((double)td < kCtrlHold * (double)p.n_tiles_total) return;
  // measured cost per unit, blended with the prior until a few units are measured.
  // The staging cost per piece counts the staging CTAs' busy cycles plus the cycles
  // compute items spent starved of staged data: both are what staging costs the launch.
  const unsigned long long sv = atomicAdd(&c->starve_cycles, 0ull);
  const double C_s = (scy + kStarveWeight * (double)sv + (double)p.c_s0 * 4.0) / ((double)sd + 4.0);
  const double C_p = (ccy + (double)p.c_p0 * 64.0) / ((double)td + 64.0);
  int n = controller_rule((int)gridDim.x, R_s, (double)p.update_headroom * C_s, R_p, C_p, p.n_min, p.n_max);
  // equal-length compute items: the launch's wave cap holds while items remain unclaimed (a
  // CTA taken from compute then delays one of its items to an extra wave)
  if (n > p.n_wave_cap && ld_relaxed(&c->item_next) < p.n_wave_items) n = p.n_wave_cap;
  const int cur = current_target(p);
  // hysteresis (move only by a margin unless the staging work is finished) and a rate
  // limit (each evaluation moves the target by at most max(2, cur/8) CTAs): a CTA changes
  // role only at a task boundary, so a target that jumps around costs whole tasks
  const int margin = 1 + cur / 16;
  if (n != 0 && n > cur - margin && n < cur + margin) return;
  if (n == cur) return;
  if (n != 0) {
    const int step = cur / 8 > 2 ? cur / 8 : 2;
    if (n > cur + step) n = cur + step;
    if (n < cur - step) n = cur - step;
  }
  st_relaxed(&c->target_ns, (uint32_t)n + 1u);
  atomicMax(&c->ns_min_inv, 0xFFFFu - (uint32_t)n);
  atomicMax(&c->ns_max, (uint32_t)n);
  const uint32_t k = atomicAdd(&c->traj_len, 1u);
  if (k < (uint32_t)kTrajMax) {
    const unsigned long long now = globaltimer_ns();
    const unsigned long long t0 = c->t0_ns;
    p.traj[2 * k] = (uint32_t)((now > t0 ? now - t0 : 0) / 1000ull);
    p.traj[2 * k + 1] = (uint32_t)n;
  }
}

// Called by thread 0 of a CTA at its task boundaries: each CTA offers an evaluation at most
// every kCtrlMinIntervalNs of its own (no shared counter on the task path); controller_update
// then lets one CTA evaluate per interval.
template <class KP>
__device__ __forceinline__ void controller_tick(const KP& p, unsigned long long& next_offer_ns) {
  if (p.mode != PSR_ADAPTIVE) return;
  const unsigned long long now = globaltimer_ns();
  if (now < next_offer_ns) return;
  next_offer_ns = now + kCtrlMinIntervalNs;
  controller_update(p);
}

}  // namespace psr
