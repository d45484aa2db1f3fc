"""Benchmark: Ring Attention forward on GB300 (one JSON line on rank 0).

Workload (the headline case): B=1, H=32, S=32768 as P=16 shards of 2048, d=128,
bf16 Q,K,V ~ N(0,1) seeded (synthetic), scale 1/sqrt(128); one step = one
non-causal pass followed by one causal pass, each a single persistent launch.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --sweep [d]      # partition-stress sweep: static 2..64 staging CTAs vs adaptive
  python bench.py --ag-gemm        # AllGather+GEMM, M8192 K8192 N28672 over 8 ranks
  python bench.py --gemm-rs        # GEMM+ReduceScatter, M8192 N8192 K28672 over 8 ranks
  python bench.py --bwd            # Ring Attention backward, B1 H32 S32768 P16 d128

value: algorithmic TFLOP/s over the timed steps (4*d flops per unmasked
(query, key) pair), inputs resident in HBM (805 MB per pass, larger than L2).
e2e: the same metric through psr_ring_attn_fwd_host (pinned host buffers;
H2D of Q,K,V and D2H of O,LSE inside the timed region).
--impl reference: the fp64 CPU oracle on a bounded row sample of the same
workload, on this machine's host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ring-attn fwd TFLOP/s (bf16, 1 GB300) and % of dense BF16 peak; ms/pass"
WORKLOADS = ("h32_s32k_nc", "h32_s32k_c")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
PROFILE = os.path.join(ROOT, "profiles", "ring_attn_kernel_h32_s32k.md")
KERNEL_SOURCES = [os.path.join(ROOT, "persistent_sm_ring_gb300", "csrc", f)
                  for f in ("psr_ring_attn.cu", "psr_device.cuh", "psr_schedule.h", "psr_control.cuh")]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    except Exception:
        return dict(FALLBACK_PEAKS)


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the main kernel from the committed ncu summary, if it
    was captured on the current kernel source; else None."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    m_sha = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b or m_sha.group(1) != kernel_source_sha():
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.reader.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------------------------
# distributed plumbing (one process per GPU; each rank runs an independent replica)
# ------------------------------------------------------------------------------------------------

def dist_init(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_sum(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded row sample
# ------------------------------------------------------------------------------------------------

def oracle_rows_flops(w, rows):
    import numpy as np
    i = rows % w.S
    keys = (i + 1) if w.causal else np.full_like(i, w.S)
    return float(4.0 * w.d * keys.sum())


def cpu_baseline(workloads, inputs, budget_s=12.0):
    """Time the fp64 oracle on seeded sampled rows of each workload; TFLOP/s of algorithmic work."""
    import numpy as np

    import oracle
    cores = oracle.default_threads()
    flops = 0.0
    secs = 0.0
    n_rows_total = 0
    per = budget_s / len(workloads)
    for w, (q, k, v) in zip(workloads, inputs):
        rng = np.random.default_rng(w.seed + 99)
        n = max(cores, 64)
        while True:  # calibrate, then fill the budget share
            rows = np.sort(rng.choice(w.B * w.Hq * w.S, size=n, replace=False)).astype(np.int64)
            t0 = time.perf_counter()
            oracle.for_workload(w, q, k, v, rows=rows, n_threads=cores)
            dt = time.perf_counter() - t0
            if dt >= per * 0.5 or n >= w.B * w.Hq * w.S // 4:
                break
            n = int(min(w.B * w.Hq * w.S // 4, max(2 * n, n * per * 0.7 / max(dt, 1e-3))))
        flops += oracle_rows_flops(w, rows)
        secs += dt
        n_rows_total += len(rows)
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{n_rows_total} seeded query rows of {'+'.join(w.name for w in workloads)} "
                      f"(fp64, every allowed key), {secs:.1f} s"}


# ------------------------------------------------------------------------------------------------
# every workload: the five configurations, each timed on its own
# ------------------------------------------------------------------------------------------------

# (configuration, workloads): 1 the small case, 2 the headline (both passes), 3 GQA causal, 4 the
# long causal sequence with outlier keys, 5 the partition-stress grid (adaptive partition)
CONFIGS = (("1", ("small",)), ("2", ("h32_s32k_nc", "h32_s32k_c")), ("3", ("gqa_s64k_c",)),
           ("4", ("long_s128k_c",)),
           ("5", tuple(f"sweep_d{d}_P{P}" for d in (64, 128) for P in (2, 4, 8, 16, 32, 64))))


def algorithmic_bytes(w) -> int:
    """HBM bytes a pass must move: Q, K, V read once, O and LSE written once, and every ring
    transfer read from the chunk's home and written into its slot."""
    return 2 * (w.n_q + 2 * w.n_kv) + 2 * w.n_q + 4 * w.B * w.Hq * w.S + 2 * w.staging_bytes()


def roofline_of(w, ms, peaks):
    """Roofline time of a pass (tensor flops at the measured bf16 peak, or its bytes at the measured
    HBM bandwidth, whichever is longer) over its measured time."""
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    t_flops = w.flops() / (peak * 1e12)
    t_bytes = algorithmic_bytes(w) / (hbm * 1e9)
    bound = "tensor" if t_flops >= t_bytes else "hbm"
    return bound, max(t_flops, t_bytes) / (ms / 1e3)


def time_configs(psr, torch, peaks, passes_small=50, budget_ms=400.0):
    """Median CUDA-event time of each configuration's pass (adaptive partition, inputs resident in
    HBM), with TFLOP/s, the fraction of the measured bf16 peak, the roofline fraction and the
    staging rate.  One input set is resident at a time."""
    import ring_inputs as ri
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    stream = torch.cuda.current_stream()
    part = psr.make_partition(psr.ADAPTIVE)
    out = []
    key_now, tensors = None, None
    for cfg, names in CONFIGS:
        for name in names:
            w = ri.WORKLOADS[name]
            key = (w.B, w.Hq, w.Hkv, w.S, w.d, w.seed, w.qmul, w.kmul, w.outlier_frac)
            if key != key_now:
                tensors = None
                torch.cuda.empty_cache()
                host = [torch.empty(shape, dtype=torch.int16).pin_memory()
                        for shape in ((w.B, w.Hq, w.S, w.d), (w.B, w.Hkv, w.S, w.d), (w.B, w.Hkv, w.S, w.d))]
                ri.generate(w, *(t.data_ptr() for t in host))
                tensors = [t.cuda().view(torch.bfloat16) for t in host]
                del host
                key_now = key
            q, k, v = tensors
            o = torch.empty_like(q)
            lse = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32, device=q.device)
            ws = torch.empty(psr.workspace_bytes(psr.make_shape(w.B, w.Hq, w.Hkv, w.S, w.P, w.d, w.causal)),
                             dtype=torch.uint8, device=q.device)

            def one():
                psr.ring_attn_fwd(q, k, v, P=w.P, causal=w.causal, scale=w.scale, partition=part, workspace=ws,
                                  out=o, lse=lse, stream=stream)
            for _ in range(3):
                one()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            one()
            torch.cuda.synchronize()
            est_ms = 1e3 * (time.perf_counter() - t0)
            reps = passes_small if est_ms < 1.0 else int(min(20, max(5, budget_ms / max(est_ms, 1e-3))))
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for e0, e1 in ev:
                e0.record(stream)
                one()
                e1.record(stream)
            torch.cuda.synchronize()
            st = psr.get_stats(ws)
            if st["status"] != 0:
                raise RuntimeError(f"{name}: device status {st['status']} site {st['error_site']}")
            times = sorted(e0.elapsed_time(e1) for e0, e1 in ev)
            ms = statistics.median(times)
            bound, frac = roofline_of(w, ms, peaks)
            out.append({"config": cfg, "workload": name,
                        "shape": f"B{w.B} Hq{w.Hq} Hkv{w.Hkv} S{w.S} P{w.P} d{w.d}",
                        "causal": {0: False, 1: True, 2: "balanced shards"}[int(w.causal)],
                        "ms": round(ms, 4), "ms_min_max": [round(times[0], 4), round(times[-1], 4)], "passes": reps,
                        "tflops": round(w.flops() / (ms / 1e3) / 1e12, 2),
                        "pct_bf16_peak": round(100 * w.flops() / (ms / 1e3) / 1e12 / peak, 2),
                        "roofline": {"bound": bound, "frac": round(frac, 4)},
                        "staging_GBps": round(2 * st["staging_bytes"] / (ms / 1e3) / 1e9, 1),
                        "n_s": [st["n_s_initial"], st["n_s_min"], st["n_s_max"], st["n_s_final"]]})
            del o, lse, ws
    tensors = None
    torch.cuda.empty_cache()
    return out


def cpu_baseline_cases(cores):
    """The fp64 oracle on each configuration: full runs of the small case and of the
    partition-stress grid (its result does not depend on P: once per d), and rows per second on
    the sampled rows of the large configurations with the full-configuration time extrapolated from
    the sample's algorithmic flops."""
    import numpy as np

    import oracle
    import ring_inputs as ri
    cases = []
    for name, full in (("small", True), ("sweep_d64_P2", True), ("sweep_d128_P2", True), ("h32_s32k_nc", False),
                       ("h32_s32k_c", False), ("gqa_s64k_c", False), ("long_s128k_c", False)):
        w = ri.WORKLOADS[name]
        q, k, v = ri.generate(w)
        rows = None if full else ri.sample_rows(w)
        t0 = time.perf_counter()
        oracle.for_workload(w, q, k, v, rows=rows, n_threads=cores)
        dt = time.perf_counter() - t0
        if full:
            cases.append({"workload": name if not name.startswith("sweep") else f"sweep_d{w.d} (every P)",
                          "rows": w.B * w.Hq * w.S, "seconds": round(dt, 3), "kind": "full run",
                          "tflops": round(w.flops() / dt / 1e12, 5)})
        else:
            fl = oracle_rows_flops(w, rows)
            cases.append({"workload": name, "rows": int(len(rows)), "seconds": round(dt, 3),
                          "rows_per_s": round(len(rows) / dt, 1), "tflops": round(fl / dt / 1e12, 5),
                          "full_seconds_extrapolated": round(w.flops() / (fl / dt), 1)})
        del q, k, v
    return {"cores": cores, "kind": "oracle", "cases": cases}


def run_configs(args):
    import torch

    import oracle
    import persistent_sm_ring_gb300 as psr
    psr.build()
    torch.cuda.set_device(0)
    peaks = load_peaks()
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    rows = time_configs(psr, torch, peaks)
    clk = clocks.stop()
    for r in rows:
        print(json.dumps(r), flush=True)
    cpu = None
    if not args.no_cpu_baseline:
        oracle.build()
        cpu = cpu_baseline_cases(oracle.default_threads())
    print(json.dumps({"configs": len(rows), "clocks": clk, "peak_source": peaks.get("source"),
                      "cpu_baseline_cases": cpu}), flush=True)


# ------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------

def run_ours(args):
    import numpy as np
    import torch

    import persistent_sm_ring_gb300 as psr
    import ring_inputs as ri

    rank, world, local = dist_init(args.gpus)
    psr.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    # profiling: the causal pass next to the causal pass over load-balanced shards
    names = ("h32_s32k_c", "h32_s32k_cb") if args.balanced else WORKLOADS
    wls = [ri.WORKLOADS[n] for n in names]
    if args.heads:  # a smaller same-kernel case (profiling): fewer heads, same S, P, d
        wls = [w.with_(Hq=args.heads, Hkv=args.heads) for w in wls]
    flops_step = sum(w.flops() for w in wls)
    peaks = load_peaks()

    # inputs: generated on the host (pinned) and copied once to HBM
    host = []
    devt = []
    for w in wls[:1]:  # both passes share Q,K,V (same seed and shape)
        q_h = torch.empty((w.B, w.Hq, w.S, w.d), dtype=torch.int16).pin_memory()
        k_h = torch.empty((w.B, w.Hkv, w.S, w.d), dtype=torch.int16).pin_memory()
        v_h = torch.empty((w.B, w.Hkv, w.S, w.d), dtype=torch.int16).pin_memory()
        ri.generate(w, q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr())
        host = [q_h, k_h, v_h]
        devt = [t.to(dev, non_blocking=False).view(torch.bfloat16) for t in host]
    w0 = wls[0]
    q, k, v = devt
    o = torch.empty_like(q)
    lse = torch.empty((w0.B, w0.Hq, w0.S), dtype=torch.float32, device=dev)
    shapes = [psr.make_shape(w.B, w.Hq, w.Hkv, w.S, w.P, w.d, w.causal, w.scale) for w in wls]
    ws_bytes = max(psr.workspace_bytes(s) for s in shapes)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    part = psr.make_partition(psr.ADAPTIVE)
    stream = torch.cuda.current_stream()

    def one_pass(w):
        psr.ring_attn_fwd(q, k, v, P=w.P, causal=w.causal, scale=w.scale, partition=part, workspace=ws, out=o,
                          lse=lse, stream=stream)

    def check_status():
        st = psr.get_stats(ws)
        if st["status"] != 0:
            raise RuntimeError(f"device status {st['status']} site {st['error_site']}")
        return st

    for _ in range(args.warmup):
        for w in wls:
            one_pass(w)
    check_status()

    # timed region: K steps, per-launch events on the launching stream
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in wls]
          for _ in range(args.steps)]
    stats = []
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    dist_barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        for i, w in enumerate(wls):
            ev[s][i][0].record(stream)
            one_pass(w)
            ev[s][i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    dist_barrier(world)
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    st_last = check_status()
    per_pass_ms = [[ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(args.steps)] for i in range(len(wls))]
    ms_step = dist_max(elapsed_ms / args.steps, world)
    total_flops = dist_sum(flops_step * args.steps, world)
    value = total_flops / (ms_step * args.steps / 1e3) / 1e12

    # dominant kernel: the persistent launch of each pass (same kernel); algorithmic flops / mean duration
    launch_ms = [statistics.mean(x) for x in per_pass_ms]
    kern_achieved = flops_step / (sum(launch_ms) / 1e3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    traffic = profiled_traffic()

    if args.device_only:
        if rank == 0:
            print(json.dumps({"device_only": True, "heads": wls[0].Hq, "ms_per_step": round(ms_step, 4),
                              "tflops": round(value, 2), "launch_ms": [round(x, 4) for x in launch_ms]}))
        return

    # per-pass statistics (non-causal, causal): one more instrumented pass each
    passes = []
    for i, w in enumerate(wls):
        one_pass(w)
        st = check_status()
        traj = psr.get_trajectory(ws, 64)
        passes.append({"workload": w.name, "causal": w.causal, "ms": round(launch_ms[i], 4),
                       "tflops": round(w.flops() / (launch_ms[i] / 1e3) / 1e12, 2),
                       "pct_peak": round(100 * w.flops() / (launch_ms[i] / 1e3) / 1e12 / peak, 2),
                       "staging_GBps": round(2 * st["staging_bytes"] / (launch_ms[i] / 1e3) / 1e9, 1),
                       "n_s": [st["n_s_initial"], st["n_s_min"], st["n_s_max"], st["n_s_final"]],
                       "role_switches": st["role_switches"], "traj_head": traj[:8]})

    # the causal pass over load-balanced shards (same tensors read in that shard order; the same
    # count of unmasked pairs): timed on its own, outside the headline step
    wb = ri.WORKLOADS["h32_s32k_cb"]
    if args.heads:
        wb = wb.with_(Hq=args.heads, Hkv=args.heads)
    for _ in range(2):
        one_pass(wb)
    evb = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e0, e1 in evb:
        e0.record(stream)
        one_pass(wb)
        e1.record(stream)
    torch.cuda.synchronize()
    st = check_status()
    ms_b = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evb)
    passes.append({"workload": wb.name, "causal": "balanced shards", "ms": round(ms_b, 4),
                   "tflops": round(wb.flops() / (ms_b / 1e3) / 1e12, 2),
                   "pct_peak": round(100 * wb.flops() / (ms_b / 1e3) / 1e12 / peak, 2),
                   "staging_GBps": round(2 * st["staging_bytes"] / (ms_b / 1e3) / 1e9, 1),
                   "n_s": [st["n_s_initial"], st["n_s_min"], st["n_s_max"], st["n_s_final"]],
                   "timed_in_step": False})

    # every configuration, each timed on its own (not part of the headline step)
    configs = None
    if not args.no_configs and not args.heads:
        configs = [{k2: r[k2] for k2 in ("config", "workload", "ms", "tflops", "pct_bf16_peak", "staging_GBps")}
                   | {"roofline_frac": r["roofline"]["frac"], "bound": r["roofline"]["bound"]}
                   for r in time_configs(psr, torch, peaks)]

    # e2e: host buffers through the C ABI (H2D + kernel + D2H, synchronised, per pass)
    o_h = torch.empty(host[0].shape, dtype=torch.int16).pin_memory()
    l_h = torch.empty(tuple(host[0].shape[:3]), dtype=torch.float32).pin_memory()
    dq, dk, dv = (torch.empty_like(t) for t in devt)
    h2d = sum(t.numel() * 2 for t in host) * len(wls)
    d2h = (o_h.numel() * 2 + l_h.numel() * 4) * len(wls)
    e2e_steps = max(10, args.steps)
    for w in wls:  # warm the host path once
        psr.ring_attn_fwd_host(*host, o_h, l_h, dq, dk, dv, o, lse, P=w.P, causal=w.causal, scale=w.scale,
                               partition=part, workspace=ws, stream=stream)
    # plain pinned-copy bandwidth of this machine, for reading the e2e figure (not part of the metric)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    dq.view(torch.int16).copy_(host[0], non_blocking=True)
    torch.cuda.synchronize()
    h2d_gbps = host[0].numel() * 2 / (time.perf_counter() - t0) / 1e9
    t0 = time.perf_counter()
    o_h.copy_(dq.view(torch.int16), non_blocking=True)
    torch.cuda.synchronize()
    d2h_gbps = o_h.numel() * 2 / (time.perf_counter() - t0) / 1e9
    dist_barrier(world)
    torch.cuda.synchronize()
    e2e_times = []
    t_all = time.perf_counter()
    for _ in range(e2e_steps):
        t0 = time.perf_counter()
        for w in wls:
            psr.ring_attn_fwd_host(*host, o_h, l_h, dq, dk, dv, o, lse, P=w.P, causal=w.causal, scale=w.scale,
                                   partition=part, workspace=ws, stream=stream)
        e2e_times.append(time.perf_counter() - t0)
    e2e_s = dist_max((time.perf_counter() - t_all) / e2e_steps, world)
    e2e_value = dist_sum(flops_step, world) / e2e_s / 1e12
    e2e_sorted = sorted(e2e_times)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import numpy as np  # noqa: F401
        qn = host[0].numpy().view(np.uint16)
        kn = host[1].numpy().view(np.uint16)
        vn = host[2].numpy().view(np.uint16)
        cpu = cpu_baseline(wls, [(qn, kn, vn)] * len(wls), budget_s=args.cpu_budget)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "B1 H32 S32768 P16 (L=2048) d128, one non-causal + one causal pass per step",
                       "B": 1, "H": 32, "S": 32768, "P": 16, "d": 128, "passes": list(WORKLOADS),
                       "partition": "adaptive", "l2": "inputs larger than L2 (Q,K,V 805 MB per pass)",
                       "parallelism": f"replicas x{world}"},
            "pct_of_bf16_peak": round(100 * value / peak, 2),
            "roofline": {"bound": "tensor", "achieved": round(kern_achieved, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(kern_achieved / peak, 4), "traffic": traffic,
                         "peak_source": f"{peaks.get('source')} bf16_tflops (burst)",
                         "frac_of_sustained": round(kern_achieved / peak_sus, 4)},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "ms_per_step_median": round(1e3 * statistics.median(e2e_times), 3),
                    "ms_per_step_min_max": [round(1e3 * e2e_sorted[0], 3), round(1e3 * e2e_sorted[-1], 3)],
                    "ms_per_step_all": [round(1e3 * t, 2) for t in e2e_times],
                    "pinned_copy_GBps": {"h2d": round(h2d_gbps, 1), "d2h": round(d2h_gbps, 1)}},
            "gpu_launches": args.steps * len(wls),
            "clocks": clk,
            "passes": passes,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ------------------------------------------------------------------------------------------------

def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np

    import oracle
    import ring_inputs as ri
    oracle.build()
    wls = [ri.WORKLOADS[n] for n in WORKLOADS]
    w = wls[0]
    q, k, v = ri.generate(w)
    cores = oracle.default_threads()
    rows_per_step = max(cores, args.ref_rows)
    rng = np.random.default_rng(1234)
    times, flops = [], []
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        f = 0.0
        for wl in wls:
            rows = np.sort(rng.choice(wl.B * wl.Hq * wl.S, size=rows_per_step, replace=False)).astype(np.int64)
            oracle.for_workload(wl, q, k, v, rows=rows, n_threads=cores)
            f += oracle_rows_flops(wl, rows)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
            flops.append(f)
    value = sum(flops) / sum(times) / 1e12
    sample = f"{rows_per_step} seeded query rows per pass of {'+'.join(x.name for x in wls)} per step (fp64)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "B1 H32 S32768 P16 (L=2048) d128, one non-causal + one causal pass per step",
                   "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------------------------------------
# partition-stress sweep (static staging-CTA counts vs the adaptive controller)
# ------------------------------------------------------------------------------------------------

def run_sweep(args):
    import torch

    import persistent_sm_ring_gb300 as psr
    import ring_inputs as ri
    psr.build()
    torch.cuda.set_device(0)
    ds = [args.sweep] if args.sweep in (64, 128) else [64, 128]
    statics = [2, 4, 6, 8, 12, 16, 24, 32, 48, 64, 76]  # 76 = N/2, the adaptive mode's default upper clamp
    rows = []
    for d in ds:
        base = ri.WORKLOADS[f"sweep_d{d}_P2"]
        q_h, k_h, v_h = ri.generate(base)
        import numpy as np
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
        q, k, v = dev(q_h), dev(k_h), dev(v_h)
        for P in (2, 4, 8, 16, 32, 64):
            w = ri.WORKLOADS[f"sweep_d{d}_P{P}"]
            ws = torch.empty(psr.workspace_bytes(psr.make_shape(w.B, w.Hq, w.Hkv, w.S, w.P, w.d, False)),
                             dtype=torch.uint8, device="cuda")
            o = torch.empty_like(q)
            lse = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32, device="cuda")

            def timed(part):
                for _ in range(2):
                    psr.ring_attn_fwd(q, k, v, P=P, causal=False, scale=w.scale, partition=part, workspace=ws,
                                      out=o, lse=lse)
                ts = []
                for _ in range(5):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    psr.ring_attn_fwd(q, k, v, P=P, causal=False, scale=w.scale, partition=part, workspace=ws,
                                      out=o, lse=lse)
                    b.record()
                    torch.cuda.synchronize()
                    ts.append(a.elapsed_time(b))
                st = psr.get_stats(ws)
                assert st["status"] == 0, st
                return statistics.median(ts), st

            res, cost = {}, {}
            for n in statics:
                try:
                    res[n], sst = timed(psr.make_partition(psr.STATIC, n_staging=n))
                    # measured unit costs (CTA-cycles per staging piece / per compute tile) at this split
                    cost[n] = (sst["staging_cycles"] / max(1, sst["staging_tasks"]),
                               sst["compute_cycles"] / max(1, sst["compute_tiles"]), sst["staging_tasks"],
                               sst["compute_tiles"])
                except psr.PsrError:
                    res[n] = None
            ad, st = timed(psr.make_partition(psr.ADAPTIVE))
            best_n = min((n for n in statics if res[n] is not None), key=lambda n: res[n])
            # the partition rule evaluated with the unit costs measured at the best static split
            c_s, c_p, r_s, r_p = cost[best_n]
            rule_n = psr.controller_target(psr.num_ctas(), r_s, c_s, r_p, c_p)
            rows.append({"d": d, "P": P, "adaptive_ms": round(ad, 4), "best_static_ms": round(res[best_n], 4),
                         "best_static_n": best_n, "ratio": round(ad / res[best_n], 4),
                         "worst_static_ms": round(max(v for v in res.values() if v is not None), 4),
                         "static_ms": {str(n): (round(v, 4) if v is not None else None) for n, v in res.items()},
                         "adaptive_n_s": [st["n_s_initial"], st["n_s_min"], st["n_s_max"], st["n_s_final"]],
                         "rule_n_at_best_costs": rule_n, "C_s": round(c_s, 1), "C_p": round(c_p, 1),
                         "adaptive_C_s": round(st["staging_cycles"] / max(1, st["staging_tasks"]), 1),
                         "adaptive_C_p": round(st["compute_cycles"] / max(1, st["compute_tiles"]), 1),
                         "tflops_adaptive": round(w.flops() / (ad / 1e3) / 1e12, 1)})
            print(json.dumps(rows[-1]), flush=True)
    import math
    geo = math.exp(sum(math.log(r["ratio"]) for r in rows) / len(rows))
    print(json.dumps({"sweep_geomean_adaptive_over_best_static": round(geo, 4),
                      "max_ratio": max(r["ratio"] for r in rows)}), flush=True)


# ------------------------------------------------------------------------------------------------
# AllGather + GEMM (the fused gather + contraction path; a separate line, not the headline)
# ------------------------------------------------------------------------------------------------

AG_METRIC = "allgather+gemm TFLOP/s (bf16, 1 GB300, P ranks emulated as shards)"


def ag_cpu_baseline(w, a, ww, budget_s):
    """The fp64 oracle on seeded sampled rows of the gathered A (every rank's columns)."""
    import numpy as np

    from oracle import ag_gemm as og
    rng = np.random.default_rng(w.seed + 99)
    n = 16
    while True:
        rows = np.sort(rng.choice(w.M, size=n, replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        og.for_workload(w, a, ww, rows=rows)
        dt = time.perf_counter() - t0
        if dt >= budget_s * 0.5 or n >= w.M // 4:
            break
        n = int(min(w.M // 4, max(2 * n, n * budget_s * 0.7 / max(dt, 1e-3))))
    flops = 2.0 * len(rows) * w.K * w.Ns * w.P
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{len(rows)} seeded rows of the gathered A x all {w.P} ranks' W (fp64 numpy), {dt:.1f} s"}


def run_ag(args):
    import numpy as np
    import torch

    import persistent_sm_ring_gb300 as psr
    import ring_inputs as ri
    psr.build()
    torch.cuda.set_device(0)
    w = ri.AG_WORKLOADS["ag_m8k_k8k_n28k_p8"]
    a_h, w_h = ri.generate_ag_gemm(w)
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory()
    a_p, w_p = pin(a_h), pin(w_h)
    a = a_p.cuda().view(torch.bfloat16)
    ww = w_p.cuda().view(torch.bfloat16)
    c, ws = psr.ag_gemm(a, ww, P=w.P)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))

    def timed(fn, reps):
        for _ in range(max(3, args.warmup)):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for e0, e1 in ev:
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return [e0.elapsed_time(e1) for e0, e1 in ev]

    def ours(part):
        return lambda: psr.ag_gemm(a, ww, P=w.P, partition=part, workspace=ws, out=c, stream=stream)

    adaptive = psr.make_partition(psr.ADAPTIVE)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    ts = timed(ours(adaptive), args.steps)
    clk = clocks.stop()
    st = psr.get_stats(ws)
    if st["status"] != 0:
        raise RuntimeError(f"device status {st['status']} site {st['error_site']}")
    ms = statistics.mean(ts)
    value = w.flops() / (ms / 1e3) / 1e12
    if args.device_only:  # profiling: the timed launches only
        print(json.dumps({"device_only": True, "ms_per_step": round(ms, 4), "tflops": round(value, 2)}), flush=True)
        return

    statics = {}
    for n in (4, 8, 12, 16, 24):
        t = statistics.median(timed(ours(psr.make_partition(psr.STATIC, n_staging=n)), 5))
        statics[str(n)] = round(w.flops() / (t / 1e3) / 1e12, 1)
    # context: cuBLAS on the same P products with A already gathered (no copy at all)
    wt = ww.view(w.P, w.Ns, w.K).transpose(1, 2)
    t_lib = statistics.median(timed(lambda: torch.matmul(a, wt), 5))

    # e2e: pinned host A, W in; C out; through the public binding
    c_h = torch.empty((w.P, w.M, w.Ns), dtype=torch.int16).pin_memory()
    e2e_steps = 10

    def e2e_step():
        a.view(torch.int16).copy_(a_p, non_blocking=True)
        ww.view(torch.int16).copy_(w_p, non_blocking=True)
        psr.ag_gemm(a, ww, P=w.P, partition=adaptive, workspace=ws, out=c, stream=stream)
        c_h.copy_(c.view(torch.int16), non_blocking=True)
        torch.cuda.synchronize()

    e2e_step()
    e2e_times = []
    for _ in range(e2e_steps):
        t0 = time.perf_counter()
        e2e_step()
        e2e_times.append(time.perf_counter() - t0)
    e2e_s = statistics.mean(e2e_times)

    cpu = None if args.no_cpu_baseline else ag_cpu_baseline(w, a_h, w_h, args.cpu_budget)
    print(json.dumps({
        "metric": AG_METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"AllGather+GEMM M{w.M} K{w.K} N{w.Ns * w.P} over P{w.P} (C_r = gather(A) @ W_r^T)",
                   "M": w.M, "K": w.K, "Ns": w.Ns, "P": w.P, "partition": "adaptive",
                   "l2": f"inputs larger than L2 (A {w.n_a * 2 / 1e6:.0f} MB, W {w.n_w * 2 / 1e6:.0f} MB)"},
        "roofline": {"bound": "tensor", "achieved": round(value, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(value / peak, 4), "traffic": None,
                     "peak_source": f"{peaks.get('source')} bf16_tflops (burst)"},
        "static_tflops": statics, "best_static_tflops": max(statics.values()),
        "adaptive_over_best_static_time": round(max(statics.values()) / value, 4),
        "n_s": [st["n_s_initial"], st["n_s_min"], st["n_s_max"], st["n_s_final"]],
        "gather_GBps": round(w.gather_bytes() / (ms / 1e3) / 1e9, 1),
        "cublas_no_gather_tflops": round(w.flops() / (t_lib / 1e3) / 1e12, 1),
        "cpu_baseline": cpu,
        "e2e": {"value": round(w.flops() / e2e_s / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": (w.n_a + w.n_w) * 2, "d2h_bytes_per_step": c_h.numel() * 2, "steps": e2e_steps,
                "per_step_ms_median_min_max": [round(1e3 * statistics.median(e2e_times), 3), round(1e3 * min(e2e_times), 3),
                                               round(1e3 * max(e2e_times), 3)]},
        "gpu_launches": args.steps,
        "clocks": clk,
    }), flush=True)


# ------------------------------------------------------------------------------------------------
# GEMM + ReduceScatter (compute feeds the reduce-scatter; a separate line, not the headline)
# ------------------------------------------------------------------------------------------------

RS_METRIC = "gemm+reducescatter TFLOP/s (bf16, 1 GB300, P ranks emulated as shards)"


def rs_cpu_baseline(w, a, ww, budget_s):
    """The fp64 oracle on seeded sampled output rows (every rank's partial of each row)."""
    import numpy as np

    from oracle import gemm_rs as og
    rng = np.random.default_rng(w.seed + 99)
    n = 16
    while True:
        rows = np.sort(rng.choice(w.M, size=n, replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        og.for_workload(w, a, ww, rows=rows)
        dt = time.perf_counter() - t0
        if dt >= budget_s * 0.5 or n >= w.M // 4:
            break
        n = int(min(w.M // 4, max(2 * n, n * budget_s * 0.7 / max(dt, 1e-3))))
    flops = 2.0 * len(rows) * w.N * w.Ks * w.P
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{len(rows)} seeded output rows, all {w.P} ranks' partials (fp64 numpy), {dt:.1f} s"}


def run_rs(args):
    import numpy as np
    import torch

    import persistent_sm_ring_gb300 as psr
    import ring_inputs as ri
    psr.build()
    torch.cuda.set_device(0)
    w = ri.RS_WORKLOADS["rs_m8k_n8k_k28k_p8"]
    a_h, w_h = ri.generate_gemm_rs(w)
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory()
    a_p, w_p = pin(a_h), pin(w_h)
    a = a_p.cuda().view(torch.bfloat16)
    ww = w_p.cuda().view(torch.bfloat16)
    out, ws = psr.gemm_rs(a, ww)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))

    def timed(fn, reps):
        for _ in range(max(3, args.warmup)):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for e0, e1 in ev:
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return [e0.elapsed_time(e1) for e0, e1 in ev]

    def ours(part):
        return lambda: psr.gemm_rs(a, ww, partition=part, workspace=ws, out=out, stream=stream)

    adaptive = psr.make_partition(psr.ADAPTIVE)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    ts = timed(ours(adaptive), args.steps)
    clk = clocks.stop()
    st = psr.get_stats(ws)
    if st["status"] != 0:
        raise RuntimeError(f"device status {st['status']} site {st['error_site']}")
    ms = statistics.mean(ts)
    value = w.flops() / (ms / 1e3) / 1e12
    if args.device_only:  # profiling: the timed launches only
        print(json.dumps({"device_only": True, "ms_per_step": round(ms, 4), "tflops": round(value, 2)}), flush=True)
        return

    statics = {}
    for n in (4, 8, 12, 16, 24):
        t = statistics.median(timed(ours(psr.make_partition(psr.STATIC, n_staging=n)), 5))
        statics[str(n)] = round(w.flops() / (t / 1e3) / 1e12, 1)
    # context: cuBLAS on the same P partial products, then the reduction by torch (no overlap)
    wt = ww.transpose(1, 2)
    t_lib = statistics.median(timed(lambda: torch.bmm(a, wt).float().sum(0), 5))

    # e2e: pinned host A, W in; the reduced output out; through the public binding
    o_h = torch.empty((w.M, w.N), dtype=torch.int16).pin_memory()
    e2e_steps = 10

    def e2e_step():
        a.view(torch.int16).copy_(a_p, non_blocking=True)
        ww.view(torch.int16).copy_(w_p, non_blocking=True)
        psr.gemm_rs(a, ww, partition=adaptive, workspace=ws, out=out, stream=stream)
        o_h.copy_(out.view(torch.int16), non_blocking=True)
        torch.cuda.synchronize()

    e2e_step()
    e2e_times = []
    for _ in range(e2e_steps):
        t0 = time.perf_counter()
        e2e_step()
        e2e_times.append(time.perf_counter() - t0)
    e2e_s = statistics.mean(e2e_times)

    cpu = None if args.no_cpu_baseline else rs_cpu_baseline(w, a_h, w_h, args.cpu_budget)
    print(json.dumps({
        "metric": RS_METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"GEMM+ReduceScatter M{w.M} N{w.N} K{w.Ks * w.P} over P{w.P} "
                               f"(out = sum_r A_r @ W_r^T, row block q to rank q)",
                   "M": w.M, "N": w.N, "Ks": w.Ks, "P": w.P, "partition": "adaptive",
                   "l2": f"inputs larger than L2 (A {w.n_a * 2 / 1e6:.0f} MB, W {w.n_w * 2 / 1e6:.0f} MB)"},
        "roofline": {"bound": "tensor", "achieved": round(value, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(value / peak, 4), "traffic": None,
                     "peak_source": f"{peaks.get('source')} bf16_tflops (burst)"},
        "static_tflops": statics, "best_static_tflops": max(statics.values()),
        "adaptive_over_best_static_time": round(max(statics.values()) / value, 4),
        "n_s": [st["n_s_initial"], st["n_s_min"], st["n_s_max"], st["n_s_final"]],
        "reduce_GBps": round(st["staging_bytes"] / (ms / 1e3) / 1e9, 1),
        "cublas_bmm_then_sum_tflops": round(w.flops() / (t_lib / 1e3) / 1e12, 1),
        "cpu_baseline": cpu,
        "e2e": {"value": round(w.flops() / e2e_s / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": (w.n_a + w.n_w) * 2, "d2h_bytes_per_step": o_h.numel() * 2, "steps": e2e_steps,
                "per_step_ms_median_min_max": [round(1e3 * statistics.median(e2e_times), 3), round(1e3 * min(e2e_times), 3),
                                               round(1e3 * max(e2e_times), 3)]},
        "gpu_launches": args.steps,
        "clocks": clk,
    }), flush=True)


# ------------------------------------------------------------------------------------------------
# Ring Attention backward (a separate line, not the headline)
# ------------------------------------------------------------------------------------------------

BWD_METRIC = "ring-attn bwd TFLOP/s (bf16, 1 GB300; 10*d flops per unmasked (query, key) pair)"


def bwd_flops(w):
    pairs = w.S * (w.S + 1) // 2 if w.causal else w.S * w.S
    return 10.0 * w.d * pairs * w.B * w.Hq


def bwd_cpu_baseline(w, q, k, v, do, budget_s):
    """The fp64 oracle's dQ rows (each with its own forward row) on a seeded sample of query rows."""
    import numpy as np

    from oracle import attn_bwd as ob
    rng = np.random.default_rng(w.seed + 99)
    n = 8
    while True:
        rows = np.sort(rng.choice(w.B * w.Hq * w.S, size=n, replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        ob.attn_bwd_dq_rows(q, k, v, do, causal=bool(w.causal), scale=w.scale, bh_rows=rows)
        dt = time.perf_counter() - t0
        if dt >= budget_s * 0.5 or n >= 4096:
            break
        n = int(min(4096, max(2 * n, n * budget_s * 0.7 / max(dt, 1e-3))))
    keys = (rows % w.S) + 1 if w.causal else np.full(len(rows), w.S)
    flops = float(10.0 * w.d * keys.sum())
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{len(rows)} seeded query rows of {w.name}: dQ rows with their own forward rows "
                      f"(fp64 numpy, every allowed key), {dt:.1f} s"}


def run_bwd(args):
    import numpy as np
    import torch

    import persistent_sm_ring_gb300 as psr
    import ring_inputs as ri
    psr.build()
    torch.cuda.set_device(0)
    peaks = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    base = ri.WORKLOADS["h32_s32k_c"]
    if args.heads:  # a smaller same-kernel case (profiling): fewer heads, same S, P, d
        base = base.with_(Hq=args.heads, Hkv=args.heads)
    q_h, k_h, v_h = ri.generate(base)
    do_h = ri.generate_dout(base)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.bfloat16)
    q, k, v, do = dev(q_h), dev(k_h), dev(v_h), dev(do_h)
    stream = torch.cuda.current_stream()
    passes = []
    clk = None
    for name in ("h32_s32k_c", "h32_s32k_nc", "h32_s32k_cb"):
        w = ri.WORKLOADS[name].with_(Hq=base.Hq, Hkv=base.Hkv)
        o, lse, _ = psr.ring_attn_fwd(q, k, v, P=w.P, causal=w.causal, scale=w.scale)
        dq, dk, dv, ws = psr.ring_attn_bwd(q, k, v, o, lse, do, P=w.P, causal=w.causal, scale=w.scale)

        def step():
            psr.ring_attn_bwd(q, k, v, o, lse, do, P=w.P, causal=w.causal, scale=w.scale, workspace=ws, dq=dq,
                              dk=dk, dv=dv, stream=stream)
        for _ in range(max(3, args.warmup)):
            step()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        clocks = ClockSampler(0)
        clocks.start()
        time.sleep(0.3)
        torch.cuda.synchronize()
        for e0, e1 in ev:
            e0.record(stream)
            step()
            e1.record(stream)
        torch.cuda.synchronize()
        c = clocks.stop()
        clk = clk or c
        st = psr.get_stats(ws)
        if st["status"] != 0:
            raise RuntimeError(f"device status {st['status']} site {st['error_site']}")
        ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
        passes.append({"workload": name, "causal": {0: False, 1: True, 2: "balanced shards"}[int(w.causal)],
                       "ms": round(ms, 4),
                       "tflops": round(bwd_flops(w) / (ms / 1e3) / 1e12, 2),
                       "pct_peak": round(100 * bwd_flops(w) / (ms / 1e3) / 1e12 / peak, 2), "clocks": c})
    w = ri.WORKLOADS["h32_s32k_c"].with_(Hq=base.Hq, Hkv=base.Hkv)
    ms = passes[0]["ms"]
    value = bwd_flops(w) / (ms / 1e3) / 1e12

    # e2e: pinned host Q, K, V, O, LSE, dO in and dQ, dK, dV out around the public call
    o, lse, _ = psr.ring_attn_fwd(q, k, v, P=w.P, causal=True, scale=w.scale)
    host_in = [t.cpu().pin_memory() for t in (q, k, v, o, lse, do)]
    dev_in = [torch.empty_like(t) for t in (q, k, v, o, lse, do)]
    dq, dk, dv, ws = psr.ring_attn_bwd(q, k, v, o, lse, do, P=w.P, causal=True, scale=w.scale)
    host_out = [torch.empty_like(t, device="cpu").pin_memory() for t in (dq, dk, dv)]

    def e2e_step():
        for h, d in zip(host_in, dev_in):
            d.copy_(h, non_blocking=True)
        psr.ring_attn_bwd(*dev_in, P=w.P, causal=True, scale=w.scale, workspace=ws, dq=dq, dk=dk, dv=dv,
                          stream=stream)
        for h, d in zip(host_out, (dq, dk, dv)):
            h.copy_(d, non_blocking=True)
        torch.cuda.synchronize()

    e2e_step()
    e2e_times = []
    for _ in range(10):
        t0 = time.perf_counter()
        e2e_step()
        e2e_times.append(time.perf_counter() - t0)
    e2e_s = statistics.mean(e2e_times)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    cpu = None if args.no_cpu_baseline else bwd_cpu_baseline(w, q_h, k_h, v_h, do_h, args.cpu_budget)
    print(json.dumps({
        "metric": BWD_METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "Ring Attention backward B1 H32 S32768 P16 (L=2048) d128, causal "
                               "(dQ, dK, dV from Q, K, V, O, LSE, dO)",
                   "l2": "inputs larger than L2 (Q, K, V, O, dO 1.34 GB)"},
        "roofline": {"bound": "tensor", "achieved": round(value, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(value / peak, 4), "traffic": None,
                     "peak_source": f"{peaks.get('source')} bf16_tflops (burst)"},
        "cpu_baseline": cpu,
        "e2e": {"value": round(bwd_flops(w) / e2e_s / 1e12, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": len(e2e_times),
                "per_step_ms_median_min_max": [round(1e3 * statistics.median(e2e_times), 3),
                                               round(1e3 * min(e2e_times), 3), round(1e3 * max(e2e_times), 3)]},
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
        "passes": passes,
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep", type=int, nargs="?", const=0, default=None)
    ap.add_argument("--ag-gemm", action="store_true", help="the AllGather+GEMM path instead of attention")
    ap.add_argument("--gemm-rs", action="store_true", help="the GEMM+ReduceScatter path instead of attention")
    ap.add_argument("--bwd", action="store_true", help="the Ring Attention backward instead of the forward")
    ap.add_argument("--configs", action="store_true",
                    help="time all five configurations and run the oracle's CPU-baseline cases")
    ap.add_argument("--no-configs", action="store_true", help="leave the per-configuration table out of the line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=96)
    ap.add_argument("--heads", type=int, default=0, help="profiling: run the same kernel with fewer heads")
    ap.add_argument("--device-only", action="store_true", help="profiling: timed device passes only")
    ap.add_argument("--balanced", action="store_true",
                    help="profiling (with --device-only): the causal pass and the causal pass over load-balanced shards")
    args = ap.parse_args()
    if args.balanced and not args.device_only:
        ap.error("--balanced is a profiling mode: use it with --device-only")
    if args.sweep is not None:
        run_sweep(args)
    elif args.ag_gemm:
        run_ag(args)
    elif args.gemm_rs:
        run_rs(args)
    elif args.bwd:
        run_bwd(args)
    elif args.configs:
        run_configs(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
