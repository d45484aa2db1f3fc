"""CPU tests of bench.py's host logic: rank plumbing over gloo (world size 2) and the
reference arm's JSON line (the fp64 oracle on a small row sample)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.dist_barrier(world)
    mx = bench.dist_max(10.0 * (rank + 1), world)    # per-rank times: max over ranks is the job time
    sm = bench.dist_sum(1000.0 * (rank + 1), world)  # per-rank work: the job value is the sum
    bench.dist_barrier(world)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"max": mx, "sum": sm}, f)
    dist.destroy_process_group()


def test_rank_reductions_gloo_world_size_2(tmp_path):
    import torch.multiprocessing as mp
    port = 29500 + (os.getpid() % 2000)
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    for r in range(2):
        d = json.load(open(tmp_path / f"r{r}.json"))
        assert d == {"max": 20.0, "sum": 3000.0}


def test_reference_arm_json_line():
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    env.pop("RANK", None)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0", "--ref-rows", "8"], capture_output=True, text=True, timeout=600, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["metric"].startswith("ring-attn fwd TFLOP/s")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], capture_output=True, text=True, timeout=120, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_config_roofline_arithmetic():
    # the per-configuration roofline: flops and bytes worked out by hand for the headline shape
    sys.path.insert(0, ROOT)
    import bench
    import ring_inputs as ri
    w = ri.WORKLOADS["h32_s32k_nc"]
    assert w.flops() == 4 * 128 * 32768 * 32768 * 32  # 1.759e13
    # Q, K, V read, O written (32 heads x 32768 rows x 128 x 2 B each), LSE 32 x 32768 x 4 B, and the
    # 240 ring transfers of a 2048-row chunk of K and V (1 MiB per head) read and written
    tensor = 32 * 32768 * 128 * 2
    staged = 16 * 15 * 32 * (2 * 2048 * 128 * 2)
    assert bench.algorithmic_bytes(w) == 4 * tensor + 32 * 32768 * 4 + 2 * staged
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0}
    bound, frac = bench.roofline_of(w, 1e3 * w.flops() / 1e15, peaks)  # a pass at 1000 TFLOP/s
    assert bound == "tensor" and abs(frac - 0.5) < 1e-12
    # the large-P sweep point moves more bytes than its flops take at these peaks: HBM-bound
    w64 = ri.WORKLOADS["sweep_d64_P64"]
    bound, frac = bench.roofline_of(w64, 1.0, peaks)
    assert bound == "hbm"
    assert abs(frac - bench.algorithmic_bytes(w64) / 8e12 / 1e-3) < 1e-9
    # every configuration is covered, each workload once
    names = [n for _, ns in bench.CONFIGS for n in ns]
    assert len(names) == len(set(names)) == 1 + 2 + 1 + 1 + 12
    assert all(n in ri.WORKLOADS for n in names)
