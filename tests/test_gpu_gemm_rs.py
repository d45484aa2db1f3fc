"""GPU parity of the GEMM + ReduceScatter path (psr_gemm_rs through the C ABI) against the
fp64 oracle (oracle/gemm_rs.py).

Bound: each rank's partial is an fp32 tensor-core accumulation over Ks, the P partials are
summed in fp32 in rank order and the sum is rounded to bf16 (8 significant bits, round to
nearest even: relative error <= 2^-8, the first term of the bound; the fp32 accumulation errors,
a random walk of ~sqrt(K) roundings of 2^-24, stay far below the second); every compared element
must satisfy |out - ref| <= 2^-8 |ref| + 2^-12 rms(ref), and ||out - ref||_2 / ||ref||_2 <= 3e-3.
"""
import numpy as np
import pytest

import ring_inputs as ri
from oracle import gemm_rs as og

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _dev(torch, arr):
    return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).cuda().view(torch.bfloat16)


def _check(out, ref, what):
    assert np.all(np.isfinite(out)), what
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(out - ref)
    bound = 2.0**-8 * np.abs(ref) + 2.0**-12 * rms
    worst = float(np.max(err - bound))
    assert worst <= 0.0, f"{what}: max excess over the bound {worst:.3e}"
    rel = float(np.linalg.norm(out - ref) / np.linalg.norm(ref))
    assert rel <= 3e-3, f"{what}: rel L2 {rel:.3e}"


def _run(psr, a, ww, partition=None):
    torch = _torch()
    out, ws = psr.gemm_rs(_dev(torch, a), _dev(torch, ww), partition=partition)
    st = psr.get_stats(ws)
    return out.float().cpu().numpy().astype(np.float64), st


BASE = ri.RS_WORKLOADS["rs_small"]                                   # M1024 N512 Ks256 P4
SMALL = [
    BASE,
    BASE.with_(name="rs_p1", M=512, N=768, Ks=192, P=1, seed=802),     # no reduction partner
    BASE.with_(name="rs_p8", M=2048, N=512, Ks=128, P=8, seed=803),
    BASE.with_(name="rs_p2_k64", M=512, N=1280, Ks=64, P=2, seed=804),  # one K step per tile
    BASE.with_(name="rs_p3", M=768, N=256, Ks=320, P=3, seed=805),      # P not a power of two
    BASE.with_(name="rs_two_windows", M=8192, N=512, Ks=64, P=2, seed=806),  # 32 row blocks: two task windows
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_gemm_rs_every_element(psr, w):
    a, ww = ri.generate_gemm_rs(w)
    ref = og.for_workload(w, a, ww)
    out, st = _run(psr, a, ww)
    assert st["status"] == 0, st
    _check(out, ref, w.name)
    n_out = (w.M // 256) * ((w.N + 511) // 512)  # 256 x 512 output tiles (the last one half wide when N % 512 = 256)
    assert st["compute_items"] == w.P * n_out
    assert st["staging_tasks"] == n_out
    assert st["staging_bytes"] == w.reduce_bytes()


@pytest.mark.parametrize("n_s", [1, 3, 40])
def test_gemm_rs_static_partitions(psr, n_s):
    w = SMALL[2]
    a, ww = ri.generate_gemm_rs(w)
    ref = og.for_workload(w, a, ww)
    out, st = _run(psr, a, ww, partition=psr.make_partition(psr.STATIC, n_staging=n_s))
    assert st["status"] == 0 and st["n_s_final"] == n_s, st
    _check(out, ref, f"static n_s={n_s}")


def test_gemm_rs_adaptive_with_initial_reducers(psr):
    w = SMALL[0]
    a, ww = ri.generate_gemm_rs(w)
    ref = og.for_workload(w, a, ww)
    out, st = _run(psr, a, ww, partition=psr.make_partition(psr.ADAPTIVE, n_staging=8))
    assert st["status"] == 0 and st["n_s_initial"] == 8, st
    _check(out, ref, "adaptive from 8 reducers")


def test_gemm_rs_full_size_sampled_rows(psr):
    w = ri.RS_WORKLOADS["rs_m8k_n8k_k28k_p8"]
    a, ww = ri.generate_gemm_rs(w)
    rows = ri.rs_sample_rows(w, n_random=512)
    ref = og.for_workload(w, a, ww, rows=rows)
    out, st = _run(psr, a, ww)
    assert st["status"] == 0, st
    _check(out[rows], ref, w.name)
    assert st["staging_bytes"] == w.reduce_bytes()


def test_gemm_rs_result_is_deterministic(psr):
    # the partials are summed in rank order whatever the completion order
    w = SMALL[2]
    a, ww = ri.generate_gemm_rs(w)
    o1, _ = _run(psr, a, ww)
    o2, _ = _run(psr, a, ww, partition=psr.make_partition(psr.STATIC, n_staging=5))
    assert np.array_equal(o1, o2)


def test_gemm_rs_dropped_arrival_times_out_and_context_survives(psr):
    w = SMALL[0]
    a, ww = ri.generate_gemm_rs(w)
    part = psr.make_partition(psr.ADAPTIVE, fault=psr.FAULT_DROP_FIRST_FLAG, timeout_ms=200)
    _, st = _run(psr, a, ww, partition=part)
    # one epilogue warp's arrival is dropped: that tile is never enqueued and the CTA holding
    # its ticket gives up on the queue entry (1)
    assert st["status"] == psr.ERR_TIMEOUT and st["error_site"] == 1, st
    ref = og.for_workload(w, a, ww)
    out, st2 = _run(psr, a, ww)
    assert st2["status"] == 0
    _check(out, ref, "after timeout")
