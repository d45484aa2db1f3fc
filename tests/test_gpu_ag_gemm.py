"""GPU parity of the AllGather + GEMM path (psr_ag_gemm through the C ABI) against the fp64
oracle (oracle/ag_gemm.py).

Bound: the result is the fp32-accumulated product rounded to bf16 (8 significant bits, round to
nearest even: relative error <= 2^-8, the first term of the bound; the fp32 accumulation errors, a
random walk of ~sqrt(K) roundings of 2^-24, stay far below the second); every compared element
must satisfy |C - C_ref| <= 2^-8 |C_ref| + 2^-12 rms(C_ref), and ||C - C_ref||_2 / ||C_ref||_2 <= 3e-3.
"""
import numpy as np
import pytest

import ring_inputs as ri
from oracle import ag_gemm as og

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _dev(torch, arr):
    return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).cuda().view(torch.bfloat16)


def _check(c, ref, what):
    assert np.all(np.isfinite(c)), what
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(c - ref)
    bound = 2.0**-8 * np.abs(ref) + 2.0**-12 * rms
    worst = float(np.max(err - bound))
    assert worst <= 0.0, f"{what}: max excess over the bound {worst:.3e}"
    rel = float(np.linalg.norm(c - ref) / np.linalg.norm(ref))
    assert rel <= 3e-3, f"{what}: rel L2 {rel:.3e}"


def _run(psr, w, a, ww, partition=None):
    torch = _torch()
    c, ws = psr.ag_gemm(_dev(torch, a), _dev(torch, ww), P=w.P, partition=partition)
    st = psr.get_stats(ws)
    return c.float().cpu().numpy().astype(np.float64), st


SMALL = [
    ri.AG_WORKLOADS["ag_small"],                                              # M1024 K512 Ns256 P4
    ri.AG_WORKLOADS["ag_small"].with_(name="ag_medium", M=2048, K=1024, Ns=512, P=4, seed=702),
    ri.AG_WORKLOADS["ag_small"].with_(name="ag_p1", M=512, K=256, Ns=256, P=1, seed=703),
    ri.AG_WORKLOADS["ag_small"].with_(name="ag_p8", M=2048, K=384, Ns=256, P=8, seed=704),
    # a full-width 256 x 512 tile and a half-wide last tile in every rank
    ri.AG_WORKLOADS["ag_small"].with_(name="ag_ns768", M=1024, K=384, Ns=768, P=2, seed=705),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_ag_gemm_every_element(psr, w):
    a, ww = ri.generate_ag_gemm(w)
    ref = og.for_workload(w, a, ww)
    c, st = _run(psr, w, a, ww)
    assert st["status"] == 0, st
    _check(c, ref, w.name)
    # one task per 256 x 512 output tile (a rank's last tile half wide when Ns % 512 = 256)
    assert st["compute_items"] == w.P * w.P * (w.Ms // 256) * ((w.Ns + 511) // 512)
    assert st["staging_bytes"] == w.gather_bytes()


@pytest.mark.parametrize("n_s", [1, 3, 40])
def test_ag_gemm_static_partitions(psr, n_s):
    w = SMALL[1]
    a, ww = ri.generate_ag_gemm(w)
    ref = og.for_workload(w, a, ww)
    c, st = _run(psr, w, a, ww, partition=psr.make_partition(psr.STATIC, n_staging=n_s))
    assert st["status"] == 0 and st["n_s_final"] == n_s, st
    _check(c, ref, f"static n_s={n_s}")


def test_ag_gemm_full_size_sampled_rows(psr):
    w = ri.AG_WORKLOADS["ag_m8k_k8k_n28k_p8"]
    a, ww = ri.generate_ag_gemm(w)
    rows = ri.ag_sample_rows(w, n_random=512)
    ref = og.for_workload(w, a, ww, rows=rows)
    c, st = _run(psr, w, a, ww)
    assert st["status"] == 0, st
    _check(c[:, rows], ref, w.name)


def test_ag_gemm_dropped_flag_times_out_and_context_survives(psr):
    w = SMALL[1]
    a, ww = ri.generate_ag_gemm(w)
    part = psr.make_partition(psr.ADAPTIVE, fault=psr.FAULT_DROP_FIRST_FLAG, timeout_ms=200)
    _, st = _run(psr, w, a, ww, partition=part)
    # the first wait to give up is the producer's on the flag (1) or the MMA issuer's on the
    # tile that producer never loads (2), whichever started first; or an idle stager (11)
    assert st["status"] == psr.ERR_TIMEOUT and st["error_site"] in (1, 2, 11), st
    ref = og.for_workload(w, a, ww)
    c, st2 = _run(psr, w, a, ww)
    assert st2["status"] == 0
    _check(c, ref, "after timeout")
