"""GPU parity of causal Ring Attention over load-balanced shards (causal = 2: shard r holds
half-chunks r and 2P-1-r of the sequence) against the fp64 oracle, through the C ABI.

Same tolerances as the other attention parity tests: max |dO| <= 2e-2,
||dO||_2 / ||O_ref||_2 <= 5e-3, max |dLSE| <= 1e-3.
"""
import numpy as np
import pytest

import oracle
import ring_inputs as ri

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2, LSE_ABS = 2e-2, 5e-3, 1e-3


def _torch():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def to_dev(torch, arr):
    return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).cuda().view(torch.bfloat16)


def gpu_run(psr, w, q, k, v, partition=None):
    torch = _torch()
    o, lse, ws = psr.ring_attn_fwd(to_dev(torch, q), to_dev(torch, k), to_dev(torch, v), P=w.P, causal=w.causal,
                                   scale=w.scale, partition=partition)
    st = psr.get_stats(ws)
    assert st["status"] == 0, st
    return (o.view(-1, w.d).float().cpu().numpy().astype(np.float64), lse.view(-1).cpu().numpy().astype(np.float64),
            st)


def check(o, lse, o_ref, lse_ref, what):
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    max_abs = float(np.abs(o - o_ref).max())
    rel = float(np.linalg.norm(o - o_ref) / np.linalg.norm(o_ref))
    lse_err = float(np.abs(lse - lse_ref).max())
    assert max_abs <= MAX_ABS, f"{what}: max |dO| = {max_abs:.3e}"
    assert rel <= REL_L2, f"{what}: rel L2 = {rel:.3e}"
    assert lse_err <= LSE_ABS, f"{what}: max |dLSE| = {lse_err:.3e}"


def balanced_order(S, P):
    """Natural position held by each stored row: shard r holds half-chunks r and 2P-1-r."""
    h = S // P // 2
    return np.concatenate([np.arange(c * h, (c + 1) * h) for r in range(P) for c in (r, 2 * P - 1 - r)])


BASE = ri.WORKLOADS["small"]
SMALL = [
    BASE.with_(name="cb_p4_d64", S=2048, P=4, causal=2, seed=61),
    BASE.with_(name="cb_p4_d128", S=4096, P=4, d=128, causal=2, seed=62),
    BASE.with_(name="cb_gqa_p3", B=2, Hq=6, Hkv=2, S=3072, P=3, d=128, causal=2, seed=63, qmul=2.0, kmul=2.0),
    BASE.with_(name="cb_p1", S=512, P=1, causal=2, seed=64),
    BASE.with_(name="cb_p8_d128", S=4096, P=8, d=128, causal=2, seed=65),
    BASE.with_(name="cb_p16_d64", Hq=1, Hkv=1, S=8192, P=16, causal=2, seed=66),
    ri.WORKLOADS["long_s128k_c"].with_(name="cb_outlier", S=8192, P=8, Hq=2, Hkv=2, causal=2, seed=67),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_balanced_all_rows(psr, w):
    q, k, v = ri.generate(w)
    o_ref, lse_ref = oracle.for_workload(w, q, k, v)
    o, lse, st = gpu_run(psr, w, q, k, v)
    check(o, lse, o_ref, lse_ref, w.name)
    assert st["staging_bytes"] == w.staging_bytes()
    assert st["compute_items"] == w.B * w.Hq * w.S // 256


@pytest.mark.parametrize("n_s", [1, 3, 16])
def test_balanced_static_partitions(psr, n_s):
    w = SMALL[4]
    q, k, v = ri.generate(w)
    o_ref, lse_ref = oracle.for_workload(w, q, k, v)
    o, lse, st = gpu_run(psr, w, q, k, v, partition=psr.make_partition(psr.STATIC, n_staging=n_s))
    check(o, lse, o_ref, lse_ref, f"static n_s={n_s}")
    assert st["n_s_final"] == n_s


def test_balanced_equals_contiguous_on_reordered_sequence(psr):
    # the same sequence, stored contiguously (causal = 1) and in balanced shard order
    # (causal = 2), gives the same rows up to the order of the chunk merges
    wc = BASE.with_(name="reorder_c", Hq=4, Hkv=2, S=8192, P=8, d=128, causal=1, seed=68)
    wb = wc.with_(name="reorder_cb", causal=2)
    q, k, v = ri.generate(wc)
    pos = balanced_order(wc.S, wc.P)
    oc, lc, _ = gpu_run(psr, wc, q, k, v)
    ob, lb, _ = gpu_run(psr, wb, q[:, :, pos], k[:, :, pos], v[:, :, pos])
    oc = oc.reshape(wc.B, wc.Hq, wc.S, wc.d)[:, :, pos].reshape(-1, wc.d)
    lc = lc.reshape(wc.B, wc.Hq, wc.S)[:, :, pos].reshape(-1)
    check(ob, lb, oc, lc, "balanced vs contiguous")


def test_balanced_first_position_is_v_row0_exactly(psr):
    # stored row 0 is global position 0: it sees key 0 only, with weight exactly 1
    torch = _torch()
    w = BASE.with_(name="cb_row0", B=2, Hq=4, Hkv=2, S=2048, P=4, d=128, causal=2, seed=69)
    q, k, v = ri.generate(w)
    o, lse, ws = psr.ring_attn_fwd(to_dev(torch, q), to_dev(torch, k), to_dev(torch, v), P=w.P, causal=2,
                                   scale=w.scale)
    assert psr.get_stats(ws)["status"] == 0
    o = o.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in range(w.B):
        for h in range(w.Hq):
            assert np.array_equal(o[b, h, 0], v[b, h // 2, 0])


def test_balanced_full_size_sampled_rows(psr):
    w = ri.WORKLOADS["h32_s32k_cb"]
    q, k, v = ri.generate(w)
    rows = ri.sample_rows(w)
    o_ref, lse_ref = oracle.for_workload(w, q, k, v, rows=rows)
    torch = _torch()
    o, lse, ws = psr.ring_attn_fwd(to_dev(torch, q), to_dev(torch, k), to_dev(torch, v), P=w.P, causal=2,
                                   scale=w.scale)
    st = psr.get_stats(ws)
    assert st["status"] == 0, st
    idx = torch.from_numpy(rows).cuda()
    o = o.view(-1, w.d).index_select(0, idx).float().cpu().numpy().astype(np.float64)
    lse = lse.view(-1).index_select(0, idx).cpu().numpy().astype(np.float64)
    check(o, lse, o_ref, lse_ref, w.name)
    assert st["staging_bytes"] == w.staging_bytes()
