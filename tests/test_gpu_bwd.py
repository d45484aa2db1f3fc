"""GPU parity of the Ring Attention backward (psr_ring_attn_bwd through the C ABI) against the
fp64 oracle (oracle/attn_bwd.py).  O and LSE come from this library's forward, as in training.

Bounds, derived from where the GPU path rounds (oracle/attn_bwd.py error_scales, pinned in
tests/test_oracle_attn_bwd.py against an emulation of those roundings).  The path rounds P to
bf16 in the forward before P V and in the backward before P dO and (K/V side) before forming dS,
takes O in bf16 for D = dO . O, rounds dS to bf16 before dS K and dS^T Q, accumulates in fp32
and rounds each gradient to bf16.  With u = 2^-8 (bf16 round to nearest) and n the most terms any
gradient element sums (S times the query heads per KV head):

  * every element:  |G - G_ref| <= (1.1 u + n 2^-23) E + 1.1 u |G_ref|, E the worst-case
    first-order sensitivity of error_scales (1.1: second-order terms; n 2^-23: fp32 accumulation
    with truncation);
  * L2:  ||G - G_ref|| <= u (1.1 ||G_ref|| + 2 sqrt(sum T2 / 3)) + 2 sqrt(n / 3) 2^-23 ||E||, the RMS
    of independent roundings (variance <= u^2/3 each, sums of squared terms T2; the n fp32 additions
    of an element each err by at most 2^-23 of a partial sum bounded by E) with a 2x margin.
"""
import numpy as np
import pytest

import ring_inputs as ri
from oracle import attn_bwd as ob

pytestmark = pytest.mark.gpu

U = 2.0 ** -8  # relative rounding error of bf16 (8 significant bits, round to nearest)


def _torch():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_bwd(psr, w, q, k, v, do):
    torch = _torch()
    qd, kd, vd, dod = (_dev(torch, x) for x in (q, k, v, do))
    o, lse, ws = psr.ring_attn_fwd(qd, kd, vd, P=w.P, causal=w.causal, scale=w.scale)
    assert psr.get_stats(ws)["status"] == 0
    dq, dk, dv, wsb = psr.ring_attn_bwd(qd, kd, vd, o, lse, dod, P=w.P, causal=w.causal, scale=w.scale)
    st = psr.get_stats(wsb)
    return _f64(dq), _f64(dk), _f64(dv), st


def check(name, got, ref, scales, n_terms):
    """got, ref: (dQ, dK, dV); scales: ((Eq, Ek, Ev), (T2q, T2k, T2v)) of the same elements."""
    fp32 = n_terms * 2.0 ** -23                       # worst case over n additions
    fp32_rms = 2.0 * np.sqrt(n_terms / 3.0) * 2.0 ** -23  # independent additions, 2x margin
    for g, r, e, t2, what in zip(got, ref, scales[0], scales[1], ("dQ", "dK", "dV")):
        g = g.reshape(r.shape)
        assert np.all(np.isfinite(g)), f"{name} {what}: non-finite"
        err = np.abs(g - r)
        excess = float(np.max(err - ((1.1 * U + fp32) * e + 1.1 * U * np.abs(r))))
        l2 = float(np.linalg.norm(err))
        l2_bound = U * (1.1 * np.linalg.norm(r) + 2.0 * np.sqrt(t2.sum() / 3.0)) + fp32_rms * np.linalg.norm(e)
        print(f"{name} {what}: rel L2 {l2 / np.linalg.norm(r):.2e} (bound {l2_bound / np.linalg.norm(r):.2e}), "
              f"max |err| / max |ref| {np.max(err) / np.max(np.abs(r)):.2e}")
        assert excess <= 0.0, f"{name} {what}: an element exceeds its bound by {excess:.3e}"
        assert l2 <= l2_bound, f"{name} {what}: L2 error {l2:.3e} over {l2_bound:.3e}"


def full_check(name, w, q, k, v, do, got, causal=None):
    causal = bool(w.causal) if causal is None else causal
    ref = ob.attn_bwd(q, k, v, do, causal=causal, scale=w.scale)
    check(name, got, ref, ob.error_scales(q, k, v, do, causal=causal, scale=w.scale), w.S * (w.Hq // w.Hkv))


BASE = ri.WORKLOADS["small"]                                                 # B1 H2 S1024 P4 d64
SMALL = [
    BASE.with_(name="bwd_nc_d64", seed=91),
    BASE.with_(name="bwd_c_d64", causal=True, seed=92),
    BASE.with_(name="bwd_c_d128_p4", S=2048, P=4, d=128, causal=True, seed=93),
    BASE.with_(name="bwd_gqa_c", B=2, Hq=4, Hkv=2, S=1024, P=2, d=128, causal=True, seed=94),
    BASE.with_(name="bwd_p1_nc_d128", S=512, P=1, d=128, seed=95),
    BASE.with_(name="bwd_p8_c", Hq=1, Hkv=1, S=2048, P=8, d=128, causal=True, seed=96),
    BASE.with_(name="bwd_mqa_d64_l256", Hq=4, Hkv=1, S=2048, P=8, d=64, causal=True, seed=90, qmul=2.0, kmul=2.0),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_bwd_every_element(psr, w):
    q, k, v = ri.generate(w)
    do = ri.generate_dout(w)
    dq, dk, dv, st = run_bwd(psr, w, q, k, v, do)
    assert st["status"] == 0, st
    assert st["compute_items"] == (w.B * w.Hkv + w.B * w.Hq) * w.S // 128  # K/V items + query items
    full_check(w.name, w, q, k, v, do, (dq, dk, dv))


def test_bwd_full_size_sampled_rows(psr):
    # B1 H32 S32768 P16 d128 causal on 2 heads (the fp64 LSE/D pass needs every row of a head)
    w = ri.WORKLOADS["h32_s32k_c"].with_(name="bwd_s32k_h2", Hq=2, Hkv=2, seed=97)
    q, k, v = ri.generate(w)
    do = ri.generate_dout(w)
    dq, dk, dv, st = run_bwd(psr, w, q, k, v, do)
    assert st["status"] == 0, st
    rng = np.random.default_rng(5)
    qr = np.unique(np.concatenate([[0, 1, w.S - 1, w.S, 2 * w.S - 1], rng.choice(w.B * w.Hq * w.S, 60, replace=False)]))
    kr = np.unique(np.concatenate([[0, 127, 128, w.S - 1, w.S], rng.choice(w.B * w.Hkv * w.S, 60, replace=False)]))
    ref, e, t2 = ob.attn_bwd_rows(q, k, v, do, causal=True, scale=w.scale, bh_rows=qr, kv_rows=kr, with_scales=True)
    check(w.name, (dq.reshape(-1, w.d)[qr], dk.reshape(-1, w.d)[kr], dv.reshape(-1, w.d)[kr]), ref, (e, t2), w.S)


def _balanced_order(S, P):
    """Natural position held by each stored row: shard r holds half-chunks r and 2P-1-r."""
    h = S // P // 2
    return np.concatenate([np.arange(c * h, (c + 1) * h) for r in range(P) for c in (r, 2 * P - 1 - r)])


@pytest.mark.parametrize("w", [BASE.with_(name="bwd_cb_d64", S=2048, P=4, causal=2, seed=98),
                               BASE.with_(name="bwd_cb_gqa_d128", B=1, Hq=4, Hkv=2, S=4096, P=4, d=128, causal=2,
                                          seed=99)], ids=lambda w: w.name)
def test_bwd_balanced_shards(psr, w):
    # the sequence stored in balanced shard order: the reference is the pinned oracle's causal
    # gradient of the same sequence in natural order, re-ordered the same way
    q, k, v = ri.generate(w)
    do = ri.generate_dout(w)
    pos = _balanced_order(w.S, w.P)  # stored row i holds natural row pos[i]
    nat = lambda a: a[:, :, np.argsort(pos)]
    rq, rk, rv = ob.attn_bwd(nat(q), nat(k), nat(v), nat(do), causal=True, scale=w.scale)
    ref = tuple(g[:, :, pos] for g in (rq, rk, rv))
    E, T2 = ob.error_scales(nat(q), nat(k), nat(v), nat(do), causal=True, scale=w.scale)
    scales = (tuple(x[:, :, pos] for x in E), tuple(x[:, :, pos] for x in T2))
    dq, dk, dv, st = run_bwd(psr, w, q, k, v, do)
    assert st["status"] == 0, st
    check(w.name, (dq, dk, dv), ref, scales, w.S * (w.Hq // w.Hkv))
