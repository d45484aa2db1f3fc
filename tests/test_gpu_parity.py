"""GPU parity: the CUDA ring-attention path (through the C ABI) against the fp64 oracle.

Tolerances (bf16 inputs, fp32 accumulation): max |dO| <= 2e-2,
||dO||_2 / ||O_ref||_2 <= 5e-3, max |dLSE| <= 1e-3, over the compared rows.
Small workloads compare every row; the full-size workloads compare a fixed
sample of >= 4096 rows that includes rows 0, 1, 127, 128, S-1 and the first and
last row of every shard for every (b, hq).
"""
import numpy as np
import pytest

import oracle
import ring_inputs as ri

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
REL_L2 = 5e-3
LSE_ABS = 1e-3


def _torch():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def to_dev(torch, arr):
    return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).cuda().view(torch.bfloat16)


def gpu_run(psr, w, q, k, v, partition=None, rows=None):
    torch = _torch()
    qd, kd, vd = to_dev(torch, q), to_dev(torch, k), to_dev(torch, v)
    o, lse, ws = psr.ring_attn_fwd(qd, kd, vd, P=w.P, causal=w.causal, scale=w.scale, partition=partition)
    st = psr.get_stats(ws)
    assert st["status"] == 0, st
    o = o.view(-1, w.d)
    lse = lse.view(-1)
    if rows is not None:
        idx = torch.from_numpy(rows).cuda()
        o = o.index_select(0, idx)
        lse = lse.index_select(0, idx)
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), st


def check(o, lse, o_ref, lse_ref, what=""):
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    d = np.abs(o - o_ref)
    max_abs = float(d.max())
    rel = float(np.linalg.norm(o - o_ref) / np.linalg.norm(o_ref))
    lse_err = float(np.abs(lse - lse_ref).max())
    assert max_abs <= MAX_ABS, f"{what}: max |dO| = {max_abs:.3e}"
    assert rel <= REL_L2, f"{what}: rel L2 = {rel:.3e}"
    assert lse_err <= LSE_ABS, f"{what}: max |dLSE| = {lse_err:.3e}"
    return max_abs, rel, lse_err


_cache = {}


def item_rows_allowed(w):
    # single CTAs take 256-row items; a library built with CTA pairs takes 512-row items
    # for d = 128 when a shard holds whole 512-row items
    return (256, 512) if (w.d == 128 and (w.S // w.P) % 512 == 0) else (256,)


def inputs(w):
    key = w
    if key not in _cache:
        _cache.clear()
        _cache[key] = ri.generate(w)
    return _cache[key]


# ------------------------------------------------------------------------------------------------
# small workloads: every row
# ------------------------------------------------------------------------------------------------

SMALL = [
    ri.WORKLOADS["small"],                                             # B1 H2 S1024 P4 d64
    ri.WORKLOADS["small"].with_(name="small_c", causal=True),
    ri.WORKLOADS["small"].with_(name="small_d128", d=128, seed=11),
    ri.WORKLOADS["small"].with_(name="gqa_c", B=2, Hq=6, Hkv=2, S=768, P=3, causal=True, seed=12, qmul=2.0,
                                kmul=2.0),
    ri.WORKLOADS["small"].with_(name="p1", P=1, seed=13),              # no ring: everything local
    ri.WORKLOADS["small"].with_(name="p8_c_d128", S=2048, P=8, d=128, causal=True, seed=14),
    ri.WORKLOADS["small"].with_(name="b3_p5", B=3, Hq=4, Hkv=4, S=1280, P=5, seed=15),
    ri.WORKLOADS["long_s128k_c"].with_(name="outlier_small", S=4096, P=4, Hq=2, Hkv=2, seed=16),
    # d = 128 with shards of whole 512-row items (CTA-pair items in a library built with pairs)
    ri.WORKLOADS["small"].with_(name="l1024_nc", S=2048, P=2, d=128, seed=17),
    ri.WORKLOADS["small"].with_(name="l1024_gqa_c", B=2, Hq=4, Hkv=2, S=3072, P=3, d=128, causal=True, seed=18,
                                qmul=2.0, kmul=2.0),
    ri.WORKLOADS["small"].with_(name="l1024_p1_c", S=1024, P=1, d=128, causal=True, seed=19),
    ri.WORKLOADS["small"].with_(name="l1536_p4_c", Hq=3, Hkv=3, S=6144, P=4, d=128, causal=True, seed=20),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_all_rows(psr, w):
    q, k, v = inputs(w)
    o_ref, lse_ref = oracle.for_workload(w, q, k, v)
    o, lse, st = gpu_run(psr, w, q, k, v)
    check(o, lse, o_ref, lse_ref, w.name)
    assert st["staging_bytes"] == w.staging_bytes()
    assert any(st["compute_items"] == w.B * w.Hq * w.S // r for r in item_rows_allowed(w))


@pytest.mark.parametrize("n_s", [1, 3, 16])
@pytest.mark.parametrize("d", [64, 128])
def test_small_static_partitions(psr, n_s, d):
    # d = 128 with 512-row shards runs CTA pairs (a pair stages while 2 * pair < n_s)
    w = ri.WORKLOADS["small"].with_(name=f"small_static_d{d}", S=4096 if d == 128 else 2048, P=8 if d == 64 else 4,
                                    d=d, causal=True, seed=21)
    q, k, v = inputs(w)
    o_ref, lse_ref = oracle.for_workload(w, q, k, v)
    o, lse, st = gpu_run(psr, w, q, k, v, partition=psr.make_partition(psr.STATIC, n_staging=n_s))
    check(o, lse, o_ref, lse_ref, f"static n_s={n_s}")
    assert st["n_s_final"] == n_s


def test_causal_row0_is_v_row0_exactly(psr):
    torch = _torch()
    w = ri.WORKLOADS["small"].with_(name="row0", B=2, Hq=4, Hkv=2, S=1024, P=4, d=128, causal=True, seed=31)
    q, k, v = inputs(w)
    qd, kd, vd = to_dev(torch, q), to_dev(torch, k), to_dev(torch, v)
    o, lse, ws = psr.ring_attn_fwd(qd, kd, vd, P=w.P, causal=True, scale=w.scale)
    assert psr.get_stats(ws)["status"] == 0
    o = o.view(torch.int16).cpu().numpy().view(np.uint16)
    lse = lse.cpu().numpy()
    qf, kf = ri.bf16_bits_to_f64(q), ri.bf16_bits_to_f64(k)
    for b in range(w.B):
        for h in range(w.Hq):
            kvh = h // (w.Hq // w.Hkv)
            assert np.array_equal(o[b, h, 0], v[b, kvh, 0])  # weight exactly 1, bf16 round trip exact
            s00 = w.scale * float(np.dot(qf[b, h, 0], kf[b, kvh, 0]))
            assert abs(lse[b, h, 0] - s00) <= LSE_ABS


# ------------------------------------------------------------------------------------------------
# full-size workloads: sampled rows, in the launch configuration the benchmark uses
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["h32_s32k_nc", "h32_s32k_c", "gqa_s64k_c", "long_s128k_c"])
def test_full_size_sampled_rows(psr, name):
    w = ri.WORKLOADS[name]
    q, k, v = inputs(w)
    rows = ri.sample_rows(w)
    o_ref, lse_ref = oracle.for_workload(w, q, k, v, rows=rows)
    o, lse, st = gpu_run(psr, w, q, k, v, rows=rows)
    check(o, lse, o_ref, lse_ref, name)
    assert st["staging_bytes"] == w.staging_bytes()


@pytest.mark.parametrize("d", [64, 128])
def test_sweep_against_oracle_and_across_P(psr, d):
    """Partition-stress sweep (B1 H16 S16384): every P matches the oracle on every
    row (one fp64 oracle pass per d, the same inputs for every P) and every other
    P on all rows (the result does not depend on the ring size)."""
    base = ri.WORKLOADS[f"sweep_d{d}_P2"]
    q, k, v = inputs(base)
    o_ref, lse_ref = oracle.for_workload(base, q, k, v)
    first = None
    for P in (2, 4, 8, 16, 32, 64):
        w = ri.WORKLOADS[f"sweep_d{d}_P{P}"]
        o, lse, st = gpu_run(psr, w, q, k, v)
        check(o, lse, o_ref, lse_ref, f"d{d} P{P} vs oracle")
        if first is None:
            first = (o, lse)
        else:
            check(o, lse, first[0], first[1], f"d{d} P{P} vs P2")
        assert st["staging_bytes"] == w.staging_bytes()


def test_static_and_adaptive_agree(psr):
    w = ri.WORKLOADS["sweep_d128_P16"]
    q, k, v = inputs(w)
    rows = ri.sample_rows(w, n_random=1024)
    o_ref, lse_ref = oracle.for_workload(w, q, k, v, rows=rows)
    outs = []
    for part in (psr.make_partition(psr.ADAPTIVE), psr.make_partition(psr.STATIC, n_staging=2),
                 psr.make_partition(psr.STATIC, n_staging=32), psr.make_partition(psr.ADAPTIVE, n_staging=60)):
        o, lse, _ = gpu_run(psr, w, q, k, v, partition=part)
        check(o[rows], lse[rows], o_ref, lse_ref, f"mode {part.mode} n_s {part.n_staging}")
        outs.append((o, lse))
    for o, lse in outs[1:]:
        check(o, lse, outs[0][0], outs[0][1], "across partitions")


def test_initial_split_keeps_compute_waves(psr):
    """The adaptive launch's initial split on a 152-SM GB300.  B1 H16 S16384 has 1024 equal
    (non-causal) items: at P = 16 the rule with its staging headroom asks for ~30 staging CTAs,
    which leaves 122 compute CTAs and 9 waves; 24 is the largest split with 8 waves (1024 / 128),
    so the launch starts there.  At P = 32 (4-tile ring steps) the rule asks for 51 (d = 64) and
    54 (d = 128); the split the staging work needs (41 and 43 at the wave margin) leaves 10
    waves, 49 is the largest split with 10 (152 - ceil(1024 / 10)), and 48 the largest whose
    compute CTAs hold whole two-item groups.  d = 128, P = 16 (the rule's 32 is below the
    group-aligned 9-wave cap of 36) starts at the rule's split."""
    torch = _torch()
    if psr.num_ctas() != 152:
        pytest.skip("expected splits are for 152 SMs")
    assert -(-1024 // (152 - 24)) == 8 and -(-1024 // (152 - 25)) == 9
    assert -(-1024 // (152 - 49)) == 10 and -(-1024 // (152 - 50)) == 11 and (152 - 48) % 2 == 0
    for name, want in (("sweep_d64_P16", 24), ("sweep_d64_P32", 48), ("sweep_d128_P32", 48), ("sweep_d128_P16", 32)):
        w = ri.WORKLOADS[name]
        sh = (w.B, w.Hq, w.S, w.d)
        q = torch.zeros(sh, dtype=torch.bfloat16, device="cuda")
        k = torch.zeros((w.B, w.Hkv, w.S, w.d), dtype=torch.bfloat16, device="cuda")
        o, lse, ws = psr.ring_attn_fwd(q, k, k, P=w.P, causal=w.causal, scale=w.scale)
        st = psr.get_stats(ws)
        assert st["status"] == 0 and st["n_s_initial"] == want, (name, st)


@pytest.mark.parametrize("causal,d", [(False, 64), (False, 128), (True, 128)])
def test_running_max_rescale_path(psr, causal, d):
    """Keys of later chunks scaled up by 8 (exact in bf16): the running maximum of the rows whose
    first tiles hold unscaled keys is far below the scores of the later ring steps (up to ~25 more
    in log2 units), so the softmax takes its rare path there (the tile's sum of exponentials
    exceeds 2^16: row maximum, rescale of O and l, exponentials again)."""
    w = ri.WORKLOADS["small"].with_(name=f"rescale_{'c' if causal else 'nc'}_d{d}", S=2048, P=8, d=d,
                                    causal=causal, seed=91)
    q, k, v = ri.generate(w)
    kf = ri.bf16_bits_to_f32(k).reshape(w.B, w.Hkv, w.S, w.d)
    # keys from position 512 on (chunks 2..7): x8
    kf[:, :, 512:, :] *= np.float32(8.0)
    k = ri.f32_to_bf16_bits(kf).reshape(k.shape)
    o_ref, lse_ref = oracle.for_workload(w, q, k, v)
    o, lse, st = gpu_run(psr, w, q, k, v)
    check(o, lse, o_ref, lse_ref, w.name)


# ------------------------------------------------------------------------------------------------
# host-buffer entry point and failure reporting
# ------------------------------------------------------------------------------------------------

def test_host_buffer_entry_point(psr):
    torch = _torch()
    w = ri.WORKLOADS["small"].with_(name="host", causal=True, d=128, seed=41)
    q, k, v = inputs(w)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()
    qh, kh, vh = pin(q), pin(k), pin(v)
    oh = torch.empty(q.shape, dtype=torch.int16).pin_memory()
    lh = torch.empty(q.shape[:3], dtype=torch.float32).pin_memory()
    dq = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    dk = torch.empty(k.shape, dtype=torch.bfloat16, device="cuda")
    dv = torch.empty(v.shape, dtype=torch.bfloat16, device="cuda")
    do = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    dl = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    psr.ring_attn_fwd_host(qh, kh, vh, oh, lh, dq, dk, dv, do, dl, P=w.P, causal=True, scale=w.scale)
    o_ref, lse_ref = oracle.for_workload(w, q, k, v)
    o = ri.bf16_bits_to_f64(oh.numpy().view(np.uint16)).reshape(-1, w.d)
    check(o, lh.numpy().astype(np.float64).reshape(-1), o_ref, lse_ref, "host entry")


@pytest.mark.parametrize("shape", [(1, 8, 8, 32768, 16, False), (2, 8, 2, 16384, 8, True)],
                         ids=["kv_head_units", "batch_units_gqa_causal"])
def test_host_buffer_entry_point_pipelined(psr, shape):
    """The host entry streams the inputs in and the results out unit by unit (KV heads when
    B = 1, batches otherwise) around one launch whose items wait for their unit; the result
    equals the device entry's on the same inputs and matches the oracle on sampled rows."""
    torch = _torch()
    B, H, Hkv, S, P, causal = shape
    w = ri.WORKLOADS["small"].with_(name="host_streamed", B=B, Hq=H, Hkv=Hkv, S=S, P=P, d=128, causal=causal, seed=43)
    q, k, v = inputs(w)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()
    qh, kh, vh = pin(q), pin(k), pin(v)
    oh = torch.empty(q.shape, dtype=torch.int16).pin_memory()
    lh = torch.empty(q.shape[:3], dtype=torch.float32).pin_memory()
    dq = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    dk = torch.empty(k.shape, dtype=torch.bfloat16, device="cuda")
    dv = torch.empty(v.shape, dtype=torch.bfloat16, device="cuda")
    do = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    dl = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    psr.ring_attn_fwd_host(qh, kh, vh, oh, lh, dq, dk, dv, do, dl, P=w.P, causal=causal, scale=w.scale)
    o_dev, lse_dev, ws = psr.ring_attn_fwd(to_dev(torch, q), to_dev(torch, k), to_dev(torch, v), P=w.P, causal=causal,
                                           scale=w.scale)
    assert psr.get_stats(ws)["status"] == 0
    # same per-row arithmetic in the same order: identical results
    assert np.array_equal(oh.numpy(), o_dev.view(torch.int16).cpu().numpy())
    assert np.array_equal(lh.numpy(), lse_dev.cpu().numpy())
    rows = ri.sample_rows(w, n_random=1024)
    o_ref, lse_ref = oracle.for_workload(w, q, k, v, rows=rows)
    o = ri.bf16_bits_to_f64(oh.numpy().view(np.uint16)).reshape(-1, w.d)[rows]
    check(o, lh.numpy().astype(np.float64).reshape(-1)[rows], o_ref, lse_ref, "host entry, streamed")


def test_host_entry_reports_a_device_timeout_and_recovers(psr):
    """A dropped readiness flag inside the host entry's single launch: the call returns
    PSR_ERR_TIMEOUT (the launch releases the units' completion words, so the download stream
    does not wait for items that never finish), and the next call is correct."""
    torch = _torch()
    w = ri.WORKLOADS["small"].with_(name="host_fault", Hq=4, Hkv=4, S=2048, P=8, seed=47)
    q, k, v = inputs(w)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()
    qh, kh, vh = pin(q), pin(k), pin(v)
    oh = torch.empty(q.shape, dtype=torch.int16).pin_memory()
    lh = torch.empty(q.shape[:3], dtype=torch.float32).pin_memory()
    dq = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    dk = torch.empty(k.shape, dtype=torch.bfloat16, device="cuda")
    dv = torch.empty(v.shape, dtype=torch.bfloat16, device="cuda")
    do = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    dl = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    bufs = (qh, kh, vh, oh, lh, dq, dk, dv, do, dl)
    faulty = psr.make_partition(psr.ADAPTIVE, fault=psr.FAULT_DROP_FIRST_FLAG, timeout_ms=200)
    with pytest.raises(psr.PsrError) as e:
        psr.ring_attn_fwd_host(*bufs, P=w.P, causal=False, scale=w.scale, partition=faulty)
    assert e.value.status == psr.ERR_TIMEOUT
    psr.ring_attn_fwd_host(*bufs, P=w.P, causal=False, scale=w.scale)
    o_ref, lse_ref = oracle.for_workload(w, q, k, v)
    o = ri.bf16_bits_to_f64(oh.numpy().view(np.uint16)).reshape(-1, w.d)
    check(o, lh.numpy().astype(np.float64).reshape(-1), o_ref, lse_ref, "host entry after a timeout")


@pytest.mark.parametrize("d", [64, 128])
def test_dropped_flag_times_out_and_context_survives(psr, d):
    # d = 128 with 1024-row shards runs CTA pairs: both CTAs of every pair must leave together
    torch = _torch()
    w = ri.WORKLOADS["small"].with_(name=f"fault_d{d}", S=2048 if d == 64 else 4096, P=8 if d == 64 else 4, d=d,
                                    seed=51)
    q, k, v = inputs(w)
    qd, kd, vd = to_dev(torch, q), to_dev(torch, k), to_dev(torch, v)
    part = psr.make_partition(psr.ADAPTIVE, fault=psr.FAULT_DROP_FIRST_FLAG, timeout_ms=200)
    o, lse, ws = psr.ring_attn_fwd(qd, kd, vd, P=w.P, causal=False, scale=w.scale, partition=part)
    st = psr.get_stats(ws)
    assert st["status"] == psr.ERR_TIMEOUT
    # the first wait to give up is the producer's on the dropped flag (1), the MMA issuer's on
    # the K/V tile that producer therefore never loads (2), whichever of the two began first,
    # or an idle stager's (11)
    assert st["error_site"] in (1, 2, 11)
    # the context is still usable and the next launch on the same workspace is correct
    o_ref, lse_ref = oracle.for_workload(w, q, k, v)
    o2, lse2, st2 = gpu_run(psr, w, q, k, v)
    check(o2, lse2, o_ref, lse_ref, "after timeout")


def test_slow_staging_still_correct(psr):
    w = ri.WORKLOADS["small"].with_(name="slow", S=2048, P=8, causal=True, seed=61)
    q, k, v = inputs(w)
    o_ref, lse_ref = oracle.for_workload(w, q, k, v)
    o, lse, st = gpu_run(psr, w, q, k, v, partition=psr.make_partition(psr.ADAPTIVE, fault=psr.FAULT_SLOW_STAGING))
    check(o, lse, o_ref, lse_ref, "slow staging")
