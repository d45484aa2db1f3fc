"""Pins for the fp64 oracle: checks against what attention itself fixes.

The pages print no attention values, so the oracle is pinned by mathematics
that does not go through its own code: exact Decimal brute force on tiny
inputs, closed forms, reductions to simpler cases and invariants.  A final test
plants plausible mistakes in copies of oracle.c and checks that some pin fails.
"""
import ctypes
import decimal
import itertools
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import ring_inputs as ri

D = decimal.Decimal


def rand_bf16(rng, shape, scale=1.0):
    x = (rng.standard_normal(size=shape) * scale).astype(np.float32)
    return ri.f32_to_bf16_bits(x).reshape(shape)


def make(rng, B, Hq, Hkv, S, d, scale=1.0):
    q = rand_bf16(rng, (B, Hq, S, d), scale)
    k = rand_bf16(rng, (B, Hkv, S, d), scale)
    v = rand_bf16(rng, (B, Hkv, S, d))
    return q, k, v


def run(q, k, v, causal, P=1, scale=None, rows=None, chunked=False, perm=None):
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    if chunked:
        return oracle.attn_fwd_chunked(q, k, v, B=B, Hq=Hq, Hkv=Hkv, S=S, P=P, d=d, causal=causal, scale=scale,
                                       rows=rows, perm=perm, n_threads=4)
    return oracle.attn_fwd(q, k, v, B=B, Hq=Hq, Hkv=Hkv, S=S, P=P, d=d, causal=causal, scale=scale, rows=rows,
                           n_threads=4)


# ------------------------------------------------------------------------------------------------
# Exact brute force (Python Decimal, 40 digits)
# ------------------------------------------------------------------------------------------------

def balanced_positions(S, P):
    """Global position of each stored row under load-balanced shards, built from the
    list of half-chunks each shard holds: shard r holds half-chunks r and 2P-1-r."""
    h = S // P // 2
    chunks = [c for r in range(P) for c in (r, 2 * P - 1 - r)]
    return np.concatenate([np.arange(c * h, (c + 1) * h) for c in chunks])


def decimal_attention(q, k, v, causal, scale, positions=None):
    """Softmax attention evaluated in 40-digit decimal arithmetic, one row at a time.
    With `positions`, key j is visible to row i when positions[j] <= positions[i]."""
    ctx = decimal.Context(prec=40)
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    qf, kf, vf = (ri.bf16_bits_to_f64(x) for x in (q, k, v))
    sc = D(float(scale))
    o = np.zeros((B, Hq, S, d))
    lse = np.zeros((B, Hq, S))
    for b, h, i in itertools.product(range(B), range(Hq), range(S)):
        kv = h // g
        if positions is not None:
            keys = [j for j in range(S) if positions[j] <= positions[i]]
        else:
            keys = range(i + 1) if causal else range(S)
        s = []
        for j in keys:
            acc = D(0)
            for c in range(d):
                acc = ctx.add(acc, ctx.multiply(D(float(qf[b, h, i, c])), D(float(kf[b, kv, j, c]))))
            s.append(ctx.multiply(acc, sc))
        total = D(0)
        w = []
        for sj in s:
            e = ctx.exp(sj)
            w.append(e)
            total = ctx.add(total, e)
        for c in range(d):
            acc = D(0)
            for wj, j in zip(w, keys):
                acc = ctx.add(acc, ctx.multiply(wj, D(float(vf[b, kv, j, c]))))
            o[b, h, i, c] = float(ctx.divide(acc, total))
        lse[b, h, i] = float(ctx.ln(total))
    return o.reshape(-1, d), lse.reshape(-1)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,S,d", [(1, 1, 1, 7, 4), (1, 2, 1, 16, 8), (2, 2, 2, 9, 3)])
def test_decimal_brute_force(causal, B, Hq, Hkv, S, d):
    rng = np.random.default_rng(100 + S * d + Hq + B)
    q, k, v = make(rng, B, Hq, Hkv, S, d, scale=1.5)
    scale = 1.0 / np.sqrt(d)
    o, lse = run(q, k, v, causal, scale=scale)
    o_ref, lse_ref = decimal_attention(q, k, v, causal, scale)
    assert np.max(np.abs(o - o_ref)) <= 1e-13
    assert np.max(np.abs(lse - lse_ref)) <= 1e-13


# ------------------------------------------------------------------------------------------------
# Closed forms
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_q_zero_gives_mean_of_v(causal):
    rng = np.random.default_rng(1)
    B, H, S, d = 1, 2, 64, 16
    _, k, v = make(rng, B, H, H, S, d)
    q = np.zeros((B, H, S, d), dtype=np.uint16)  # +0.0 in bf16
    o, lse = run(q, k, v, causal)
    vf = ri.bf16_bits_to_f64(v)
    for h in range(H):
        for i in range(S):
            n = i + 1 if causal else S
            exp_o = vf[0, h, :n].mean(axis=0)
            assert np.max(np.abs(o[h * S + i] - exp_o)) <= 1e-14
            assert abs(lse[h * S + i] - np.log(n)) <= 1e-14


def test_single_key_returns_v_exactly():
    rng = np.random.default_rng(2)
    q, k, v = make(rng, 1, 3, 1, 1, 32)
    o, lse = run(q, k, v, causal=False, scale=0.125)
    vf = ri.bf16_bits_to_f64(v)[0, 0, 0]
    for h in range(3):
        assert np.array_equal(o[h], vf)  # weight exactly 1
        s_h = 0.125 * float(np.dot(ri.bf16_bits_to_f64(q[0, h, 0]), ri.bf16_bits_to_f64(k[0, 0, 0])))
        assert abs(lse[h] - s_h) <= 1e-14 * max(1.0, abs(s_h))


def test_causal_row0_is_v_row0():
    rng = np.random.default_rng(3)
    q, k, v = make(rng, 2, 4, 2, 32, 8)
    o, lse = run(q, k, v, causal=True, P=4)
    vf = ri.bf16_bits_to_f64(v)
    qf, kf = ri.bf16_bits_to_f64(q), ri.bf16_bits_to_f64(k)
    for b in range(2):
        for h in range(4):
            n = (b * 4 + h) * 32
            assert np.array_equal(o[n], vf[b, h // 2, 0])
            assert abs(lse[n] - np.dot(qf[b, h, 0], kf[b, h // 2, 0]) / np.sqrt(8)) <= 1e-13


# ------------------------------------------------------------------------------------------------
# Reductions and invariants
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_mha_with_repeated_heads(causal):
    rng = np.random.default_rng(4)
    B, Hq, Hkv, S, d = 2, 6, 2, 48, 16
    q, k, v = make(rng, B, Hq, Hkv, S, d)
    o, lse = run(q, k, v, causal)
    g = Hq // Hkv
    k_rep = np.repeat(k, g, axis=1)
    v_rep = np.repeat(v, g, axis=1)
    o2, lse2 = run(q, k_rep, v_rep, causal)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    # and the mapping is consecutive: head hq uses KV head hq // g, not hq % Hkv
    k_alt = np.tile(k, (1, g, 1, 1))
    v_alt = np.tile(v, (1, g, 1, 1))
    o3, _ = run(q, k_alt, v_alt, causal)
    assert not np.allclose(o, o3)


def test_causal_row_equals_noncausal_prefix():
    rng = np.random.default_rng(5)
    B, H, S, d = 1, 2, 40, 8
    q, k, v = make(rng, B, H, H, S, d)
    o, lse = run(q, k, v, True, scale=0.3)
    for i in (0, 1, 7, 22, 39):
        qs = np.ascontiguousarray(q[:, :, : i + 1])
        ks = np.ascontiguousarray(k[:, :, : i + 1])
        vs = np.ascontiguousarray(v[:, :, : i + 1])
        o2, lse2 = run(qs, ks, vs, False, scale=0.3)
        for h in range(H):
            assert np.max(np.abs(o[h * S + i] - o2[h * (i + 1) + i])) <= 1e-14
            assert abs(lse[h * S + i] - lse2[h * (i + 1) + i]) <= 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_bounds(causal):
    rng = np.random.default_rng(6)
    B, H, S, d = 1, 2, 96, 16
    q, k, v = make(rng, B, H, H, S, d, scale=2.0)
    o, lse = run(q, k, v, causal)
    qf, kf, vf = (ri.bf16_bits_to_f64(x) for x in (q, k, v))
    for h in range(H):
        s = qf[0, h] @ kf[0, h].T / np.sqrt(d)
        for i in range(S):
            n = i + 1 if causal else S
            row = h * S + i
            m = s[i, :n].max()
            assert m - 1e-12 <= lse[row] <= m + np.log(n) + 1e-12
            assert np.all(o[row] >= vf[0, h, :n].min(axis=0) - 1e-12)
            assert np.all(o[row] <= vf[0, h, :n].max(axis=0) + 1e-12)


def test_key_permutation_invariance():
    rng = np.random.default_rng(7)
    B, H, S, d = 1, 2, 64, 8
    q, k, v = make(rng, B, H, H, S, d)
    o, lse = run(q, k, v, False)
    perm = rng.permutation(S)
    o2, lse2 = run(q, np.ascontiguousarray(k[:, :, perm]), np.ascontiguousarray(v[:, :, perm]), False)
    assert np.max(np.abs(o - o2)) <= 1e-14 and np.max(np.abs(lse - lse2)) <= 1e-13


def test_key_duplication_adds_ln2():
    rng = np.random.default_rng(8)
    B, H, S, d = 1, 2, 32, 8
    q, k, v = make(rng, B, H, H, S, d)
    o, lse = run(q, k, v, False, scale=0.25)
    q2 = np.concatenate([q, q], axis=2)
    k2 = np.concatenate([k, k], axis=2)
    v2 = np.concatenate([v, v], axis=2)
    o2, lse2 = run(q2, k2, v2, False, scale=0.25)
    o2 = o2.reshape(H, 2 * S, d)[:, :S].reshape(-1, d)
    lse2 = lse2.reshape(H, 2 * S)[:, :S].reshape(-1)
    assert np.max(np.abs(o - o2)) <= 1e-14
    assert np.max(np.abs(lse2 - lse - np.log(2.0))) <= 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_chunked_merge_equals_direct_for_every_P(causal):
    rng = np.random.default_rng(9)
    B, Hq, Hkv, S, d = 1, 4, 2, 128, 16
    q, k, v = make(rng, B, Hq, Hkv, S, d, scale=1.5)
    o, lse = run(q, k, v, causal)
    for P in (1, 2, 4, 8, 16, 32, 64):
        oc, lsec = run(q, k, v, causal, P=P, chunked=True)
        assert np.max(np.abs(o - oc)) <= 1e-12, P
        assert np.max(np.abs(lse - lsec)) <= 1e-12, P
    for trial in range(3):
        perm = rng.permutation(8)
        oc, lsec = run(q, k, v, causal, P=8, chunked=True, perm=perm)
        assert np.max(np.abs(o - oc)) <= 1e-12
        assert np.max(np.abs(lse - lsec)) <= 1e-12


# ------------------------------------------------------------------------------------------------
# Load-balanced causal shards (causal=2)
# ------------------------------------------------------------------------------------------------

def test_balanced_positions_are_a_permutation():
    for S, P in ((8, 2), (12, 3), (64, 4), (4096, 16)):
        pos = balanced_positions(S, P)
        assert np.array_equal(np.sort(pos), np.arange(S))
        # every shard holds the same number of (query, key) pairs under the mask
        L = S // P
        work = [int(np.sum(pos[r * L:(r + 1) * L] + 1)) for r in range(P)]
        assert len(set(work)) == 1, work


@pytest.mark.parametrize("B,Hq,Hkv,S,P,d", [(1, 1, 1, 8, 2, 4), (1, 2, 1, 12, 3, 4), (2, 2, 2, 16, 4, 3)])
def test_balanced_decimal_brute_force(B, Hq, Hkv, S, P, d):
    rng = np.random.default_rng(300 + S + P)
    q, k, v = make(rng, B, Hq, Hkv, S, d, scale=1.5)
    scale = 1.0 / np.sqrt(d)
    o, lse = run(q, k, v, 2, P=P, scale=scale)
    o_ref, lse_ref = decimal_attention(q, k, v, True, scale, positions=balanced_positions(S, P))
    assert np.max(np.abs(o - o_ref)) <= 1e-13
    assert np.max(np.abs(lse - lse_ref)) <= 1e-13


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_balanced_equals_contiguous_on_the_reordered_sequence(P):
    # attention under a positional mask depends on positions only: storing the natural
    # sequence in balanced shard order must give the contiguous causal rows, re-ordered
    rng = np.random.default_rng(20 + P)
    B, Hq, Hkv, S, d = 1, 4, 2, 64, 8
    q, k, v = make(rng, B, Hq, Hkv, S, d, scale=1.5)
    o_nat, lse_nat = run(q, k, v, True)
    pos = balanced_positions(S, P)  # stored row i holds natural row pos[i]
    o_bal, lse_bal = run(q[:, :, pos], k[:, :, pos], v[:, :, pos], 2, P=P)
    o_nat = o_nat.reshape(B, Hq, S, d)[:, :, pos].reshape(-1, d)
    lse_nat = lse_nat.reshape(B, Hq, S)[:, :, pos].reshape(-1)
    if P == 1:  # identity layout: the same arithmetic in the same order
        assert np.array_equal(o_bal, o_nat) and np.array_equal(lse_bal, lse_nat)
    assert np.max(np.abs(o_bal - o_nat)) <= 1e-12
    assert np.max(np.abs(lse_bal - lse_nat)) <= 1e-12


def test_balanced_chunked_merge_equals_direct():
    rng = np.random.default_rng(21)
    B, Hq, Hkv, S, d = 1, 2, 1, 128, 16
    q, k, v = make(rng, B, Hq, Hkv, S, d, scale=1.5)
    for P in (1, 2, 4, 8, 16, 32, 64):
        o, lse = run(q, k, v, 2, P=P)
        oc, lsec = run(q, k, v, 2, P=P, chunked=True)
        assert np.max(np.abs(o - oc)) <= 1e-12, P
        assert np.max(np.abs(lse - lsec)) <= 1e-12, P


def test_balanced_rejects_odd_shards():
    rng = np.random.default_rng(22)
    q, k, v = make(rng, 1, 1, 1, 12, 4)
    with pytest.raises(ValueError):
        run(q, k, v, 2, P=4)  # L = 3 cannot be split in two halves


def test_row_subset_matches_full():
    w = ri.WORKLOADS["small"]
    q, k, v = ri.generate(w)
    o, lse = oracle.for_workload(w, q, k, v, n_threads=4)
    rows = np.array([0, 1, 255, 256, 1023, 1024, 2047], dtype=np.int64)
    o2, lse2 = oracle.for_workload(w, q, k, v, rows=rows, n_threads=2)
    assert np.array_equal(o[rows], o2) and np.array_equal(lse[rows], lse2)


def test_rejects_bad_arguments():
    rng = np.random.default_rng(10)
    q, k, v = make(rng, 1, 3, 2, 8, 4)
    with pytest.raises(ValueError):
        run(q, k, v, False)  # Hq % Hkv != 0
    q, k, v = make(rng, 1, 2, 2, 9, 4)
    with pytest.raises(ValueError):
        run(q, k, v, False, P=2)  # S % P != 0
    with pytest.raises(ValueError):
        run(q, k, v, False, rows=np.array([18]))  # row id out of range
    q, k, v = make(rng, 1, 2, 2, 8, 4)
    with pytest.raises(ValueError):
        run(q, k, v, False, P=4, chunked=True, perm=[0, 1, 1, 2])


# ------------------------------------------------------------------------------------------------
# Planted mistakes: each mutant of oracle.c must fail at least one pin above
# ------------------------------------------------------------------------------------------------

MUTANTS = {
    "lse_log2": ("return m + log(l);", "return m + log2(l);"),
    "dropped_max": ("double p = exp(s_buf[j - k0] - m);", "double p = exp(s_buf[j - k0]);\n    (void)m;"),
    "gqa_modulo": ("const int64_t kv = hq / g;", "const int64_t kv = hq % sh->Hkv;"),
    "causal_off_by_one": ("return sh->causal ? i + 1 : sh->S;", "return sh->causal ? i : sh->S;"),
    "no_scale": ("double s = sh->scale * dot_bf16(qrow, kbase + j * d, d);",
                 "double s = dot_bf16(qrow, kbase + j * d, d);"),
    "unnormalised": ("for (int c = 0; c < d; ++c) out[c] /= l;", "(void)0;"),
    "transposed_kv": ("const uint16_t *vr = vbase + j * d;", "const uint16_t *vr = kbase + j * d;"),
    "merge_sign": ("const double w = exp(part_lse[t] - lse);", "const double w = exp(lse - part_lse[t]);"),
    "balanced_half_order": ("(2 * (int64_t)sh->P - 1 - r) * h", "(sh->P + r) * h"),
    "balanced_mask_strict": ("position(sh, j) > qpos", "position(sh, j) >= qpos"),
    "balanced_first_half": ("return loc < h ? r * h + loc", "return loc < h ? r * L + loc"),
}


def _build_mutant(tmpdir, name, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert old in src, name
    path = os.path.join(tmpdir, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new, 1))
    shutil.copy(os.path.join(os.path.dirname(oracle.__file__), "oracle.h"), tmpdir)
    so = os.path.join(tmpdir, f"{name}.so")
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", path, "-o", so, "-lm", "-lpthread"])
    return so


def _pins_pass(so):
    """A compact re-run of the pins above against a given build of oracle.c."""
    lib = ctypes.CDLL(so)
    vp = ctypes.c_void_p
    lib.oracle_attn_fwd.argtypes = [ctypes.POINTER(oracle.OracleShape), vp, vp, vp, vp, ctypes.c_int64, vp, vp,
                                    ctypes.c_int]
    lib.oracle_attn_fwd_chunked.argtypes = [ctypes.POINTER(oracle.OracleShape), vp, vp, vp, vp, ctypes.c_int64,
                                            vp, vp, vp, ctypes.c_int]

    def call(q, k, v, causal, P=1, chunked=False):
        B, Hq, S, d = q.shape
        sh = oracle.OracleShape(B, Hq, k.shape[1], S, P, d, int(causal), 1.0 / np.sqrt(d))
        n = B * Hq * S
        o = np.empty((n, d))
        lse = np.empty(n)
        if chunked:
            lib.oracle_attn_fwd_chunked(ctypes.byref(sh), q.ctypes.data, k.ctypes.data, v.ctypes.data, None, n,
                                        None, o.ctypes.data, lse.ctypes.data, 2)
        else:
            lib.oracle_attn_fwd(ctypes.byref(sh), q.ctypes.data, k.ctypes.data, v.ctypes.data, None, n,
                                o.ctypes.data, lse.ctypes.data, 2)
        return o, lse

    rng = np.random.default_rng(11)
    for causal in (False, True):
        q, k, v = make(rng, 1, 4, 2, 6, 4, scale=1.5)
        o, lse = call(q, k, v, causal)
        o_ref, lse_ref = decimal_attention(q, k, v, causal, 1.0 / np.sqrt(4))
        if np.max(np.abs(o - o_ref)) > 1e-13 or np.max(np.abs(lse - lse_ref)) > 1e-13:
            return False
        q, k, v = make(rng, 1, 2, 2, 16, 4, scale=1.5)
        o, lse = call(q, k, v, causal)
        oc, lsec = call(q, k, v, causal, P=4, chunked=True)
        if np.max(np.abs(o - oc)) > 1e-12 or np.max(np.abs(lse - lsec)) > 1e-12:
            return False
    # load-balanced shards: brute force over the half-chunk positions
    for S, P in ((8, 2), (12, 3)):
        q, k, v = make(rng, 1, 2, 1, S, 4, scale=1.5)
        o, lse = call(q, k, v, 2, P=P)
        o_ref, lse_ref = decimal_attention(q, k, v, True, 1.0 / np.sqrt(4), positions=balanced_positions(S, P))
        if np.max(np.abs(o - o_ref)) > 1e-13 or np.max(np.abs(lse - lse_ref)) > 1e-13:
            return False
    return True


def test_pins_catch_planted_mistakes():
    tmp = tempfile.mkdtemp(prefix="oracle_mutants_")
    try:
        ok = _build_mutant(tmp, "unchanged", "int err;", "int err;")
        assert _pins_pass(ok), "unmodified oracle must pass the pins"
        for name, (old, new) in MUTANTS.items():
            so = _build_mutant(tmp, name, old, new)
            assert not _pins_pass(so), f"planted mistake '{name}' was not caught"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
