"""Pins of the attention-backward oracle (oracle/attn_bwd.py) against things other than its
own formulas: central finite differences of the forward (a float64 forward written here and
itself checked against the pinned C forward oracle on the bf16 grid), the single-key and
uniform-attention closed forms, GQA as a sum over repeated heads, and mutants of plausible
mistakes that the pins must catch."""
import numpy as np
import pytest

import oracle
import ring_inputs as ri
from oracle import attn_bwd as ob


def _bits(rng, shape, scale=1.0):
    return ri.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def forward64(q, k, v, causal, scale):
    """Real-valued forward (float64 arrays in, O out): the definition the C oracle computes."""
    B, Hq, S, d = q.shape
    g = Hq // k.shape[1]
    o = np.zeros_like(q)
    for b in range(B):
        for h in range(Hq):
            s = scale * q[b, h] @ k[b, h // g].T
            if causal:
                s = np.where(np.triu(np.ones((S, S), dtype=bool), 1), -np.inf, s)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            o[b, h] = (p / p.sum(axis=1, keepdims=True)) @ v[b, h // g]
    return o


def test_forward64_matches_the_c_oracle():
    rng = np.random.default_rng(7)
    for causal in (False, True):
        q, k, v = _bits(rng, (1, 4, 12, 8), 1.5), _bits(rng, (1, 2, 12, 8), 1.5), _bits(rng, (1, 2, 12, 8))
        o_c, _ = oracle.attn_fwd(q, k, v, B=1, Hq=4, Hkv=2, S=12, d=8, causal=causal, n_threads=2)
        f = ri.bf16_bits_to_f64
        o64 = forward64(f(q), f(k), f(v), causal, 1.0 / np.sqrt(8))
        assert np.max(np.abs(o64.reshape(-1, 8) - o_c)) <= 1e-13


def pin_finite_differences(impl):
    """<dL/dX, E> for L = sum(dO * O) against central differences of forward64 along random E."""
    rng = np.random.default_rng(11)
    for causal, (B, Hq, Hkv, S, d) in ((False, (1, 2, 1, 6, 4)), (True, (1, 2, 2, 7, 3)), (True, (2, 2, 1, 5, 4))):
        q, k, v, do = (_bits(rng, s, 1.2) for s in ((B, Hq, S, d), (B, Hkv, S, d), (B, Hkv, S, d), (B, Hq, S, d)))
        scale = 1.0 / np.sqrt(d)
        dq, dk, dv = impl(q, k, v, do, causal=causal, scale=scale)
        f = ri.bf16_bits_to_f64
        X = [f(q), f(k), f(v)]
        dOf = f(do)
        loss = lambda xs: float(np.sum(dOf * forward64(xs[0], xs[1], xs[2], causal, scale)))
        for which, grad in enumerate((dq, dk, dv)):
            for _ in range(2):
                E = rng.standard_normal(X[which].shape)
                h = 1e-5
                xp = [x.copy() for x in X]
                xm = [x.copy() for x in X]
                xp[which] += h * E
                xm[which] -= h * E
                fd = (loss(xp) - loss(xm)) / (2 * h)
                if not abs(fd - float(np.sum(grad * E))) <= 1e-7 * max(1.0, abs(fd)):  # NaN fails too
                    return False
    return True


def pin_single_key(impl):
    # S = 1: the only key gets weight 1, so dV = dO (summed over the group) and dQ = dK = 0
    rng = np.random.default_rng(12)
    q, k, v, do = _bits(rng, (1, 2, 1, 4)), _bits(rng, (1, 1, 1, 4)), _bits(rng, (1, 1, 1, 4)), _bits(rng, (1, 2, 1, 4))
    dq, dk, dv = impl(q, k, v, do, causal=False, scale=0.5)
    f = ri.bf16_bits_to_f64
    return (np.allclose(dq, 0, atol=1e-15) and np.allclose(dk, 0, atol=1e-15)
            and np.allclose(dv[0, 0], f(do)[0, 0] + f(do)[0, 1], rtol=0, atol=1e-15))


def pin_uniform_attention(impl):
    # Q = 0 (non-causal): P = 1/S everywhere, so dV_j = mean_i dO_i, dK = 0 and
    # dQ_i = scale/S * sum_j (dO_i . (v_j - mean v)) k_j
    rng = np.random.default_rng(13)
    S, d = 6, 4
    q = np.zeros((1, 1, S, d), dtype=np.uint16)
    k, v, do = _bits(rng, (1, 1, S, d)), _bits(rng, (1, 1, S, d)), _bits(rng, (1, 1, S, d))
    scale = 0.7
    dq, dk, dv = impl(q, k, v, do, causal=False, scale=scale)
    f = ri.bf16_bits_to_f64
    K, V, dO = f(k)[0, 0], f(v)[0, 0], f(do)[0, 0]
    want_dv = np.tile(dO.mean(axis=0), (S, 1))
    want_dq = scale / S * (dO @ (V - V.mean(axis=0)).T) @ K
    return (np.allclose(dv[0, 0], want_dv, rtol=1e-13, atol=1e-14) and np.allclose(dk, 0, atol=1e-14)
            and np.allclose(dq[0, 0], want_dq, rtol=1e-12, atol=1e-13))


def pin_gqa_is_a_sum_over_heads(impl):
    # two query heads sharing one KV head = the same heads over two copies of it, summed
    rng = np.random.default_rng(14)
    q, k, v, do = _bits(rng, (1, 2, 5, 4)), _bits(rng, (1, 1, 5, 4)), _bits(rng, (1, 1, 5, 4)), _bits(rng, (1, 2, 5, 4))
    g1 = impl(q, k, v, do, causal=True, scale=0.5)
    g2 = impl(q, np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1), do, causal=True, scale=0.5)
    return (np.allclose(g1[0], g2[0], rtol=1e-13, atol=1e-14) and np.allclose(g1[1][0, 0], g2[1][0].sum(axis=0))
            and np.allclose(g1[2][0, 0], g2[2][0].sum(axis=0)))


PINS = [pin_finite_differences, pin_single_key, pin_uniform_attention, pin_gqa_is_a_sum_over_heads]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_passes_pin(pin):
    assert pin(ob.attn_bwd)


def _mutant(change):
    """A copy of attn_bwd with one plausible mistake (the chain-rule steps written out again
    with the change applied)."""
    def impl(q_bits, k_bits, v_bits, do_bits, *, causal, scale=None):
        q, k, v, do = (ob.bf16_to_f64(x) for x in (q_bits, k_bits, v_bits, do_bits))
        B, Hq, S, d = q.shape
        g = Hq // k.shape[1]
        scale = 1.0 / np.sqrt(d) if scale is None else scale
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for b in range(B):
            for h in range(Hq):
                kv = h // g
                s = scale * q[b, h] @ k[b, kv].T
                if causal and change != "mask_open":
                    s = np.where(np.triu(np.ones((S, S), dtype=bool), 1), -np.inf, s)
                p = np.exp(s - s.max(axis=1, keepdims=True))
                p /= p.sum(axis=1, keepdims=True)
                o = p @ v[b, kv]
                dv[b, kv] += (p if change == "dv_untransposed" else p.T) @ do[b, h]
                dp = do[b, h] @ v[b, kv].T
                D = 0.0 if change == "no_delta" else np.sum(do[b, h] * o, axis=1)[:, None]
                ds = p * (dp - D)
                dq[b, h] = (1.0 if change == "dq_unscaled" else scale) * (ds @ k[b, kv])
                dk[b, kv] += scale * ((ds if change == "dk_untransposed" else ds.T) @ q[b, h])
        return dq, dk, dv
    return impl


@pytest.mark.parametrize("change", ["dv_untransposed", "no_delta", "dq_unscaled", "dk_untransposed", "mask_open"])
def test_pins_catch_mutant(change):
    assert not all(pin(_mutant(change)) for pin in PINS)


def test_unchanged_mutant_copy_passes():
    # the mutant copy without a change is the same computation (so the mutants above fail
    # because of their one change)
    assert all(pin(_mutant("none")) for pin in PINS)


def test_sampled_rows_match_full():
    rng = np.random.default_rng(15)
    for causal in (False, True):
        B, Hq, Hkv, S, d = 2, 4, 2, 40, 8
        q, k, v, do = _bits(rng, (B, Hq, S, d)), _bits(rng, (B, Hkv, S, d)), _bits(rng, (B, Hkv, S, d)), \
            _bits(rng, (B, Hq, S, d))
        dq, dk, dv = ob.attn_bwd(q, k, v, do, causal=causal, scale=0.3)
        qr = np.array([0, 5, S - 1, S + 3, 3 * S + 7, B * Hq * S - 1])
        kr = np.array([0, 1, S - 1, S + 2, 2 * S + 9, B * Hkv * S - 1])
        sq, sk, sv = ob.attn_bwd_rows(q, k, v, do, causal=causal, scale=0.3, bh_rows=qr, kv_rows=kr)
        assert np.allclose(sq, dq.reshape(-1, d)[qr], rtol=1e-12, atol=1e-13)
        assert np.allclose(sk, dk.reshape(-1, d)[kr], rtol=1e-12, atol=1e-13)
        assert np.allclose(sv, dv.reshape(-1, d)[kr], rtol=1e-12, atol=1e-13)


def test_dq_rows_match_full():
    rng = np.random.default_rng(16)
    for causal in (False, True):
        B, Hq, Hkv, S, d = 1, 4, 2, 32, 8
        q, k, v, do = _bits(rng, (B, Hq, S, d)), _bits(rng, (B, Hkv, S, d)), _bits(rng, (B, Hkv, S, d)), \
            _bits(rng, (B, Hq, S, d))
        dq, _, _ = ob.attn_bwd(q, k, v, do, causal=causal, scale=0.4)
        rows = np.array([0, 3, S - 1, S + 1, 2 * S + 30, B * Hq * S - 1])
        got = ob.attn_bwd_dq_rows(q, k, v, do, causal=causal, scale=0.4, bh_rows=rows)
        assert np.allclose(got, dq.reshape(-1, d)[rows], rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------------------------------------
# The GPU parity bounds come from error_scales.  Pin it against an emulation of the roundings it
# models (numpy, float64 between the bf16 roundings): the emulated gradients must stay inside the
# worst-case bound, and their L2 deviation inside the independent-rounding bound.
# ------------------------------------------------------------------------------------------------
U = 2.0 ** -8  # relative rounding error of bf16 (8 significant bits, round to nearest)


def _bf16(x):
    """Round float64 to the nearest bf16 (via float32; ties to even), as float64."""
    b = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def _emulated_bf16_path(q_bits, k_bits, v_bits, do_bits, causal, scale):
    """Forward and backward with bf16 roundings where a bf16 tensor-core path makes them: P before
    P V, O; P before P dO and before dS (the K/V side), dS before dS K and dS^T Q, the gradients.
    The query side forms dS from the unrounded P, as the dQ pass does."""
    f = ri.bf16_bits_to_f64
    q, k, v, do = f(q_bits), f(k_bits), f(v_bits), f(do_bits)
    B, Hq, S, d = q.shape
    g = Hq // k.shape[1]
    dq = np.zeros_like(q)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    mask = np.triu(np.ones((S, S), dtype=bool), 1) if causal else np.zeros((S, S), dtype=bool)
    for b in range(B):
        for h in range(Hq):
            kh, vh = k[b, h // g], v[b, h // g]
            s = np.where(mask, -np.inf, scale * q[b, h] @ kh.T)
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            l = e.sum(axis=1, keepdims=True)
            o = _bf16((_bf16(e) @ vh) / l)
            lse = m + np.log(l)
            p = np.exp(s - lse)
            pr = _bf16(p)
            dp = do[b, h] @ vh.T
            D = np.sum(do[b, h] * o, axis=1, keepdims=True)
            dv[b, h // g] += pr.T @ do[b, h]
            dk[b, h // g] += scale * (_bf16(pr * (dp - D)).T @ q[b, h])
            dq[b, h] = _bf16(scale * (_bf16(p * (dp - D)) @ kh))
    return dq, _bf16(dk), _bf16(dv)


@pytest.mark.parametrize("causal,Hq,Hkv,seed", [(False, 2, 2, 31), (True, 2, 2, 32), (True, 4, 2, 33)])
def test_error_scales_cover_emulated_bf16_roundings(causal, Hq, Hkv, seed):
    rng = np.random.default_rng(seed)
    S, d, scale = 256, 32, 0.3
    q, k, v = _bits(rng, (1, Hq, S, d), 1.5), _bits(rng, (1, Hkv, S, d), 1.5), _bits(rng, (1, Hkv, S, d))
    do = _bits(rng, (1, Hq, S, d))
    exact = ob.attn_bwd(q, k, v, do, causal=causal, scale=scale)
    emul = _emulated_bf16_path(q, k, v, do, causal, scale)
    (E, T2) = ob.error_scales(q, k, v, do, causal=causal, scale=scale)
    for g_em, g_ex, e, t2 in zip(emul, exact, E, T2):
        err = np.abs(g_em - g_ex)
        # worst case, first order in U (second-order terms are below 1 % of it)
        assert np.all(err <= 1.01 * U * (e + np.abs(g_ex)) + 1e-300)
        # independent roundings: L2 deviation within twice its RMS bound, plus the outputs' rounding
        rms = U * np.sqrt(t2.sum() / 3.0)
        assert np.linalg.norm(err) <= 2.0 * rms + U * np.linalg.norm(g_ex)
        # and the bounds are not vacuous: the deviation is a visible share of them
        assert np.linalg.norm(err) >= 0.1 * rms


def test_error_scale_rows_match_full():
    rng = np.random.default_rng(41)
    q, k, v = _bits(rng, (1, 4, 64, 16), 1.5), _bits(rng, (1, 2, 64, 16), 1.5), _bits(rng, (1, 2, 64, 16))
    do = _bits(rng, (1, 4, 64, 16))
    for causal in (False, True):
        (E, T2) = ob.error_scales(q, k, v, do, causal=causal, scale=0.3)
        qr, kr = np.array([0, 9, 64 + 63, 3 * 64 + 5]), np.array([0, 17, 64 + 63])
        _, e_rows, t_rows = ob.attn_bwd_rows(q, k, v, do, causal=causal, scale=0.3, bh_rows=qr, kv_rows=kr,
                                             with_scales=True)
        for got, full, rows in zip(e_rows + t_rows, E + T2, (qr, kr, kr, qr, kr, kr)):
            assert np.allclose(got, full.reshape(-1, 16)[rows], rtol=1e-12, atol=1e-300)
