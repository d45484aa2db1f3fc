"""Pins of the AllGather + GEMM oracle (oracle/ag_gemm.py) against things other than itself:
40-digit Decimal brute force, closed forms (identity and one-hot weights), row locality
and linearity, the rank order of the gather, and mutants of plausible mistakes that each
of these must catch."""
from decimal import Decimal, getcontext

import numpy as np
import pytest

import ring_inputs as ri
from oracle import ag_gemm as og


def _bits(rng, shape, scale=1.0):
    return ri.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def brute_force(a_bits, w_bits, P):
    """sum_k A[m,k] * W_r[n,k] in 40-digit decimal arithmetic, straight from the definition:
    rank r's A is every shard, in rank order."""
    getcontext().prec = 40
    a = ri.bf16_bits_to_f64(a_bits)
    w = ri.bf16_bits_to_f64(w_bits)
    M, K = a.shape
    Ms = M // P
    out = np.zeros((P, M, w.shape[1]))
    for r in range(P):
        for j in range(P):                      # shard j, received by rank r
            for i in range(Ms):
                m = j * Ms + i
                for n in range(w.shape[1]):
                    s = sum(Decimal(float(a[m, k])) * Decimal(float(w[r, n, k])) for k in range(K))
                    out[r, m, n] = float(s)
    return out


# ------------------------------------------------------------------------------------------------
# pins (each takes the implementation under test)
# ------------------------------------------------------------------------------------------------

def pin_brute_force(impl):
    rng = np.random.default_rng(1)
    for (M, K, Ns, P) in ((8, 6, 3, 2), (6, 5, 2, 3), (4, 9, 4, 1)):
        a, w = _bits(rng, (M, K)), _bits(rng, (P, Ns, K))
        got, want = impl(a, w, P), brute_force(a, w, P)
        if not np.allclose(got, want, rtol=1e-13, atol=1e-13):
            return False
    return True


def pin_identity_weights(impl):
    # K = P*Ns and W_r = rows r*Ns..(r+1)*Ns of the identity: C_r = the columns of gathered A
    rng = np.random.default_rng(2)
    P, Ns, M = 4, 3, 8
    K = P * Ns
    a = _bits(rng, (M, K))
    eye = ri.f32_to_bf16_bits(np.eye(K, dtype=np.float32))
    w = eye.reshape(P, Ns, K)
    got = impl(a, w, P)
    af = ri.bf16_bits_to_f64(a)
    return all(np.array_equal(got[r], af[:, r * Ns:(r + 1) * Ns]) for r in range(P))


def pin_one_hot_a(impl):
    # A has a single nonzero a at (m, k): C_r[m, n] = a * W_r[n, k], every other row is 0
    rng = np.random.default_rng(3)
    P, Ms, K, Ns = 3, 2, 5, 4
    M = P * Ms
    w = _bits(rng, (P, Ns, K))
    for m, k in ((0, 0), (M - 1, K - 1), (Ms + 1, 2)):
        a = np.zeros((M, K), dtype=np.uint16)
        a[m, k] = ri.f32_to_bf16_bits(np.array([1.5], dtype=np.float32))[0]
        got = impl(a, w, P)
        want = np.zeros((P, M, Ns))
        want[:, m, :] = 1.5 * ri.bf16_bits_to_f64(w[:, :, k])
        if not np.array_equal(got, want):
            return False
    return True


def pin_row_locality_and_linearity(impl):
    rng = np.random.default_rng(4)
    P, Ms, K, Ns = 2, 4, 7, 3
    M = P * Ms
    a, w = _bits(rng, (M, K)), _bits(rng, (P, Ns, K))
    base = impl(a, w, P)
    a2 = a.copy()
    a2[5] = _bits(rng, (K,))
    changed = impl(a2, w, P)
    others = [m for m in range(M) if m != 5]
    if not np.array_equal(base[:, others], changed[:, others]) or np.array_equal(base[:, 5], changed[:, 5]):
        return False
    # linear in W: doubling W_1 (exact in bf16) doubles C_1 and leaves C_0
    w2 = w.copy()
    w2[1] = ri.f32_to_bf16_bits(ri.bf16_bits_to_f32(w[1]) * np.float32(2.0))
    c2 = impl(a, w2, P)
    return np.array_equal(c2[0], base[0]) and np.allclose(c2[1], 2.0 * base[1], rtol=0, atol=0)


PINS = [pin_brute_force, pin_identity_weights, pin_one_hot_a, pin_row_locality_and_linearity]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_passes_pin(pin):
    assert pin(og.ag_gemm)


# plausible mistakes: every one must fail at least one pin
def _mut_local_only(a, w, P):          # forgets the gather: only the rank's own shard, zeros elsewhere
    af, wf = og.bf16_to_f64(a), og.bf16_to_f64(w)
    Ms = af.shape[0] // P
    out = np.zeros((P, af.shape[0], wf.shape[1]))
    for r in range(P):
        out[r, r * Ms:(r + 1) * Ms] = af[r * Ms:(r + 1) * Ms] @ wf[r].T
    return out


def _mut_reversed_gather(a, w, P):     # gathers the shards in reverse rank order
    af, wf = og.bf16_to_f64(a), og.bf16_to_f64(w)
    Ms = af.shape[0] // P
    g = np.concatenate([af[j * Ms:(j + 1) * Ms] for j in reversed(range(P))])
    return np.stack([g @ wf[r].T for r in range(P)])


def _mut_wrong_rank_weight(a, w, P):   # uses rank (r+1)'s weights
    af, wf = og.bf16_to_f64(a), og.bf16_to_f64(w)
    return np.stack([af @ wf[(r + 1) % P].T for r in range(P)])


def _mut_fp32_accumulate(a, w, P):     # accumulates in fp32: caught by the 1e-13 brute force
    af, wf = og.bf16_to_f64(a).astype(np.float32), og.bf16_to_f64(w).astype(np.float32)
    return np.stack([(af @ wf[r].T).astype(np.float64) for r in range(P)])


def _mut_k_off_by_one(a, w, P):        # drops the last k of the contraction
    af, wf = og.bf16_to_f64(a), og.bf16_to_f64(w)
    return np.stack([af[:, :-1] @ wf[r][:, :-1].T for r in range(P)])


@pytest.mark.parametrize("mutant", [_mut_local_only, _mut_reversed_gather, _mut_wrong_rank_weight,
                                     _mut_fp32_accumulate, _mut_k_off_by_one], ids=lambda f: f.__name__)
def test_pins_catch_mutant(mutant):
    assert not all(pin(mutant) for pin in PINS)


def test_rows_option_matches_full():
    w = ri.AG_WORKLOADS["ag_small"].with_(M=64, K=32, Ns=16, P=4)
    a, ww = ri.generate_ag_gemm(w)
    full = og.for_workload(w, a, ww)
    rows = ri.ag_sample_rows(w, n_random=20)
    assert np.array_equal(og.for_workload(w, a, ww, rows=rows), full[:, rows])


def test_ag_inputs_share_the_seeded_stream():
    # A is elements [0, M*K) of the stream, W the next P*Ns*K, checked against the numpy restatement
    w = ri.AG_WORKLOADS["ag_small"].with_(M=16, K=8, Ns=4, P=2)
    a, ww = ri.generate_ag_gemm(w)
    assert np.array_equal(a.reshape(-1), ri.normal_bf16_numpy(w.seed, 0, w.n_a))
    assert np.array_equal(ww.reshape(-1), ri.normal_bf16_numpy(w.seed, w.n_a, w.n_w, w.wmul))
