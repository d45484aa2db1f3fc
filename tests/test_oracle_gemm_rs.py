"""Pins of the GEMM + ReduceScatter oracle (oracle/gemm_rs.py) against things other than
itself: 40-digit Decimal brute force, closed forms (one rank, one nonzero), additivity over
ranks, invariance under relabelling the ranks, and mutants of plausible mistakes that each
of these must catch."""
from decimal import Decimal, getcontext

import numpy as np
import pytest

import ring_inputs as ri
from oracle import gemm_rs as og


def _bits(rng, shape, scale=1.0):
    return ri.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def brute_force(a_bits, w_bits):
    """out[m, n] = sum_r sum_k A_r[m, k] * W_r[n, k] in 40-digit decimal, straight from the
    definition of the reduced partial products."""
    getcontext().prec = 40
    a = ri.bf16_bits_to_f64(a_bits)
    w = ri.bf16_bits_to_f64(w_bits)
    P, M, Ks = a.shape
    out = np.zeros((M, w.shape[1]))
    for m in range(M):
        for n in range(w.shape[1]):
            s = sum(Decimal(float(a[r, m, k])) * Decimal(float(w[r, n, k])) for r in range(P) for k in range(Ks))
            out[m, n] = float(s)
    return out


def pin_brute_force(impl):
    rng = np.random.default_rng(1)
    for (P, M, N, Ks) in ((2, 4, 3, 5), (3, 6, 2, 4), (1, 3, 4, 7), (2, 4, 4, 4)):
        a, w = _bits(rng, (P, M, Ks)), _bits(rng, (P, N, Ks))
        if not np.allclose(impl(a, w), brute_force(a, w), rtol=1e-13, atol=1e-13):
            return False
    return True


def pin_single_rank_identity(impl):
    # P = 1 and W = identity: out = A exactly
    rng = np.random.default_rng(2)
    a = _bits(rng, (1, 6, 5))
    eye = ri.f32_to_bf16_bits(np.eye(5, dtype=np.float32)).reshape(1, 5, 5)
    return np.array_equal(impl(a, eye), ri.bf16_bits_to_f64(a[0]))


def pin_one_hot(impl):
    # a single nonzero a at A_r[m, k]: out[m, :] = a * W_r[:, k], every other row 0
    rng = np.random.default_rng(3)
    P, M, N, Ks = 3, 6, 4, 5
    w = _bits(rng, (P, N, Ks))
    for r, m, k in ((0, 0, 0), (2, M - 1, Ks - 1), (1, 3, 2)):
        a = np.zeros((P, M, Ks), dtype=np.uint16)
        a[r, m, k] = ri.f32_to_bf16_bits(np.array([1.5], dtype=np.float32))[0]
        want = np.zeros((M, N))
        want[m] = 1.5 * ri.bf16_bits_to_f64(w[r, :, k])
        if not np.array_equal(impl(a, w), want):
            return False
    return True


def pin_additive_over_ranks(impl):
    # the reduction is a sum: zeroing every rank but r leaves rank r's partial, and the
    # per-rank results add up to the full one
    rng = np.random.default_rng(4)
    P, M, N, Ks = 3, 6, 3, 4
    a, w = _bits(rng, (P, M, Ks)), _bits(rng, (P, N, Ks))
    full = impl(a, w)
    total = np.zeros_like(full)
    for r in range(P):
        ar = np.zeros_like(a)
        ar[r] = a[r]
        one = impl(ar, w)
        if not np.allclose(one, ri.bf16_bits_to_f64(a[r]) @ ri.bf16_bits_to_f64(w[r]).T, rtol=1e-14, atol=1e-14):
            return False
        total += one
    return np.allclose(total, full, rtol=1e-13, atol=1e-13)


def pin_rank_relabelling(impl):
    # which rank holds which K-shard does not matter, as long as A_r and W_r move together
    rng = np.random.default_rng(5)
    P, M, N, Ks = 4, 8, 3, 5
    a, w = _bits(rng, (P, M, Ks)), _bits(rng, (P, N, Ks))
    perm = np.array([2, 0, 3, 1])
    return np.allclose(impl(a[perm], w[perm]), impl(a, w), rtol=1e-13, atol=1e-13)


PINS = [pin_brute_force, pin_single_rank_identity, pin_one_hot, pin_additive_over_ranks, pin_rank_relabelling]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_passes_pin(pin):
    assert pin(og.gemm_rs)


# plausible mistakes: every one must fail at least one pin
def _mut_own_rank_only(a, w):          # each owner keeps only its own partial (no reduction)
    parts = og.partials(a, w)
    P, M = parts.shape[0], parts.shape[1]
    Mq = M // P
    return np.concatenate([parts[q, q * Mq:(q + 1) * Mq] for q in range(P)])


def _mut_wrong_rank_weight(a, w):      # rank r uses rank (r+1)'s weights
    return og.gemm_rs(a, np.roll(w, -1, axis=0))


def _mut_reversed_blocks(a, w):        # owners' blocks assembled in reverse rank order
    P = a.shape[0]
    return np.concatenate(og.reduce_scatter(og.partials(a, w), P)[::-1])


def _mut_fp32_partials(a, w):          # partials accumulated in fp32: caught by the 1e-13 brute force
    af = og.bf16_to_f64(a).astype(np.float32)
    wf = og.bf16_to_f64(w).astype(np.float32)
    return sum((af[r] @ wf[r].T).astype(np.float64) for r in range(a.shape[0]))


def _mut_drop_last_rank(a, w):         # the last rank's partial never arrives
    return og.partials(a, w)[:-1].sum(axis=0) if a.shape[0] > 1 else og.partials(a, w)[0] * 0


def _mut_transposed_w(a, w):           # W read as [Ks][N] instead of [N][Ks] (only where square)
    if w.shape[1] != w.shape[2]:
        return og.gemm_rs(a, w)
    return og.gemm_rs(a, np.ascontiguousarray(np.transpose(w, (0, 2, 1))))


@pytest.mark.parametrize("mutant", [_mut_own_rank_only, _mut_wrong_rank_weight, _mut_reversed_blocks,
                                     _mut_fp32_partials, _mut_drop_last_rank, _mut_transposed_w],
                         ids=lambda f: f.__name__)
def test_pins_catch_mutant(mutant):
    assert not all(pin(mutant) for pin in PINS)


def test_rows_option_matches_full():
    w = ri.RS_WORKLOADS["rs_small"].with_(M=64, N=32, Ks=16, P=4)
    a, ww = ri.generate_gemm_rs(w)
    full = og.for_workload(w, a, ww)
    rows = ri.rs_sample_rows(w, n_random=20)
    assert np.array_equal(og.for_workload(w, a, ww, rows=rows), full[rows])


def test_rs_inputs_share_the_seeded_stream():
    w = ri.RS_WORKLOADS["rs_small"].with_(M=16, N=8, Ks=8, P=2)
    a, ww = ri.generate_gemm_rs(w)
    assert np.array_equal(a.reshape(-1), ri.normal_bf16_numpy(w.seed, 0, w.n_a))
    assert np.array_equal(ww.reshape(-1), ri.normal_bf16_numpy(w.seed, w.n_a, w.n_w, w.wmul))
