"""fp64 CPU oracle for the GEMM + ReduceScatter step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may use
it; the GPU library never does.

What the step computes (mKernel pages: dataforcee / chathome "five fused kernels" table,
GEMM + ReduceScatter row -- the ranks compute C = A @ B and reduce-scatter the output, each
output tile reduced and forwarded to its owner as soon as it is produced; pwwt.cn analysis
§2.6 Table 3 -- tensor parallel, compute feeds communication): rank r holds the K-shard A_r
([M][Ks]) of the activations and W_r ([N][Ks], K-major) of the weights,

    C_r = A_r @ W_r^T                              (rank r's partial product, [M][N])
    S   = C_0 + C_1 + ... + C_{P-1}                (the reduction)
    out_q = S[q*M/P : (q+1)*M/P]                   (the scatter: rank q keeps its row block)

in fp64 from the bf16 input values; the returned array is the owners' blocks in rank
order, i.e. S itself.  Neither the order in which partials arrive nor the tiling changes
the result; the definition is written with the three steps explicit.  The matrix product is
numpy's float64 matmul, a library primitive used as one step.

Parity status: pinned (tests/test_oracle_gemm_rs.py): 40-digit Decimal brute force on
small shapes, the single-rank and one-hot closed forms, additivity over ranks and
invariance under relabelling the ranks, and a mutation check that plausible mistakes are
caught.
"""
from __future__ import annotations

import numpy as np

from .ag_gemm import bf16_to_f64


def partials(a_bits: np.ndarray, w_bits: np.ndarray, rows=None) -> np.ndarray:
    """C_r = A_r @ W_r^T for every rank r (optionally only the given output rows)."""
    a = bf16_to_f64(a_bits)
    w = bf16_to_f64(w_bits)
    P, M, Ks = a.shape
    if w.shape[0] != P or w.shape[2] != Ks:
        raise ValueError("W must be [P][N][Ks] with A [P][M][Ks]")
    if rows is not None:
        a = a[:, np.asarray(rows, dtype=np.int64)]
    return np.stack([a[r] @ w[r].T for r in range(P)])


def reduce_scatter(parts: np.ndarray, P: int) -> list:
    """Sum the ranks' partials and give rank q its row block [q*M/P, (q+1)*M/P)."""
    s = parts.sum(axis=0)
    M = s.shape[0]
    if M % P != 0:
        raise ValueError("M must be a multiple of P")
    Mq = M // P
    return [s[q * Mq:(q + 1) * Mq] for q in range(P)]


def gemm_rs(a_bits: np.ndarray, w_bits: np.ndarray, rows=None) -> np.ndarray:
    """The owners' output blocks in rank order ([M][N] float64), or only the given rows."""
    P = a_bits.shape[0]
    parts = partials(a_bits, w_bits, rows=rows)
    if rows is not None:  # a row sample spans owners: the reduction alone, per sampled row
        return parts.sum(axis=0)
    return np.concatenate(reduce_scatter(parts, P), axis=0)


def for_workload(wl, a_bits, w_bits, rows=None) -> np.ndarray:
    return gemm_rs(a_bits, w_bits, rows=rows)
