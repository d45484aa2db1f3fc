"""fp64 CPU oracle for the AllGather + GEMM step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may use
it; the GPU library never does.

What the step computes (mKernel pages: dataforcee / chathome "five fused kernels" table,
AllGather+GEMM row -- every rank holds a shard of A; while the ranks gather the peers'
shards the local GEMM consumes tiles as they arrive; pwwt.cn analysis §2.6 -- 128-row
chunks, local inputs first): rank r's output is the product of the all-gathered A with
rank r's weight slice,

    G   = concat(A_0, A_1, ..., A_{P-1})      (the all-gather, shards in rank order)
    C_r = G @ W_r^T                           (W_r is [Ns][K], K-major)

in fp64 from the bf16 input values.  The order in which a rank receives the shards does
not change C_r; the definition is written with the gather explicit.  The matrix product is
numpy's float64 matmul, a library primitive used as one step.

Parity status: pinned (tests/test_oracle_ag_gemm.py): 40-digit Decimal brute force on
small shapes, identity-weight and single-nonzero closed forms, row locality and
linearity, and a mutation check that plausible mistakes are caught.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def all_gather(a_shards) -> np.ndarray:
    """The gathered A: the shards concatenated in rank order."""
    return np.concatenate(list(a_shards), axis=0)


def ag_gemm(a_bits: np.ndarray, w_bits: np.ndarray, P: int, rows=None) -> np.ndarray:
    """C[r] = gather(A) @ W_r^T in fp64.

    a_bits: [M][K] bf16 bits, rank j's shard = rows [j*M/P, (j+1)*M/P).
    w_bits: [P][Ns][K] bf16 bits.
    rows:   optional indices of gathered-A rows to compute (the same for every rank).
    Returns [P][M or len(rows)][Ns] float64.
    """
    a = bf16_to_f64(a_bits)
    M, K = a.shape
    if M % P != 0:
        raise ValueError("M must be a multiple of P")
    Ms = M // P
    w = bf16_to_f64(w_bits)
    if w.shape[0] != P or w.shape[2] != K:
        raise ValueError("W must be [P][Ns][K]")
    g = all_gather(a[j * Ms:(j + 1) * Ms] for j in range(P))
    if rows is not None:
        g = g[np.asarray(rows, dtype=np.int64)]
    return np.stack([g @ w[r].T for r in range(P)])


def for_workload(wl, a_bits, w_bits, rows=None) -> np.ndarray:
    return ag_gemm(a_bits, w_bits, wl.P, rows=rows)
