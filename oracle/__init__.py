"""fp64 CPU oracle for the Ring Attention forward step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The GPU library never does: the two share no
code, and the product path fails loudly instead of falling back to this.

``oracle.c`` computes softmax(scale * Q K^T [+ causal mask]) V and the per-row
natural-log LSE directly from the definition, in fp64, from the bf16 input
bytes.  The pages describe Ring Attention only as "each step rotates a KV chunk
while the local FlashAttention consumes the chunk received before"
(dataforcee / chathome kernel tables, Ring Attention row; pwwt.cn analysis,
Table 3); the definition of attention and the LSE-exact chunk merge are the
plain mathematics that step reaches.

Parity status of each function (pins in tests/test_oracle_pins.py):
  attn_fwd          pinned: Decimal brute force, Q=0 and single-key closed
                    forms, causal prefix, GQA reduction, LSE/convexity bounds,
                    key permutation and key duplication invariants.
  attn_fwd_chunked  pinned: equals attn_fwd for every P dividing S and for
                    random chunk orders (the merge identity).
  causal=2          (load-balanced shards: shard r holds half-chunks r and
                    2P-1-r) pinned: Decimal brute force over positions built
                    from the half-chunk list, equality with the contiguous
                    causal result on the same sequence re-ordered, P = 1
                    reduces bit for bit to causal=1, chunked merge identity.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
_lib = None
_lock = threading.Lock()


class OracleShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("S", ctypes.c_int),
                ("P", ctypes.c_int), ("d", ctypes.c_int), ("causal", ctypes.c_int), ("scale", ctypes.c_double)]


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (plain -O2, no fast-math, no machine flags)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            vp = ctypes.c_void_p
            lib.oracle_attn_fwd.argtypes = [ctypes.POINTER(OracleShape), vp, vp, vp, vp, ctypes.c_int64, vp, vp,
                                            ctypes.c_int]
            lib.oracle_attn_fwd.restype = ctypes.c_int
            lib.oracle_attn_fwd_chunked.argtypes = [ctypes.POINTER(OracleShape), vp, vp, vp, vp, ctypes.c_int64,
                                                    vp, vp, vp, ctypes.c_int]
            lib.oracle_attn_fwd_chunked.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _prep(q, k, v, B, Hq, Hkv, S, P, d, causal, scale, rows):
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    if q.size != B * Hq * S * d or k.size != B * Hkv * S * d or v.size != B * Hkv * S * d:
        raise ValueError("oracle: tensor sizes do not match the shape")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    causal = int(causal)  # 0, 1, or 2 = causal over load-balanced shards
    if causal not in (0, 1, 2):
        raise ValueError("oracle: causal must be 0, 1 or 2")
    sh = OracleShape(B, Hq, Hkv, S, P, d, causal, float(scale))
    if rows is None:
        n = B * Hq * S
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.size
    return q, k, v, sh, rows_arr, n


def attn_fwd(q, k, v, *, B, Hq, Hkv, S, d, causal, P=1, scale=None, rows=None, n_threads=None):
    """fp64 attention from the definition.  q,k,v: uint16 bf16 bit patterns.

    Returns (o [n_rows][d] float64, lse [n_rows] float64); rows=None means all
    rows in [B][Hq][S] order.
    """
    q, k, v, sh, rows_arr, n = _prep(q, k, v, B, Hq, Hkv, S, P, d, causal, scale, rows)
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    rc = _load().oracle_attn_fwd(ctypes.byref(sh), q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                 None if rows_arr is None else rows_arr.ctypes.data, n, o.ctypes.data,
                                 lse.ctypes.data, int(n_threads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_attn_fwd rejected its arguments")
    return o, lse


def attn_fwd_chunked(q, k, v, *, B, Hq, Hkv, S, P, d, causal, scale=None, rows=None, perm=None, n_threads=None):
    """fp64 ring-chunked attention with the exact LSE merge (see oracle.c)."""
    q, k, v, sh, rows_arr, n = _prep(q, k, v, B, Hq, Hkv, S, P, d, causal, scale, rows)
    perm_arr = None if perm is None else np.ascontiguousarray(perm, dtype=np.int32)
    o = np.empty((n, d), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    rc = _load().oracle_attn_fwd_chunked(ctypes.byref(sh), q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                         None if rows_arr is None else rows_arr.ctypes.data, n,
                                         None if perm_arr is None else perm_arr.ctypes.data, o.ctypes.data,
                                         lse.ctypes.data, int(n_threads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_chunked rejected its arguments")
    return o, lse


def for_workload(w, q, k, v, rows=None, n_threads=None):
    """Run attn_fwd on a ring_inputs.Workload's tensors."""
    return attn_fwd(q, k, v, B=w.B, Hq=w.Hq, Hkv=w.Hkv, S=w.S, P=w.P, d=w.d, causal=w.causal, scale=w.scale,
                    rows=rows, n_threads=n_threads)
