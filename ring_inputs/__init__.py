"""Seeded synthetic inputs for the ring-attention workloads (no attention math).

The generator itself lives in ``gen.c`` (SplitMix64 counter stream followed by
Box-Muller, rounded to bf16 with round-to-nearest-even); this module builds it
with gcc, loads it with ctypes, and describes the workloads:

* the shapes of the five workloads in the mKernel pages' Ring Attention setting
  (sequence-parallel attention over P shards; arxivdaily abstract and the
  pwwt.cn analysis, Table 3 "Ring Attention" row),
* the element order (Q, then K, then V, each in [B][H][S][d] order),
* the power-of-two multipliers (x2 for the sharper-softmax GQA workload, x8 for
  the 1 % outlier K rows of the long-sequence workload),
* the fixed row samples used where the oracle cannot compute every row.

Both the fp64 oracle and the GPU library consume the bytes produced here and
nothing else is shared between them.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "_gen.so")
_lib = None
_lock = threading.Lock()

GAMMA = 0x9E3779B97F4A7C15
OUTLIER_STREAM = 0x5EED0000  # added to the seed to draw the outlier-row mask


def build(force: bool = False) -> str:
    """Compile gen.c into _gen.so (gcc, no machine-specific flags)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
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
            lib.ri_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_float,
                                           ctypes.c_void_p, ctypes.c_int]
            lib.ri_normal_bf16.restype = ctypes.c_int
            lib.ri_splitmix64.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.ri_splitmix64.restype = ctypes.c_uint64
            lib.ri_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.ri_uniform.restype = ctypes.c_double
            _lib = lib
    return _lib


def n_threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


# ----------------------------------------------------------------------------------------------
# Low-level stream access
# ----------------------------------------------------------------------------------------------

def splitmix64(seed: int, n: int) -> int:
    return int(_load().ri_splitmix64(seed & (2**64 - 1), n))


def normal_bf16_into(addr: int, seed: int, first: int, count: int, mult: float = 1.0) -> None:
    """Write `count` bf16 bit patterns (uint16) of stream elements [first, first+count) to `addr`."""
    rc = _load().ri_normal_bf16(seed & (2**64 - 1), first, count, float(mult), ctypes.c_void_p(addr), n_threads())
    if rc != 0:
        raise RuntimeError("ri_normal_bf16 failed")


def normal_bf16(seed: int, first: int, count: int, mult: float = 1.0) -> np.ndarray:
    out = np.empty(count, dtype=np.uint16)
    if count:
        normal_bf16_into(out.ctypes.data, seed, first, count, mult)
    return out


def normal_bf16_numpy(seed: int, first: int, count: int, mult: float = 1.0) -> np.ndarray:
    """Slow pure-numpy restatement of the same stream (used to cross-check gen.c)."""
    n = np.arange(first, first + count, dtype=np.uint64)
    p = n >> np.uint64(1)

    def mix(idx):
        with np.errstate(over="ignore"):
            z = np.uint64(seed) + (idx + np.uint64(1)) * np.uint64(GAMMA)
            z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
            z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))

    x1 = mix(np.uint64(2) * p)
    x2 = mix(np.uint64(2) * p + np.uint64(1))
    u1 = ((x1 >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * 2.0**-53
    u2 = (x2 >> np.uint64(11)).astype(np.float64) * 2.0**-53
    r = np.sqrt(-2.0 * np.log(u1))
    th = 2.0 * np.pi * u2
    val = np.where((n & np.uint64(1)) == 1, r * np.sin(th), r * np.cos(th)).astype(np.float32)
    b = f32_to_bf16_bits(val)
    if mult != 1.0:
        b = f32_to_bf16_bits(bf16_bits_to_f32(b) * np.float32(mult))
    return b


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(b).astype(np.float64)


# ----------------------------------------------------------------------------------------------
# Workloads
# ----------------------------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    P: int
    d: int
    causal: int      # 0, 1, or 2 = causal over load-balanced shards
    seed: int
    qmul: float = 1.0
    kmul: float = 1.0
    vmul: float = 1.0
    outlier_frac: float = 0.0   # fraction of K rows multiplied by outlier_mul
    outlier_mul: float = 8.0

    @property
    def L(self) -> int:
        return self.S // self.P

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    @property
    def n_q(self) -> int:
        return self.B * self.Hq * self.S * self.d

    @property
    def n_kv(self) -> int:
        return self.B * self.Hkv * self.S * self.d

    def flops(self) -> float:
        """Algorithmic flops: 4*d per unmasked (query, key) pair, times B*Hq."""
        pairs = self.S * (self.S + 1) // 2 if self.causal else self.S * self.S
        return 4.0 * self.d * pairs * self.B * self.Hq

    def staging_transfers(self) -> int:
        """(shard, chunk) transfers the ring performs: the local chunk is never moved."""
        return self.P * (self.P - 1) // 2 if self.causal == 1 else self.P * (self.P - 1)

    def staging_bytes(self) -> int:
        """Bytes written into ring slots (K and V); the same amount is read from home.  Over
        load-balanced shards half of the transfers (chunks below the shard) move half a chunk."""
        rows = self.staging_transfers() * self.L
        if self.causal == 2:
            rows -= self.P * (self.P - 1) // 2 * (self.L // 2)
        return rows * 2 * self.d * 2 * self.B * self.Hkv

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _cfg5(d: int, P: int) -> Workload:
    return Workload(f"sweep_d{d}_P{P}", 1, 16, 16, 16384, P, d, False, seed=500 + d)


WORKLOADS = {
    # B1 H2 S1024 P4 d64, non-causal: the small case the oracle computes in full
    "small": Workload("small", 1, 2, 2, 1024, 4, 64, False, seed=1),
    # B1 H32 S32768 P16 d128, non-causal and causal: the headline throughput case
    "h32_s32k_nc": Workload("h32_s32k_nc", 1, 32, 32, 32768, 16, 128, False, seed=2),
    "h32_s32k_c": Workload("h32_s32k_c", 1, 32, 32, 32768, 16, 128, True, seed=2),
    # the same causal pass over load-balanced shards (shard r holds half-chunks r and 2P-1-r)
    "h32_s32k_cb": Workload("h32_s32k_cb", 1, 32, 32, 32768, 16, 128, 2, seed=2),
    # GQA, causal, B2 Hq32 Hkv8 S65536 P16 d128, Q and K x2
    "gqa_s64k_c": Workload("gqa_s64k_c", 2, 32, 8, 65536, 16, 128, True, seed=3, qmul=2.0, kmul=2.0),
    # long sequence, causal, B1 H8 S131072 P32 d128, 1 % of K rows x8
    "long_s128k_c": Workload("long_s128k_c", 1, 8, 8, 131072, 32, 128, True, seed=4, outlier_frac=0.01),
}
for _d in (64, 128):
    for _P in (2, 4, 8, 16, 32, 64):
        WORKLOADS[f"sweep_d{_d}_P{_P}"] = _cfg5(_d, _P)


def outlier_rows(w: Workload) -> np.ndarray:
    """Boolean mask [B][Hkv][S]: K rows multiplied by w.outlier_mul (drawn from a separate stream)."""
    n = w.B * w.Hkv * w.S
    if w.outlier_frac <= 0:
        return np.zeros(n, dtype=bool).reshape(w.B, w.Hkv, w.S)
    seed = (w.seed + OUTLIER_STREAM) & (2**64 - 1)
    idx = np.arange(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + (idx + np.uint64(1)) * np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    z = z ^ (z >> np.uint64(31))
    u = (z >> np.uint64(11)).astype(np.float64) * 2.0**-53
    return (u < w.outlier_frac).reshape(w.B, w.Hkv, w.S)


def generate(w: Workload, q_addr: int | None = None, k_addr: int | None = None, v_addr: int | None = None):
    """Produce Q, K, V as uint16 bf16 bit patterns in [B][H][S][d] order.

    If addresses are given (e.g. pinned host buffers), the values are written
    there and None is returned for that tensor; otherwise numpy arrays are made.
    """
    out = []
    first = 0
    for name, count, mult, addr, shape in (
        ("q", w.n_q, w.qmul, q_addr, (w.B, w.Hq, w.S, w.d)),
        ("k", w.n_kv, w.kmul, k_addr, (w.B, w.Hkv, w.S, w.d)),
        ("v", w.n_kv, w.vmul, v_addr, (w.B, w.Hkv, w.S, w.d)),
    ):
        if addr is None:
            arr = normal_bf16(w.seed, first, count, mult).reshape(shape)
            out.append(arr)
            addr_used = arr.ctypes.data
        else:
            normal_bf16_into(addr, w.seed, first, count, mult)
            out.append(None)
            addr_used = addr
        if name == "k" and w.outlier_frac > 0:
            mask = outlier_rows(w).reshape(-1)
            kview = np.ctypeslib.as_array(ctypes.cast(addr_used, ctypes.POINTER(ctypes.c_uint16)), shape=(count,))
            kview = kview.reshape(-1, w.d)
            rows = np.nonzero(mask)[0]
            kview[rows] = f32_to_bf16_bits(bf16_bits_to_f32(kview[rows]) * np.float32(w.outlier_mul))
        first += count
    return tuple(out)


def sample_rows(w: Workload, n_random: int = 4096) -> np.ndarray:
    """Fixed row sample: flat row ids ((b*Hq + hq)*S + i), sorted and unique.

    For every (b, hq): rows 0, 1, 127, 128, each shard's first and last row (and, over
    load-balanced shards, the two rows at its half boundary) and S-1; then uniformly
    drawn rows (seeded) until at least `n_random` rows in total.
    """
    base = {0, 1, 127, 128, w.S - 1}
    for r in range(w.P):
        base.add(r * w.L)
        base.add((r + 1) * w.L - 1)
        if w.causal == 2:  # load-balanced shards: the rows on either side of the half boundary
            base.add(r * w.L + w.L // 2 - 1)
            base.add(r * w.L + w.L // 2)
    base = sorted(i for i in base if 0 <= i < w.S)
    ids = []
    for bh in range(w.B * w.Hq):
        ids.extend(bh * w.S + i for i in base)
    ids = set(ids)
    seed = (w.seed * 7919 + 17) & (2**64 - 1)
    n = 0
    total = w.B * w.Hq * w.S
    while len(ids) < n_random:
        ids.add(splitmix64(seed, n) % total)
        n += 1
    return np.array(sorted(ids), dtype=np.int64)


# ----------------------------------------------------------------------------------------------
# AllGather + GEMM (tensor-parallel linear layer) workloads
# ----------------------------------------------------------------------------------------------
# The mKernel pages' AllGather+GEMM kernel (dataforcee / chathome "five fused kernels" table,
# AllGather+GEMM row; pwwt.cn analysis §2.6): every rank holds a row shard of A, gathers the
# other ranks' shards, and its local GEMM consumes A tiles as they arrive.  Emulated on one
# GPU: P ranks, rank r owns rows [r*M/P, (r+1)*M/P) of A and the weight slice W_r
# ([Ns][K], K-major), and produces C_r = gather(A) @ W_r^T ([M][Ns]).

@dataclasses.dataclass(frozen=True)
class AgGemmWorkload:
    name: str
    M: int      # rows of the gathered A (tokens)
    K: int      # contraction (hidden size)
    Ns: int     # output columns per rank (N / P)
    P: int      # ranks
    seed: int
    amul: float = 1.0
    wmul: float = 1.0 / 64.0   # power of two: exact in bf16; keeps |C| near 1 for K ~ 4096

    @property
    def Ms(self) -> int:
        return self.M // self.P

    @property
    def n_a(self) -> int:
        return self.M * self.K

    @property
    def n_w(self) -> int:
        return self.P * self.Ns * self.K

    def flops(self) -> float:
        """2*M*K*Ns per rank, times P."""
        return 2.0 * self.M * self.K * self.Ns * self.P

    def gather_bytes(self) -> int:
        """A bytes copied by the emulated all-gather: every rank receives the P-1 other shards."""
        return self.P * (self.P - 1) * self.Ms * self.K * 2

    def with_(self, **kw) -> "AgGemmWorkload":
        return dataclasses.replace(self, **kw)


AG_WORKLOADS = {
    # small: every output element is checked against the oracle
    "ag_small": AgGemmWorkload("ag_small", 1024, 512, 256, 4, seed=700),
    # a tensor-parallel MLP up-projection: 8192 tokens, hidden 8192, N = 28672 over 8 ranks
    "ag_m8k_k8k_n28k_p8": AgGemmWorkload("ag_m8k_k8k_n28k_p8", 8192, 8192, 3584, 8, seed=701),
}


def generate_ag_gemm(w: AgGemmWorkload, a_addr: int | None = None, w_addr: int | None = None):
    """A ([M][K]) then W ([P][Ns][K]) as uint16 bf16 bit patterns, from the same stream as the
    attention inputs (A first).  With addresses, values are written there and None returned."""
    out = []
    first = 0
    for count, mult, addr, shape in ((w.n_a, w.amul, a_addr, (w.M, w.K)), (w.n_w, w.wmul, w_addr, (w.P, w.Ns, w.K))):
        if addr is None:
            out.append(normal_bf16(w.seed, first, count, mult).reshape(shape))
        else:
            normal_bf16_into(addr, w.seed, first, count, mult)
            out.append(None)
        first += count
    return tuple(out)


def ag_sample_rows(w: AgGemmWorkload, n_random: int = 1024) -> np.ndarray:
    """Fixed sample of row indices of the gathered A (the same rows for every rank): each
    shard's first, second and last rows, then seeded uniform rows up to `n_random`."""
    ids = set()
    for j in range(w.P):
        ids.update((j * w.Ms, j * w.Ms + 1, (j + 1) * w.Ms - 1))
    seed = (w.seed * 7919 + 23) & (2**64 - 1)
    n = 0
    while len(ids) < n_random:
        ids.add(splitmix64(seed, n) % w.M)
        n += 1
    return np.array(sorted(ids), dtype=np.int64)


# ----------------------------------------------------------------------------------------------
# GEMM + ReduceScatter (tensor-parallel row-parallel linear layer) workloads
# ----------------------------------------------------------------------------------------------
# P ranks; rank r holds its K-shard A_r ([M][Ks]) of the activations and W_r ([N][Ks], K-major)
# of the weights; the output rows [q*M/P, (q+1)*M/P) of sum_r A_r @ W_r^T belong to rank q.

@dataclasses.dataclass(frozen=True)
class GemmRsWorkload:
    name: str
    M: int      # output rows (tokens)
    N: int      # output columns (hidden size)
    Ks: int     # contraction per rank (K / P)
    P: int      # ranks
    seed: int
    amul: float = 1.0
    wmul: float = 1.0 / 64.0   # power of two: exact in bf16; keeps |out| near 1 for K ~ 4096

    @property
    def Mq(self) -> int:
        return self.M // self.P

    @property
    def n_a(self) -> int:
        return self.P * self.M * self.Ks

    @property
    def n_w(self) -> int:
        return self.P * self.N * self.Ks

    def flops(self) -> float:
        """2*M*N*Ks per rank, times P."""
        return 2.0 * self.M * self.N * self.Ks * self.P

    def reduce_bytes(self) -> int:
        """fp32 partial bytes the emulated reduce-scatter reads: every rank's [M][N] partial."""
        return self.P * self.M * self.N * 4

    def with_(self, **kw) -> "GemmRsWorkload":
        return dataclasses.replace(self, **kw)


RS_WORKLOADS = {
    # small: every output element is checked against the oracle
    "rs_small": GemmRsWorkload("rs_small", 1024, 512, 256, 4, seed=800),
    # a tensor-parallel MLP down-projection: 8192 tokens, hidden 8192, K = 28672 over 8 ranks
    "rs_m8k_n8k_k28k_p8": GemmRsWorkload("rs_m8k_n8k_k28k_p8", 8192, 8192, 3584, 8, seed=801),
}


def generate_gemm_rs(w: GemmRsWorkload, a_addr: int | None = None, w_addr: int | None = None):
    """A ([P][M][Ks]) then W ([P][N][Ks]) as uint16 bf16 bit patterns, from the same stream as
    the other inputs (A first).  With addresses, values are written there and None returned."""
    out = []
    first = 0
    for count, mult, addr, shape in ((w.n_a, w.amul, a_addr, (w.P, w.M, w.Ks)),
                                     (w.n_w, w.wmul, w_addr, (w.P, w.N, w.Ks))):
        if addr is None:
            out.append(normal_bf16(w.seed, first, count, mult).reshape(shape))
        else:
            normal_bf16_into(addr, w.seed, first, count, mult)
            out.append(None)
        first += count
    return tuple(out)


def rs_sample_rows(w: GemmRsWorkload, n_random: int = 1024) -> np.ndarray:
    """Fixed sample of output rows: each owner's first, second and last rows, then seeded
    uniform rows up to `n_random`."""
    ids = set()
    for q in range(w.P):
        ids.update((q * w.Mq, q * w.Mq + 1, (q + 1) * w.Mq - 1))
    seed = (w.seed * 7919 + 29) & (2**64 - 1)
    n = 0
    while len(ids) < n_random:
        ids.add(splitmix64(seed, n) % w.M)
        n += 1
    return np.array(sorted(ids), dtype=np.int64)


def generate_dout(w: Workload) -> np.ndarray:
    """The upstream gradient dO ([B][Hq][S][d] bf16 bits) of an attention workload: the next
    elements of the workload's seeded stream, after Q, K and V."""
    return normal_bf16(w.seed, w.n_q + 2 * w.n_kv, w.n_q).reshape(w.B, w.Hq, w.S, w.d)
