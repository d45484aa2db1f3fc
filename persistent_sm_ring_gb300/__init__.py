"""persistent_sm_ring_gb300: Ring Attention forward on one GB300 (sm_103a).

Thin Python binding over the C ABI of ``libpsr.so`` (declared in
``include/psr.h``).  It only marshals arguments: every step of the ring
(staging, readiness flags, the tcgen05 FlashAttention pass, the LSE-exact
merge, the on-GPU partition controller) runs in the library's CUDA kernel.
PyTorch supplies device memory and streams.  There is no fallback: if the
library is missing or the device is not an sm_103 GPU, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB, LIB_PAIRS, LIB_TRACE, build as _build

__all__ = ["build", "load", "Shape", "AgShape", "RsShape", "Partition", "Stats", "ring_attn_fwd", "ring_attn_fwd_host",
           "workspace_bytes", "ag_gemm", "ag_gemm_workspace_bytes", "gemm_rs", "gemm_rs_workspace_bytes",
           "ring_attn_bwd", "ring_attn_bwd_workspace_bytes",
           "get_stats", "get_trajectory", "controller_target", "num_ctas", "status_string", "PsrError",
           "STATIC", "ADAPTIVE", "FAULT_NONE", "FAULT_DROP_FIRST_FLAG", "FAULT_SLOW_STAGING", "CAUSAL",
           "CAUSAL_BALANCED"]

OK, ERR_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4
STATIC, ADAPTIVE = 0, 1
FAULT_NONE, FAULT_DROP_FIRST_FLAG, FAULT_SLOW_STAGING = 0, 1, 2
CAUSAL, CAUSAL_BALANCED = 1, 2

EXPORTED = ("psr_workspace_bytes", "psr_ring_attn_fwd", "psr_ring_attn_fwd_host", "psr_get_stats",
            "psr_get_trajectory", "psr_controller_target", "psr_status_string", "psr_num_ctas",
            "psr_ring_attn_fwd_noalloc", "psr_noalloc_get_stats", "psr_ag_gemm_workspace_bytes", "psr_ag_gemm", "psr_gemm_rs_workspace_bytes",
            "psr_gemm_rs", "psr_ring_attn_bwd_workspace_bytes", "psr_ring_attn_bwd")


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("S", ctypes.c_int),
                ("P", ctypes.c_int), ("d", ctypes.c_int), ("causal", ctypes.c_int), ("scale", ctypes.c_float)]


class AgShape(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int), ("K", ctypes.c_int), ("Ns", ctypes.c_int), ("P", ctypes.c_int)]


class RsShape(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int), ("N", ctypes.c_int), ("Ks", ctypes.c_int), ("P", ctypes.c_int)]


class Partition(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("n_staging", ctypes.c_int), ("n_min", ctypes.c_int),
                ("n_max", ctypes.c_int), ("fault", ctypes.c_int), ("timeout_ms", ctypes.c_int)]


class Stats(ctypes.Structure):
    _fields_ = [("status", ctypes.c_int), ("error_site", ctypes.c_int), ("n_cta", ctypes.c_int),
                ("n_s_initial", ctypes.c_int), ("n_s_final", ctypes.c_int), ("n_s_min", ctypes.c_int),
                ("n_s_max", ctypes.c_int), ("traj_len", ctypes.c_int),
                ("staging_cycles", ctypes.c_ulonglong), ("compute_cycles", ctypes.c_ulonglong),
                ("staging_tasks", ctypes.c_ulonglong), ("compute_items", ctypes.c_ulonglong),
                ("compute_tiles", ctypes.c_ulonglong), ("staging_bytes", ctypes.c_ulonglong),
                ("role_switches", ctypes.c_ulonglong), ("idle_polls", ctypes.c_ulonglong),
                ("trace_softmax_wait", ctypes.c_ulonglong), ("trace_softmax_busy", ctypes.c_ulonglong),
                ("trace_mma_issue", ctypes.c_ulonglong), ("trace_mma_wait_kv", ctypes.c_ulonglong),
                ("trace_producer_wait_empty", ctypes.c_ulonglong), ("trace_producer_wait_flag", ctypes.c_ulonglong)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class PsrError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib = None
_lock = threading.Lock()


def build(force: bool = False, trace: bool = False, variant: str = "") -> str:
    """Compile libpsr.so in-tree for sm_103a, or a variant: "trace" (trace=True; cycle-tracing
    libpsr_trace.so) or "pairs" (libpsr_pairs.so, CTA-pair compute units for d = 128)."""
    return _build(force=force, trace=trace, variant=variant)


def load(trace: bool = False, variant: str = "") -> ctypes.CDLL:
    """Load libpsr.so (or the variant built by build(variant=...)); raises if it has not been built
    (no fallback path exists).

    One library per process: the first call decides which."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = LIB_TRACE if (trace or variant == "trace") else (LIB_PAIRS if variant == "pairs" else LIB)
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run persistent_sm_ring_gb300.build() (nvcc, sm_103a) first")
        lib = ctypes.CDLL(path)
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        P_shape, P_part = ctypes.POINTER(Shape), ctypes.POINTER(Partition)
        lib.psr_workspace_bytes.argtypes = [P_shape]
        lib.psr_workspace_bytes.restype = sz
        lib.psr_ring_attn_fwd.argtypes = [P_shape, vp, vp, vp, vp, vp, vp, sz, P_part, vp]
        lib.psr_ring_attn_fwd.restype = ctypes.c_int
        lib.psr_ring_attn_fwd_host.argtypes = [P_shape, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, P_part, vp]
        lib.psr_ring_attn_fwd_host.restype = ctypes.c_int
        lib.psr_get_stats.argtypes = [vp, ctypes.POINTER(Stats), vp]
        lib.psr_get_stats.restype = ctypes.c_int
        lib.psr_get_trajectory.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, vp]
        lib.psr_get_trajectory.restype = ctypes.c_int
        lib.psr_controller_target.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                              ctypes.c_double, ctypes.c_int, ctypes.c_int]
        lib.psr_controller_target.restype = ctypes.c_int
        lib.psr_status_string.argtypes = [ctypes.c_int]
        lib.psr_status_string.restype = ctypes.c_char_p
        P_ag = ctypes.POINTER(AgShape)
        lib.psr_ag_gemm_workspace_bytes.argtypes = [P_ag]
        lib.psr_ag_gemm_workspace_bytes.restype = sz
        lib.psr_ag_gemm.argtypes = [P_ag, vp, vp, vp, vp, sz, P_part, vp]
        lib.psr_ag_gemm.restype = ctypes.c_int
        lib.psr_ring_attn_bwd_workspace_bytes.argtypes = [ctypes.POINTER(Shape)]
        lib.psr_ring_attn_bwd_workspace_bytes.restype = sz
        lib.psr_ring_attn_bwd.argtypes = [ctypes.POINTER(Shape), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                                          ctypes.c_int, vp]
        lib.psr_ring_attn_bwd.restype = ctypes.c_int
        P_rs = ctypes.POINTER(RsShape)
        lib.psr_gemm_rs_workspace_bytes.argtypes = [P_rs]
        lib.psr_gemm_rs_workspace_bytes.restype = sz
        lib.psr_gemm_rs.argtypes = [P_rs, vp, vp, vp, vp, sz, P_part, vp]
        lib.psr_gemm_rs.restype = ctypes.c_int
        lib.psr_ring_attn_fwd_noalloc.argtypes = [P_shape, vp, vp, vp, vp, vp, P_part, vp]
        lib.psr_ring_attn_fwd_noalloc.restype = ctypes.c_int
        lib.psr_noalloc_get_stats.argtypes = [ctypes.POINTER(Stats), vp]
        lib.psr_noalloc_get_stats.restype = ctypes.c_int
        lib.psr_num_ctas.argtypes = []
        lib.psr_num_ctas.restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().psr_status_string(int(status)).decode()


def make_shape(B, Hq, Hkv, S, P, d, causal, scale=None) -> Shape:
    """causal: False/0, True/1 (CAUSAL), or 2 (CAUSAL_BALANCED: load-balanced shards)."""
    return Shape(int(B), int(Hq), int(Hkv), int(S), int(P), int(d), int(causal),
                 float(scale) if scale is not None else 0.0)


def make_partition(mode=ADAPTIVE, n_staging=0, n_min=0, n_max=0, fault=FAULT_NONE, timeout_ms=0) -> Partition:
    return Partition(int(mode), int(n_staging), int(n_min), int(n_max), int(fault), int(timeout_ms))


def workspace_bytes(shape: Shape) -> int:
    n = load().psr_workspace_bytes(ctypes.byref(shape))
    if n == 0:
        raise PsrError(ERR_UNSUPPORTED, "psr_workspace_bytes")
    return int(n)


def controller_target(n_cta, R_s, C_s, R_p, C_p, n_min=1, n_max=1 << 30) -> int:
    return int(load().psr_controller_target(int(n_cta), float(R_s), float(C_s), float(R_p), float(C_p), int(n_min),
                                            int(n_max)))


def num_ctas() -> int:
    n = load().psr_num_ctas()
    if n < 0:
        raise PsrError(-n, "psr_num_ctas")
    return n


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_tensor(t, name, shape, dtype):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_host(t, name, shape, dtypes):
    import torch
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must be one of {dtypes}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _same_device(tensors, what):
    devs = {t.device for t in tensors}
    if len(devs) != 1:
        raise ValueError(f"{what}: all device tensors must be on one GPU, got {sorted(map(str, devs))}")


def ring_attn_fwd(q, k, v, *, P, causal, scale=None, partition=None, workspace=None, out=None, lse=None,
                  stream=None):
    """Ring Attention forward over P shards held on this GPU.

    q: [B, Hq, S, d] bf16; k, v: [B, Hkv, S, d] bf16 (CUDA, contiguous).
    Returns (o [B, Hq, S, d] bf16, lse [B, Hq, S] fp32, workspace).  The call is
    asynchronous on `stream`; use get_stats(workspace) to read the device
    status (timeouts) and the controller's statistics.
    """
    import torch
    lib = load()
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q, k, v must be 4-d [B, H, S, d]")
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    _check_tensor(q, "q", (B, Hq, S, d), torch.bfloat16)
    _check_tensor(k, "k", (B, Hkv, S, d), torch.bfloat16)
    _check_tensor(v, "v", (B, Hkv, S, d), torch.bfloat16)
    shape = make_shape(B, Hq, Hkv, S, P, d, causal, scale)
    need = workspace_bytes(shape)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    elif not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must be a CUDA tensor of at least {need} bytes")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_tensor(out, "out", (B, Hq, S, d), torch.bfloat16)
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    else:
        _check_tensor(lse, "lse", (B, Hq, S), torch.float32)
    _same_device((q, k, v, out, lse, workspace), "ring_attn_fwd")
    part = partition if partition is not None else make_partition()
    rc = lib.psr_ring_attn_fwd(ctypes.byref(shape), q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               lse.data_ptr(), workspace.data_ptr(), need, ctypes.byref(part),
                               _stream_handle(stream))
    if rc != OK:
        raise PsrError(rc, "psr_ring_attn_fwd")
    return out, lse, workspace


def ring_attn_fwd_host(q_host, k_host, v_host, o_host, lse_host, dq, dk, dv, d_o, d_lse, *, P, causal, scale=None,
                       partition=None, workspace=None, stream=None):
    """Host-buffer variant: copies in, runs, copies out and synchronises (one C call; large shapes
    run in slices whose copies overlap the kernels).

    q_host, o_host: [B, Hq, S, d]; k_host, v_host: [B, Hkv, S, d] -- pinned host tensors holding
    bf16 values (dtype bfloat16, or int16 carrying the bf16 bit patterns); lse_host: [B, Hq, S]
    fp32, pinned.  dq, d_o: [B, Hq, S, d] and dk, dv: [B, Hkv, S, d] bf16, d_lse: [B, Hq, S] fp32 --
    the device buffers the copies land in (CUDA, contiguous, one GPU)."""
    import torch
    lib = load()
    if not isinstance(q_host, torch.Tensor) or q_host.dim() != 4 or not isinstance(k_host, torch.Tensor) \
            or k_host.dim() != 4:
        raise ValueError("q_host, k_host, v_host must be 4-d [B, H, S, d] tensors")
    B, Hq, S, d = q_host.shape
    Hkv = k_host.shape[1]
    bits = (torch.bfloat16, torch.int16)
    _check_host(q_host, "q_host", (B, Hq, S, d), bits)
    _check_host(k_host, "k_host", (B, Hkv, S, d), bits)
    _check_host(v_host, "v_host", (B, Hkv, S, d), bits)
    _check_host(o_host, "o_host", (B, Hq, S, d), bits)
    _check_host(lse_host, "lse_host", (B, Hq, S), (torch.float32,))
    _check_tensor(dq, "dq", (B, Hq, S, d), torch.bfloat16)
    _check_tensor(dk, "dk", (B, Hkv, S, d), torch.bfloat16)
    _check_tensor(dv, "dv", (B, Hkv, S, d), torch.bfloat16)
    _check_tensor(d_o, "d_o", (B, Hq, S, d), torch.bfloat16)
    _check_tensor(d_lse, "d_lse", (B, Hq, S), torch.float32)
    _same_device((dq, dk, dv, d_o, d_lse), "ring_attn_fwd_host")
    for t, name in ((q_host, "q_host"), (k_host, "k_host"), (v_host, "v_host"), (o_host, "o_host"),
                    (lse_host, "lse_host")):
        if not t.is_pinned():
            raise ValueError(f"{name} must be in pinned host memory (tensor.pin_memory()): the copies run "
                             f"asynchronously on the library's streams")
    shape = make_shape(B, Hq, Hkv, S, P, d, causal, scale)
    need = workspace_bytes(shape)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dq.device)
    elif not workspace.is_cuda or workspace.device != dq.device or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must be a CUDA tensor on {dq.device} of at least {need} bytes")
    part = partition if partition is not None else make_partition()
    rc = lib.psr_ring_attn_fwd_host(ctypes.byref(shape), q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(),
                                    o_host.data_ptr(), lse_host.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                    dv.data_ptr(), d_o.data_ptr(), d_lse.data_ptr(), workspace.data_ptr(), need,
                                    ctypes.byref(part), _stream_handle(stream))
    if rc != OK:
        raise PsrError(rc, "psr_ring_attn_fwd_host")
    return workspace


def ag_gemm_workspace_bytes(M, K, Ns, P) -> int:
    n = load().psr_ag_gemm_workspace_bytes(ctypes.byref(AgShape(int(M), int(K), int(Ns), int(P))))
    if n == 0:
        raise PsrError(ERR_UNSUPPORTED, "psr_ag_gemm_workspace_bytes")
    return int(n)


def ag_gemm(a, w, *, P, partition=None, workspace=None, out=None, stream=None):
    """AllGather + GEMM through the C ABI: a [M][K] bf16 (rank j's shard = rows j*M/P..),
    w [P][Ns][K] bf16 -> c [P][M][Ns] bf16, C_r = gather(A) @ W_r^T.  Returns (c, workspace)."""
    import torch
    lib = load()
    if a.dim() != 2 or w.dim() != 3:
        raise ValueError("ag_gemm: a must be [M, K] and w [P, Ns, K]")
    M, K = a.shape
    Ns = w.shape[1]
    shape = AgShape(int(M), int(K), int(Ns), int(P))
    need = ag_gemm_workspace_bytes(M, K, Ns, P)
    _check_tensor(a, "a", (M, K), torch.bfloat16)
    _check_tensor(w, "w", (P, Ns, K), torch.bfloat16)
    if out is None:
        out = torch.empty((P, M, Ns), dtype=torch.bfloat16, device=a.device)
    _check_tensor(out, "out", (P, M, Ns), torch.bfloat16)
    _same_device((a, w, out), "ag_gemm")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=a.device)
    elif not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"ag_gemm: workspace must be a CUDA tensor of at least {need} bytes")
    part = partition if partition is not None else make_partition()
    rc = lib.psr_ag_gemm(ctypes.byref(shape), a.data_ptr(), w.data_ptr(), out.data_ptr(), workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(), ctypes.byref(part), _stream_handle(stream))
    if rc != OK:
        raise PsrError(rc, "psr_ag_gemm")
    return out, workspace


def ring_attn_bwd_workspace_bytes(shape: Shape) -> int:
    n = load().psr_ring_attn_bwd_workspace_bytes(ctypes.byref(shape))
    if n == 0:
        raise PsrError(ERR_UNSUPPORTED, "psr_ring_attn_bwd_workspace_bytes")
    return int(n)


def ring_attn_bwd(q, k, v, o, lse, dout, *, P, causal, scale=None, workspace=None, dq=None, dk=None, dv=None,
                  timeout_ms=0, stream=None):
    """Ring Attention backward through the C ABI: q, o, dout [B][Hq][S][d], k, v [B][Hkv][S][d]
    (bf16), lse [B][Hq][S] fp32 (the forward's) -> (dq, dk, dv, workspace)."""
    import torch
    lib = load()
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("ring_attn_bwd: q, k, v must be 4-d [B, H, S, d]")
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    shape = make_shape(B, Hq, Hkv, S, P, d, causal, scale)
    need = ring_attn_bwd_workspace_bytes(shape)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, name in ((q, "q"), (o, "o"), (dout, "dout"), (dq, "dq")):
        _check_tensor(t, name, (B, Hq, S, d), torch.bfloat16)
    for t, name in ((k, "k"), (v, "v"), (dk, "dk"), (dv, "dv")):
        _check_tensor(t, name, (B, Hkv, S, d), torch.bfloat16)
    _check_tensor(lse, "lse", (B, Hq, S), torch.float32)
    _same_device((q, k, v, o, lse, dout, dq, dk, dv), "ring_attn_bwd")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    elif not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"ring_attn_bwd: workspace must be a CUDA tensor of at least {need} bytes")
    rc = lib.psr_ring_attn_bwd(ctypes.byref(shape), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(), int(timeout_ms),
                               _stream_handle(stream))
    if rc != OK:
        raise PsrError(rc, "psr_ring_attn_bwd")
    return dq, dk, dv, workspace


def gemm_rs_workspace_bytes(M, N, Ks, P) -> int:
    n = load().psr_gemm_rs_workspace_bytes(ctypes.byref(RsShape(int(M), int(N), int(Ks), int(P))))
    if n == 0:
        raise PsrError(ERR_UNSUPPORTED, "psr_gemm_rs_workspace_bytes")
    return int(n)


def gemm_rs(a, w, *, partition=None, workspace=None, out=None, stream=None):
    """GEMM + ReduceScatter through the C ABI: a [P][M][Ks] bf16 (rank r's activations),
    w [P][N][Ks] bf16 (rank r's weights) -> out [M][N] bf16 = sum_r a[r] @ w[r]^T, rows
    q*M/P .. belonging to rank q.  Returns (out, workspace)."""
    import torch
    lib = load()
    if a.dim() != 3 or w.dim() != 3:
        raise ValueError("gemm_rs: a must be [P, M, Ks] and w [P, N, Ks]")
    P, M, Ks = a.shape
    N = w.shape[1]
    shape = RsShape(int(M), int(N), int(Ks), int(P))
    need = gemm_rs_workspace_bytes(M, N, Ks, P)
    _check_tensor(a, "a", (P, M, Ks), torch.bfloat16)
    _check_tensor(w, "w", (P, N, Ks), torch.bfloat16)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    _check_tensor(out, "out", (M, N), torch.bfloat16)
    _same_device((a, w, out), "gemm_rs")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=a.device)
    elif not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"gemm_rs: workspace must be a CUDA tensor of at least {need} bytes")
    part = partition if partition is not None else make_partition()
    rc = lib.psr_gemm_rs(ctypes.byref(shape), a.data_ptr(), w.data_ptr(), out.data_ptr(), workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(), ctypes.byref(part), _stream_handle(stream))
    if rc != OK:
        raise PsrError(rc, "psr_gemm_rs")
    return out, workspace


def get_stats(workspace, stream=None) -> dict:
    st = Stats()
    rc = load().psr_get_stats(ctypes.c_void_p(workspace.data_ptr()), ctypes.byref(st), _stream_handle(stream))
    if rc not in (OK, ERR_TIMEOUT):
        raise PsrError(rc, "psr_get_stats")
    return st.as_dict()


def get_trajectory(workspace, max_entries=4096, stream=None):
    buf = (ctypes.c_uint32 * (2 * max_entries))()
    n = load().psr_get_trajectory(ctypes.c_void_p(workspace.data_ptr()), buf, max_entries, _stream_handle(stream))
    if n < 0:
        raise PsrError(-n, "psr_get_trajectory")
    return [(int(buf[2 * i]), int(buf[2 * i + 1])) for i in range(n)]
