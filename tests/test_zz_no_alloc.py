"""The allocation-free entry point, psr_ring_attn_fwd_noalloc, called through the C ABI.

It serves callers that must not call cudaMalloc (a framework pool that owns the
device memory, a plug-in that may not allocate, a path that cannot take
cudaMalloc's implicit synchronisation).  Its scratch is a fixed device array in
the library; its results must equal those of psr_ring_attn_fwd, which uses a
caller-provided workspace, within the parity tolerances, on consecutive calls
that share that array, and its device status must be readable through
psr_noalloc_get_stats.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

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


def _close(a, b, la, lb):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    la = la.cpu().numpy().astype(np.float64)
    lb = lb.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(a)) and np.all(np.isfinite(la))
    assert np.abs(a - b).max() <= MAX_ABS
    assert np.linalg.norm(a - b) / np.linalg.norm(b) <= REL_L2
    assert np.abs(la - lb).max() <= LSE_ABS


def _stats(lib, psr, stream):
    st = psr.Stats()
    rc = lib.psr_noalloc_get_stats(ctypes.byref(st), ctypes.c_void_p(stream.cuda_stream))
    return rc, st


class _Case:
    """Device inputs of a workload and the workspace entry's result on them."""

    def __init__(self, psr, torch, w):
        self.w = w
        q, k, v = ri.generate(w)
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
        self.q, self.k, self.v = dev(q), dev(k), dev(v)
        self.o_ref, self.lse_ref, ws = psr.ring_attn_fwd(self.q, self.k, self.v, P=w.P, causal=w.causal,
                                                         scale=w.scale)
        assert psr.get_stats(ws)["status"] == 0
        self.shape = psr.make_shape(w.B, w.Hq, w.Hkv, w.S, w.P, w.d, w.causal, w.scale)

    def outputs(self, torch):
        return (torch.full_like(self.q, float("nan")),
                torch.full((self.w.B, self.w.Hq, self.w.S), float("nan"), dtype=torch.float32, device="cuda"))

    def call(self, lib, o, lse, part, stream):
        return lib.psr_ring_attn_fwd_noalloc(ctypes.byref(self.shape), self.q.data_ptr(), self.k.data_ptr(),
                                             self.v.data_ptr(), o.data_ptr(), lse.data_ptr(), ctypes.byref(part),
                                             ctypes.c_void_p(stream.cuda_stream))


SMALL = ri.WORKLOADS["small"]
GQA_CAUSAL = SMALL.with_(name="noalloc_gqa_c_d128", B=2, Hq=4, Hkv=2, S=2048, P=8, d=128, causal=True, seed=71)


@pytest.mark.parametrize("w", [SMALL, GQA_CAUSAL], ids=lambda w: w.name)
def test_noalloc_matches_workspace_entry_point(psr, w):
    torch = _torch()
    lib = psr.load()
    case = _Case(psr, torch, w)
    part = psr.make_partition(psr.ADAPTIVE)
    stream = torch.cuda.current_stream()
    # output buffers made up front, so that only the library call runs between the memory readings
    outs = [case.outputs(torch) for _ in range(2)]
    torch.cuda.synchronize()
    for call, (o, lse) in enumerate(outs):
        free_before = torch.cuda.mem_get_info()[0]
        rc = case.call(lib, o, lse, part, stream)
        assert rc == 0, psr.status_string(rc)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        if call == 1:
            assert free_after == free_before  # the call took no device memory (the array exists since call 0)
        rc, st = _stats(lib, psr, stream)
        assert rc == 0 and st.status == 0 and st.compute_items > 0
        _close(o, case.o_ref, lse, case.lse_ref)


def test_noalloc_back_to_back_shapes_share_the_scratch(psr):
    # the larger workspace first (more groups, flags and queue entries), then a smaller one: the
    # second call must not see control words the first left in the shared array
    torch = _torch()
    lib = psr.load()
    big, small = _Case(psr, torch, GQA_CAUSAL), _Case(psr, torch, SMALL)
    assert psr.workspace_bytes(big.shape) > psr.workspace_bytes(small.shape)
    part = psr.make_partition(psr.ADAPTIVE)
    stream = torch.cuda.current_stream()
    for case in (big, small, big):
        o, lse = case.outputs(torch)
        rc = case.call(lib, o, lse, part, stream)
        assert rc == 0, psr.status_string(rc)
        rc, st = _stats(lib, psr, stream)
        assert rc == 0 and st.status == 0
        _close(o, case.o_ref, lse, case.lse_ref)


def test_noalloc_reports_a_device_timeout_and_recovers(psr):
    # a dropped readiness flag (host-visible protocol only) makes the bounded waits expire; the
    # status must reach the caller through psr_noalloc_get_stats, and the next call must be right
    torch = _torch()
    lib = psr.load()
    case = _Case(psr, torch, SMALL)
    stream = torch.cuda.current_stream()
    o, lse = case.outputs(torch)
    faulty = psr.make_partition(psr.ADAPTIVE, fault=psr.FAULT_DROP_FIRST_FLAG, timeout_ms=200)
    assert case.call(lib, o, lse, faulty, stream) == 0
    rc, st = _stats(lib, psr, stream)
    assert rc == psr.ERR_TIMEOUT and st.status == psr.ERR_TIMEOUT and st.error_site != 0
    o, lse = case.outputs(torch)
    assert case.call(lib, o, lse, psr.make_partition(psr.ADAPTIVE), stream) == 0
    rc, st = _stats(lib, psr, stream)
    assert rc == 0 and st.status == 0
    _close(o, case.o_ref, lse, case.lse_ref)


def test_noalloc_status_codes_match_the_workspace_entry(psr):
    torch = _torch()
    lib = psr.load()
    part = psr.make_partition(psr.ADAPTIVE)
    ptr = 1 << 20  # never dereferenced: every case below is rejected on the host
    ws = 1 << 21
    cases = [
        psr.make_shape(1, 2, 2, 1000, 4, 64, False),   # S % P != 0
        psr.make_shape(1, 2, 2, 1024, 4, 96, False),   # d = 96
        psr.make_shape(0, 2, 2, 1024, 4, 64, False),   # empty batch
        psr.make_shape(1, 3, 2, 1024, 4, 64, False),   # Hq % Hkv != 0
    ]
    for sh in cases:
        want = lib.psr_ring_attn_fwd(ctypes.byref(sh), ptr, ptr, ptr, ptr, ptr, ws, 1 << 40, ctypes.byref(part), None)
        got = lib.psr_ring_attn_fwd_noalloc(ctypes.byref(sh), ptr, ptr, ptr, ptr, ptr, ctypes.byref(part), None)
        assert want != 0 and got == want, (sh.S, sh.d, sh.B, sh.Hq, want, got)
    sh = psr.make_shape(1, 2, 2, 1024, 4, 64, False)
    assert lib.psr_ring_attn_fwd_noalloc(ctypes.byref(sh), None, ptr, ptr, ptr, ptr, ctypes.byref(part),
                                         None) == psr.ERR_ARG
    assert lib.psr_ring_attn_fwd_noalloc(ctypes.byref(sh), ptr + 8, ptr, ptr, ptr, ptr, ctypes.byref(part),
                                         None) == psr.ERR_ARG
    assert lib.psr_noalloc_get_stats(None, None) == psr.ERR_ARG
    torch.cuda.synchronize()


def test_noalloc_rejects_shapes_beyond_the_scratch(psr):
    _torch()
    lib = psr.load()
    big = psr.make_shape(1, 32, 32, 32768, 16, 128, False)  # needs ~1.6 GB of ring slots
    assert psr.workspace_bytes(big) > (64 << 20)
    part = psr.make_partition(psr.ADAPTIVE)
    ptr = 1 << 20  # never dereferenced: the size check comes before any launch
    rc = lib.psr_ring_attn_fwd_noalloc(ctypes.byref(big), ptr, ptr, ptr, ptr, ptr, ctypes.byref(part), None)
    assert rc == psr.ERR_UNSUPPORTED
