"""The allocation-free entry point, psr_ring_attn_fwd_noalloc, called through the C ABI.

It serves callers that must not call cudaMalloc (a framework pool that owns the
device memory, a plug-in that may not allocate, a path that cannot take
cudaMalloc's implicit synchronisation).  Its scratch is a fixed device array in
the library; its results must equal those of psr_ring_attn_fwd, which uses a
caller-provided workspace, within the parity tolerances, on consecutive calls
that share that array.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import ring_inputs as ri

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
REL_L2 = 5e-3
LSE_ABS = 1e-3


def _bind(lib):
    fn = lib.psr_ring_attn_fwd_noalloc
    fn.argtypes = [ctypes.c_void_p] + [ctypes.c_void_p] * 5 + [ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _close(a, b, la, lb):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    la = la.cpu().numpy().astype(np.float64)
    lb = lb.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(a)) and np.all(np.isfinite(la))
    assert np.abs(a - b).max() <= MAX_ABS
    assert np.linalg.norm(a - b) / np.linalg.norm(b) <= REL_L2
    assert np.abs(la - lb).max() <= LSE_ABS


@pytest.mark.parametrize("w", [
    ri.WORKLOADS["small"],
    ri.WORKLOADS["small"].with_(name="noalloc_gqa_c_d128", B=2, Hq=4, Hkv=2, S=2048, P=8, d=128, causal=True,
                                seed=71),
], ids=lambda w: w.name)
def test_noalloc_matches_workspace_entry_point(psr, w):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fn = _bind(psr.load())
    q, k, v = ri.generate(w)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    qd, kd, vd = dev(q), dev(k), dev(v)
    o_ref, lse_ref, ws = psr.ring_attn_fwd(qd, kd, vd, P=w.P, causal=w.causal, scale=w.scale)
    assert psr.get_stats(ws)["status"] == 0
    shape = psr.make_shape(w.B, w.Hq, w.Hkv, w.S, w.P, w.d, w.causal, w.scale)
    part = psr.make_partition(psr.ADAPTIVE)
    stream = torch.cuda.current_stream()
    # output buffers made up front, so that only the library call runs between the memory readings
    outs = [(torch.full_like(qd, float("nan")),
             torch.full((w.B, w.Hq, w.S), float("nan"), dtype=torch.float32, device="cuda")) for _ in range(2)]
    torch.cuda.synchronize()
    for call, (o, lse) in enumerate(outs):
        free_before = torch.cuda.mem_get_info()[0]
        rc = fn(ctypes.addressof(shape), qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                ctypes.addressof(part), ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, psr.status_string(rc)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        if call == 1:
            assert free_after == free_before  # the call took no device memory (the array exists since call 0)
        _close(o, o_ref, lse, lse_ref)


def test_noalloc_rejects_shapes_beyond_the_scratch(psr):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fn = _bind(psr.load())
    big = psr.make_shape(1, 32, 32, 32768, 16, 128, False)  # needs ~1 GB of ring slots
    assert psr.workspace_bytes(big) > (64 << 20)
    part = psr.make_partition(psr.ADAPTIVE)
    ptr = 1 << 20  # never dereferenced: the size check comes first
    rc = fn(ctypes.addressof(big), ptr, ptr, ptr, ptr, ptr, ctypes.addressof(part), None)
    assert rc == psr.ERR_UNSUPPORTED
