"""CPU tests of the Python binding's argument checks: every entry point rejects a buffer of
the wrong dtype, shape, layout or memory kind before anything reaches the C ABI.  No GPU is
needed; where a check that runs earlier needs a CUDA or pinned tensor, the test stands in for
one by patching the tensor's is_cuda / is_pinned."""
import pytest
import torch


@pytest.fixture
def fake_device(monkeypatch):
    """Make CPU tensors pass the binding's CUDA-tensor and pinned-memory tests."""
    monkeypatch.setattr(torch.Tensor, "is_cuda", property(lambda self: True))
    monkeypatch.setattr(torch.Tensor, "is_pinned", lambda self: True)


SHAPE = dict(B=1, Hq=2, Hkv=2, S=1024, d=64)


def _host_args(B=1, Hq=2, Hkv=2, S=1024, d=64):
    q = torch.zeros((B, Hq, S, d), dtype=torch.int16)
    k = torch.zeros((B, Hkv, S, d), dtype=torch.int16)
    v = torch.zeros((B, Hkv, S, d), dtype=torch.int16)
    o = torch.zeros((B, Hq, S, d), dtype=torch.int16)
    lse = torch.zeros((B, Hq, S), dtype=torch.float32)
    dq = torch.zeros((B, Hq, S, d), dtype=torch.bfloat16)
    dk = torch.zeros((B, Hkv, S, d), dtype=torch.bfloat16)
    dv = torch.zeros((B, Hkv, S, d), dtype=torch.bfloat16)
    do = torch.zeros((B, Hq, S, d), dtype=torch.bfloat16)
    dl = torch.zeros((B, Hq, S), dtype=torch.float32)
    return [q, k, v, o, lse, dq, dk, dv, do, dl]


NAMES = ["q_host", "k_host", "v_host", "o_host", "lse_host", "dq", "dk", "dv", "d_o", "d_lse"]


def test_host_entry_rejects_pageable_host_memory(psr):
    with pytest.raises(ValueError, match="dq must be a CUDA tensor"):
        psr.ring_attn_fwd_host(*_host_args(), P=4, causal=False)


def test_host_entry_requires_pinned_host_buffers(psr, monkeypatch):
    monkeypatch.setattr(torch.Tensor, "is_cuda", property(lambda self: self.device.type == "cpu"))
    with pytest.raises(ValueError, match="q_host must be in pinned host memory"):
        psr.ring_attn_fwd_host(*_host_args(), P=4, causal=False)


@pytest.mark.parametrize("i", range(10), ids=NAMES)
def test_host_entry_rejects_a_wrong_shape(psr, fake_device, i):
    args = _host_args()
    if i == 0:  # q_host fixes the shape: a wrong k_host head count then mismatches the others
        args[0] = args[0][:, :, :512].contiguous()
        pat = "k_host|q_host|must have shape"
    else:
        args[i] = args[i][..., :-1].contiguous() if args[i].dim() == 4 else args[i][..., :-8].contiguous()
        pat = f"{NAMES[i]} must have shape"
    with pytest.raises(ValueError, match=pat):
        psr.ring_attn_fwd_host(*args, P=4, causal=False)


@pytest.mark.parametrize("i", range(10), ids=NAMES)
def test_host_entry_rejects_a_wrong_dtype(psr, fake_device, i):
    args = _host_args()
    args[i] = args[i].to(torch.float64)
    with pytest.raises(ValueError, match=f"{NAMES[i]} must be"):
        psr.ring_attn_fwd_host(*args, P=4, causal=False)


def test_host_entry_rejects_a_device_tensor_as_host_buffer(psr, fake_device):
    args = _host_args()
    args[3] = torch.zeros((1, 2, 1024, 64), dtype=torch.int16, device="meta")
    with pytest.raises(ValueError, match="o_host must be a host"):
        psr.ring_attn_fwd_host(*args, P=4, causal=False)


def test_host_entry_rejects_non_contiguous(psr, fake_device):
    args = _host_args()
    args[1] = torch.zeros((1, 2, 64, 1024), dtype=torch.int16).transpose(2, 3)
    with pytest.raises(ValueError, match="k_host must be contiguous"):
        psr.ring_attn_fwd_host(*args, P=4, causal=False)


def test_device_entry_rejects_wrong_shapes(psr, fake_device):
    q = torch.zeros((1, 2, 1024, 64), dtype=torch.bfloat16)
    k = torch.zeros((1, 2, 1024, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="v must have shape"):
        psr.ring_attn_fwd(q, k, k[:, :1].contiguous(), P=4, causal=False)
    with pytest.raises(ValueError, match="lse must have shape"):
        psr.ring_attn_fwd(q, k, k, P=4, causal=False, out=torch.zeros_like(q),
                          lse=torch.zeros((1, 2, 512), dtype=torch.float32))


def test_ag_gemm_rejects_wrong_shapes(psr, fake_device):
    M, K, Ns, P = 1024, 256, 256, 4
    a = torch.zeros((M, K), dtype=torch.bfloat16)
    w = torch.zeros((P, Ns, K), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="out must have shape"):
        psr.ag_gemm(a, w, P=P, out=torch.zeros((P, M, Ns - 8), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="w must have shape"):
        psr.ag_gemm(a, w[:2].contiguous(), P=P)
    with pytest.raises(ValueError, match="out must be"):
        psr.ag_gemm(a, w, P=P, out=torch.zeros((P, M, Ns), dtype=torch.float32))


def test_gemm_rs_rejects_wrong_shapes(psr, fake_device):
    P, M, N, Ks = 4, 1024, 256, 64
    a = torch.zeros((P, M, Ks), dtype=torch.bfloat16)
    w = torch.zeros((P, N, Ks), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="out must have shape"):
        psr.gemm_rs(a, w, out=torch.zeros((M, N + 256), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="w must have shape"):
        psr.gemm_rs(a, torch.zeros((P, N, 2 * Ks), dtype=torch.bfloat16))


def test_bwd_rejects_wrong_shapes(psr, fake_device):
    q = torch.zeros((1, 2, 1024, 64), dtype=torch.bfloat16)
    k = torch.zeros((1, 2, 1024, 64), dtype=torch.bfloat16)
    lse = torch.zeros((1, 2, 1024), dtype=torch.float32)
    with pytest.raises(ValueError, match="dout must have shape"):
        psr.ring_attn_bwd(q, k, k, q, lse, q[:, :, :512].contiguous(), P=4, causal=False)
    with pytest.raises(ValueError, match="lse must be"):
        psr.ring_attn_bwd(q, k, k, q, lse.double(), q, P=4, causal=False)
    with pytest.raises(ValueError, match="dk must have shape"):
        psr.ring_attn_bwd(q, k, k, q, lse, q, P=4, causal=False, dk=k[:, :1].contiguous())
