"""The PyTorch front end checks its arguments before any CUDA work (CPU)."""

import pytest
import torch

from chunked_gated_delta_03_gb300 import ops


def _inputs(dev="cpu", B=1, T=64, Hq=2, Hv=2, K=64, V=64):
    q = torch.zeros(B, T, Hq, K, dtype=torch.bfloat16, device=dev)
    k = torch.zeros_like(q)
    v = torch.zeros(B, T, Hv, V, dtype=torch.bfloat16, device=dev)
    g = torch.zeros(B, T, Hv, K, dtype=torch.float32, device=dev)
    beta = torch.zeros(B, T, Hv, dtype=torch.float32, device=dev)
    return q, k, v, g, beta


def test_cpu_tensors_are_rejected():
    with pytest.raises(ValueError, match="CUDA"):
        ops.chunk_kda_fwd(*_inputs())


def test_checks_run_before_cuda(monkeypatch):
    # dtype and shape errors are found by the same checks (here on CPU
    # tensors made to look like CUDA ones); nothing reaches the library
    q, k, v, g, beta = _inputs()
    monkeypatch.setattr(torch.Tensor, "is_cuda", property(lambda self: True))
    with pytest.raises(ValueError, match="bfloat16"):
        ops.make_args(q.float(), k, v, g, beta)
    with pytest.raises(ValueError, match="float32"):
        ops.make_args(q, k, v, g.bfloat16(), beta)
    with pytest.raises(ValueError, match="beta"):
        ops.make_args(q, k, v, g, beta.half())
    with pytest.raises(ValueError, match="must match"):
        ops.make_args(q, k, v, g[:, :32], beta)
    with pytest.raises(ValueError, match="initial_state"):
        ops.make_args(q, k, v, g, beta, initial_state=torch.zeros(1, 2, 64, 32))
    cu = torch.tensor([0, 64], dtype=torch.int64)
    with pytest.raises(ValueError, match="cu_seqlens"):
        ops.make_args(q, k, v, g, beta, cu_seqlens=cu)


def test_args_carry_sizes_and_options(monkeypatch):
    q, k, v, g, beta = _inputs(B=2, T=100, Hq=2, Hv=4, K=64, V=128)
    monkeypatch.setattr(torch.Tensor, "is_cuda", property(lambda self: True))
    a, (B, T, Hq, Hv, K, V, N) = ops.make_args(q, k, v, g, beta)
    assert (a.B, a.T, a.Hq, a.Hv, a.K, a.V, a.chunk) == (2, 100, 2, 4, 64, 128, 64) == (B, T, Hq, Hv, K, V, 64)
    assert a.N == 0 and N == 2 and a.cu_seqlens is None
    assert a.beta_dtype == 1 and abs(a.scale - 64 ** -0.5) < 1e-7
    assert a.QG is None and a.intra_tf32 == 0


def _fake_devices(monkeypatch):
    # every tensor looks like a CUDA tensor on device 0, unless it carries
    # `_host` (a host tensor) or `_ordinal` (another device)
    monkeypatch.setattr(torch.Tensor, "is_cuda", property(lambda self: not getattr(self, "_host", False)))
    monkeypatch.setattr(torch.Tensor, "device",
                        property(lambda self: torch.device("cuda", getattr(self, "_ordinal", 0))))


def test_host_initial_state_and_cu_seqlens_are_rejected(monkeypatch):
    # a host pointer passed as a device pointer would be dereferenced by the
    # kernels: the front end refuses it first
    q, k, v, g, beta = _inputs()
    _fake_devices(monkeypatch)
    h0 = torch.zeros(1, 2, 64, 64)
    h0._host = True
    with pytest.raises(ValueError, match="initial_state must be a CUDA tensor"):
        ops.make_args(q, k, v, g, beta, initial_state=h0)
    cu = torch.tensor([0, 64], dtype=torch.int32)
    cu._host = True
    with pytest.raises(ValueError, match="cu_seqlens must be a CUDA tensor"):
        ops.make_args(q, k, v, g, beta, cu_seqlens=cu)


@pytest.mark.parametrize("name", ["k", "v", "g", "beta", "initial_state", "cu_seqlens"])
def test_tensors_on_another_device_are_rejected(monkeypatch, name):
    q, k, v, g, beta = _inputs()
    _fake_devices(monkeypatch)
    t = {"k": k, "v": v, "g": g, "beta": beta, "initial_state": torch.zeros(1, 2, 64, 64),
         "cu_seqlens": torch.tensor([0, 64], dtype=torch.int32)}
    t[name]._ordinal = 1
    with pytest.raises(ValueError, match="one device"):
        ops.make_args(q, t["k"], t["v"], t["g"], t["beta"], initial_state=t["initial_state"],
                      cu_seqlens=t["cu_seqlens"])


def test_unknown_path_is_rejected(monkeypatch):
    q, k, v, g, beta = _inputs()
    _fake_devices(monkeypatch)
    with pytest.raises(ValueError, match="path"):
        ops.chunk_kda_fwd(q, k, v, g, beta, path="three_pass")
