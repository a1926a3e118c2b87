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
