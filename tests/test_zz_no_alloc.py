"""kda_chunk_fwd_static_scratch: the entry point for callers that cannot allocate.

Plug-ins that a host runtime hands only input and output buffers (the runtime
owns the device memory pool), and latency-critical code that must not
allocate, call this variant: it runs the same kernels as kda_chunk_fwd on a
fixed scratch array inside the library instead of a caller workspace.  This
test calls it through the C ABI, twice in a row, and checks every output
against the ordinary entry point's within the parity tolerances of
test_kda_gpu.py; it also checks that a problem too large for the fixed scratch
is refused before any work is queued.  It lives in its own file so that pytest
collects it last.
"""

import numpy as np
import pytest
import torch

from chunked_gated_delta_03_gb300 import _lib, build, ops
from chunked_gated_delta_03_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

TOL = {"o": (2e-2, 5e-3), "final_state": (2e-2, 5e-3), "Aqk": (None, 1e-4), "Akk_inv": (None, 1e-4),
       "W": (2e-2, 5e-3), "U": (2e-2, 5e-3)}


def _close(name, got, want):
    got = got.double().cpu().numpy()
    want = want.double().cpu().numpy()
    atol, rel = TOL[name]
    assert np.all(np.isfinite(got)), name
    err = np.abs(got - want)
    if atol is not None:
        assert np.all(err <= atol + 1e-2 * np.abs(want)), f"{name}: max err {err.max():.3e}"
    denom = max(np.linalg.norm(want), 1e-30)
    assert np.linalg.norm(got - want) / denom <= rel, name


def _static_call(inp):
    a, (B, T, Hq, Hv, K, V, N) = ops.make_args(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                                               inp["initial_state"], inp["cu_seqlens"])
    out = {
        "o": torch.full((B, T, Hv, V), float("nan"), dtype=torch.bfloat16, device="cuda"),
        "final_state": torch.full((N, Hv, K, V), float("nan"), dtype=torch.float32, device="cuda"),
        "Aqk": torch.full((B, T, Hv, 64), float("nan"), dtype=torch.float32, device="cuda"),
        "Akk_inv": torch.full((B, T, Hv, 64), float("nan"), dtype=torch.float32, device="cuda"),
        "W": torch.full((B, T, Hv, K), float("nan"), dtype=torch.bfloat16, device="cuda"),
        "U": torch.full((B, T, Hv, V), float("nan"), dtype=torch.bfloat16, device="cuda"),
    }
    a.o, a.final_state = out["o"].data_ptr(), out["final_state"].data_ptr()
    a.Aqk, a.Akk_inv = out["Aqk"].data_ptr(), out["Akk_inv"].data_ptr()
    a.W, a.U = out["W"].data_ptr(), out["U"].data_ptr()
    assert _lib.kda_workspace_size(a) <= _lib.KDA_STATIC_SCRATCH_BYTES
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    rc = _lib.kda_chunk_fwd_static_scratch(a, status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.KDA_OK, _lib.status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == _lib.KDA_OK
    return out


CASES = {
    "varlen_gva": dict(lengths=(1, 63, 64, 65, 130, 7, 0, 200), Hq=2, Hv=4, K=128, V=128, initial_state=True,
                       beta_dtype="bf16", seed=31),
    "fixed_k64": dict(B=2, T=300, Hq=4, Hv=4, K=64, V=64, seed=32),
}


def test_static_scratch_matches_workspace_entry_point():
    build.build()
    _lib.load()
    inputs = {}
    for name, kw in CASES.items():
        host = make_inputs(WORKLOADS["tiny"], **kw)
        inputs[name] = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    for _ in range(2):  # two calls in a row on the shared scratch
        for name, inp in inputs.items():
            o, fin, im = ops.chunk_kda_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                                           inp["initial_state"], inp["cu_seqlens"], return_intermediates=True)
            got = _static_call(inp)
            want = {"o": o, "final_state": fin, **im}
            for key in TOL:
                _close(key, got[key], want[key])


def test_static_scratch_refuses_oversized_problems():
    build.build()
    _lib.load()
    a = _lib.KdaArgs()
    base = 1 << 20  # never dereferenced: the size check comes first
    a.q = a.k = a.v = a.g = a.beta = a.o = base
    a.B, a.T, a.Hq, a.Hv, a.K, a.V, a.chunk, a.scale = 2, 8192, 64, 64, 128, 128, 64, 0.088
    assert _lib.kda_workspace_size(a) > _lib.KDA_STATIC_SCRATCH_BYTES
    assert _lib.kda_chunk_fwd_static_scratch(a, 0, 0) == _lib.KDA_ERR_WORKSPACE
