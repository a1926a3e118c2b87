"""kda_chunk_fwd_static_scratch: the entry point for callers that cannot allocate.

Plug-ins that a host runtime hands only input and output buffers (the runtime
owns the device memory pool), and latency-critical code that must not
allocate, call this variant: it runs the same kernels as kda_chunk_fwd on a
fixed scratch array inside the library instead of a caller workspace.  These
tests call it through the C ABI:

* twice in a row on two problems, on both forward paths: every output equals
  the ordinary entry point's bit for bit (same kernels on the same inputs;
  a stale read of the shared array would show up as a difference);
* a device-side error (a decreasing cu_seqlens) reaches its device_status
  output, and the next valid call on the same shared array starts clean;
* a problem too large for the fixed scratch is refused before any work is
  queued.

It lives in its own file so that pytest collects it last.
"""

import pytest
import torch

from chunked_gated_delta_03_gb300 import _lib, build, ops
from chunked_gated_delta_03_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

KEYS = ("o", "final_state", "Aqk", "Akk_inv", "W", "U")


def _outputs(B, T, Hv, K, V, N):
    nan = float("nan")
    return {
        "o": torch.full((B, T, Hv, V), nan, dtype=torch.bfloat16, device="cuda"),
        "final_state": torch.full((N, Hv, K, V), nan, dtype=torch.float32, device="cuda"),
        "Aqk": torch.full((B, T, Hv, 64), nan, dtype=torch.float32, device="cuda"),
        "Akk_inv": torch.full((B, T, Hv, 64), nan, dtype=torch.float32, device="cuda"),
        "W": torch.full((B, T, Hv, K), nan, dtype=torch.bfloat16, device="cuda"),
        "U": torch.full((B, T, Hv, V), nan, dtype=torch.bfloat16, device="cuda"),
    }


def _static_call(inp, path, cu=None):
    cu = inp["cu_seqlens"] if cu is None else cu
    a, (B, T, Hq, Hv, K, V, N) = ops.make_args(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                                               inp["initial_state"], cu)
    a.path = ops._PATHS[path]
    out = _outputs(B, T, Hv, K, V, N)
    a.o, a.final_state = out["o"].data_ptr(), out["final_state"].data_ptr()
    a.Aqk, a.Akk_inv = out["Aqk"].data_ptr(), out["Akk_inv"].data_ptr()
    a.W, a.U = out["W"].data_ptr(), out["U"].data_ptr()
    assert _lib.kda_workspace_size(a) <= _lib.KDA_STATIC_SCRATCH_BYTES
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    rc = _lib.kda_chunk_fwd_static_scratch(a, status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.KDA_OK, _lib.status_string(rc)
    torch.cuda.synchronize()
    return out, int(status.item())


CASES = {
    "varlen_gva": dict(lengths=(1, 63, 64, 65, 130, 7, 0, 200), Hq=2, Hv=4, K=128, V=128, initial_state=True,
                       beta_dtype="bf16", seed=31),
    "fixed_k64": dict(B=2, T=300, Hq=4, Hv=4, K=64, V=64, seed=32),
}


def _inputs():
    inputs = {}
    for name, kw in CASES.items():
        host = make_inputs(WORKLOADS["tiny"], **kw)
        inputs[name] = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    return inputs


@pytest.mark.parametrize("path", ["fused", "two_pass"])
def test_static_scratch_matches_workspace_entry_point(path):
    build.build()
    _lib.load()
    inputs = _inputs()
    for _ in range(2):  # two calls in a row on the shared scratch
        for name, inp in inputs.items():
            o, fin, im = ops.chunk_kda_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                                           inp["initial_state"], inp["cu_seqlens"], return_intermediates=True,
                                           path=path)
            got, status = _static_call(inp, path)
            assert status == _lib.KDA_OK, _lib.status_string(status)
            want = {"o": o, "final_state": fin, **im}
            for key in KEYS:
                assert torch.equal(got[key], want[key]), f"{name} {key}"


@pytest.mark.parametrize("path", ["fused", "two_pass"])
def test_static_scratch_reports_device_errors_then_recovers(path):
    build.build()
    _lib.load()
    inp = _inputs()["varlen_gva"]
    bad = inp["cu_seqlens"].clone()
    bad[4] = int(bad[3]) - 5  # no longer non-decreasing
    got, status = _static_call(inp, path, cu=bad)
    assert status == _lib.KDA_ERR_BAD_SEQLENS
    assert torch.isnan(got["o"].float()).all()  # the kernels saw the status and wrote nothing
    # the next valid call on the same shared array starts from a clean status
    o, fin, im = ops.chunk_kda_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                                   inp["initial_state"], inp["cu_seqlens"], return_intermediates=True, path=path)
    got, status = _static_call(inp, path)
    assert status == _lib.KDA_OK
    want = {"o": o, "final_state": fin, **im}
    for key in KEYS:
        assert torch.equal(got[key], want[key]), key


def test_static_scratch_refuses_oversized_problems():
    build.build()
    _lib.load()
    a = _lib.KdaArgs()
    base = 1 << 20  # never dereferenced: the size check comes first
    a.q = a.k = a.v = a.g = a.beta = a.o = base
    a.B, a.T, a.Hq, a.Hv, a.K, a.V, a.chunk, a.scale = 2, 8192, 64, 64, 128, 128, 64, 0.088
    a.path = _lib.KDA_PATH_TWO_PASS  # the two-pass path keeps its state-pass operands in the scratch
    assert _lib.kda_workspace_size(a) > _lib.KDA_STATIC_SCRATCH_BYTES
    assert _lib.kda_chunk_fwd_static_scratch(a, 0, 0) == _lib.KDA_ERR_WORKSPACE
