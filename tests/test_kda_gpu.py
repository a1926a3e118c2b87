"""GPU parity of the CUDA path against the FP64 oracle, through the C ABI.

Both forward paths are covered: the fused kernel (the default) and the
two-pass kernels (intra-chunk, then state/output); PATHS parametrises the
parity tests over them.

Tolerances (floating point): o and final_state max |err| <= 2e-2 and relative
L2 <= 5e-3 (bf16 I/O); Akk_inv and Aqk relative L2 <= 1e-4 (FP32 outputs of an
~FP32-accurate hi/lo-split product and an FP32 inverse); W, U elementwise
|err| <= 2e-2 + 1e-2 |ref| and relative L2 <= 5e-3 (bf16 outputs whose values
reach several units: a bf16 half-ulp alone is 2^-9 |x|, and their MMA
operands k*e^G, v and Akk_inv diag(beta) are bf16 too); G relative L2 <= 1e-5
(FP32 cumsum); QG = q*e^G elementwise |err| <= 2^-8 |ref| + 1e-6 (one bf16
rounding of an FP32 product).  Chunk indices and offsets: bit-exact.
"""

import numpy as np
import pytest
import torch

from chunked_gated_delta_03_gb300 import _lib, build
from chunked_gated_delta_03_gb300 import ops
from chunked_gated_delta_03_gb300.workloads import WORKLOADS, Workload, make_inputs
from oracle import kda_ref as ref

pytestmark = pytest.mark.gpu

TOL_STATE = dict(max_abs=2e-2, rel=5e-3)
TOL_WU = dict(atol=2e-2, rtol=1e-2, rel=5e-3)
TOL_FP32 = dict(rel=1e-4)
TOL_G = dict(rel=1e-5)
# The TF32 option rounds the gated q and k factors to TF32 (10-bit mantissa)
# before one MMA pass: a few 1e-4 relative error in Aqk
TOL_AQK_TF32 = dict(rel=1e-3)
# QG = q e^G is rounded once from an FP32 product to bf16 (8 significant
# bits): |err| <= 2^-8 |ref| plus the FP32 exp error
TOL_QG = dict(atol=1e-6, rtol=2.0 ** -8 + 1e-5, rel=3e-3)


PATHS = ["fused", "two_pass"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    _lib.load()


def _np(t):
    return None if t is None else t.detach().double().cpu().numpy()


def _oracle(inp, heads=None):
    """FP64 oracle on the CPU copy of the inputs; with ``heads``, only those
    value heads (each run as its own single-head problem, results stacked on
    the head axis in the order given)."""
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].cpu().numpy()
    if heads is None:
        return ref.kda_chunked(_np(inp["q"]), _np(inp["k"]), _np(inp["v"]), _np(inp["g"]), _np(inp["beta"]),
                               inp["scale"], _np(inp["initial_state"]), cu, chunk_size=64)
    grp = inp["Hv"] // inp["Hq"]
    parts = []
    for hv in heads:
        hq = hv // grp
        h0 = inp["initial_state"]
        parts.append(ref.kda_chunked(
            _np(inp["q"][:, :, hq:hq + 1]), _np(inp["k"][:, :, hq:hq + 1]), _np(inp["v"][:, :, hv:hv + 1]),
            _np(inp["g"][:, :, hv:hv + 1]), _np(inp["beta"][:, :, hv:hv + 1]), inp["scale"],
            None if h0 is None else _np(h0[:, hv:hv + 1]), cu, chunk_size=64))
    out = {}
    for key in parts[0]:
        axis = 1 if key == "final_state" else 2
        out[key] = np.concatenate([p[key] for p in parts], axis=axis)
    return out


def _cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _ours(inp, inter=True, G=False, QG=False, tf32=False, path="auto", chunk_table=None):
    return ops.chunk_kda_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                             inp["initial_state"], inp["cu_seqlens"], output_final_state=True,
                             return_intermediates=inter, return_G=G, return_QG=QG, tf32=tf32, path=path,
                             chunk_table=chunk_table)


def _check(name, got, want, max_abs=None, rel=None, atol=None, rtol=None):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - want)
    nrm = np.linalg.norm(want)
    r = np.linalg.norm(got - want) / (nrm if nrm > 0 else 1.0)
    if max_abs is not None:
        assert err.max() <= max_abs, f"{name}: max abs err {err.max():.3e} > {max_abs}"
    if atol is not None:
        bound = atol + rtol * np.abs(want)
        worst = np.max(err - bound)
        assert worst <= 0, f"{name}: |err| exceeds {atol} + {rtol}|ref| by {worst:.3e}"
    if rel is not None:
        assert r <= rel, f"{name}: rel L2 err {r:.3e} > {rel}"
    return float(err.max()), float(r)


def _compare(inp, out, want, heads=None, inter=True):
    """Compare our outputs (optionally only value heads ``heads``) with the oracle's."""
    o, final, im = out
    sel = slice(None) if heads is None else list(heads)
    _check("o", _np(o[:, :, sel]), want["o"], **TOL_STATE)
    _check("final_state", _np(final[:, sel]), want["final_state"], **TOL_STATE)
    if inter:
        _check("Akk_inv", _np(im["Akk_inv"][:, :, sel]), want["Akk_inv"], **TOL_FP32)
        _check("Aqk", _np(im["Aqk"][:, :, sel]), want["Aqk"], **TOL_FP32)
        _check("W", _np(im["W"][:, :, sel]), want["W"], **TOL_WU)
        _check("U", _np(im["U"][:, :, sel]), want["U"], **TOL_WU)
        if "G" in im:
            _check("G", _np(im["G"][:, :, sel]), want["G"], **TOL_G)
        if "QG" in im:
            _check("QG", _np(im["QG"][:, :, sel]), want["QG"], **TOL_QG)


SMALL_CASES = {
    "tiny": dict(),
    "ragged_k64_v128": dict(T=130, K=64, V=128, B=2, beta_dtype="bf16"),
    "ragged_k128_v64": dict(T=37, K=128, V=64, B=1),
    "gva_init": dict(T=200, Hq=2, Hv=4, K=128, V=128, initial_state=True, B=2),
    "varlen": dict(lengths=(1, 63, 64, 65, 130, 7, 0, 200), Hq=2, Hv=2, K=128, V=128, initial_state=True,
                   beta_dtype="bf16"),
    "varlen_gva_k64": dict(lengths=(5, 129, 64), Hq=1, Hv=3, K=64, V=64, initial_state=True),
}


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", sorted(SMALL_CASES))
def test_small_cases_match_oracle(case, path):
    inp = make_inputs(WORKLOADS["tiny"], seed=100 + len(case), **SMALL_CASES[case])
    want = _oracle(inp)
    out = _ours(_cuda(inp), inter=True, G=True, QG=True, path=path)
    _compare(inp, out, want, inter=True)


@pytest.mark.parametrize("case", ["tiny", "ragged_k64_v128", "ragged_k128_v64", "gva_init", "varlen"])
def test_tf32_option_matches_oracle(case):
    # The TF32 option (single-pass Aqk / Akk on TF32 operands) keeps Akk_inv
    # within the specified 1e-4; Aqk takes the TF32 bar; everything else the
    # default bars.
    inp = make_inputs(WORKLOADS["tiny"], seed=300 + len(case), **SMALL_CASES[case])
    want = _oracle(inp)
    o, final, im = _ours(_cuda(inp), inter=True, G=True, QG=True, tf32=True)
    _check("o", _np(o), want["o"], **TOL_STATE)
    _check("final_state", _np(final), want["final_state"], **TOL_STATE)
    _check("Akk_inv", _np(im["Akk_inv"]), want["Akk_inv"], **TOL_FP32)
    _check("Aqk", _np(im["Aqk"]), want["Aqk"], **TOL_AQK_TF32)
    _check("W", _np(im["W"]), want["W"], **TOL_WU)
    _check("U", _np(im["U"]), want["U"], **TOL_WU)
    _check("G", _np(im["G"]), want["G"], **TOL_G)
    _check("QG", _np(im["QG"]), want["QG"], **TOL_QG)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", ["gva_init", "varlen"])
def test_outputs_without_intermediates(case, path):
    # Without exports (W and U then stay in the workspace on the two-pass
    # path, on chip on the fused one) o and the final state must match the
    # oracle and, bit for bit, the call that exports them.
    inp = make_inputs(WORKLOADS["tiny"], seed=200 + len(case), **SMALL_CASES[case])
    want = _oracle(inp)
    dev = _cuda(inp)
    o, final, im = _ours(dev, inter=False, path=path)
    assert im is None
    _check("o", _np(o), want["o"], **TOL_STATE)
    _check("final_state", _np(final), want["final_state"], **TOL_STATE)
    o2, final2, _ = _ours(dev, inter=True, path=path)
    assert torch.equal(o, o2) and torch.equal(final, final2)


def test_intra_primitive_matches_oracle_and_full_path():
    # the standalone primitive runs the two-pass path's intra kernel: its
    # outputs equal that path's exports bit for bit
    inp = _cuda(make_inputs(WORKLOADS["tiny"], seed=7, **SMALL_CASES["varlen"]))
    intra = ops.chunk_kda_fwd_intra(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                                    inp["cu_seqlens"], return_G=True, return_QG=True)
    _, _, im = _ours(inp, inter=True, G=True, QG=True, path="two_pass")
    for key in ("Aqk", "Akk_inv", "W", "U", "G", "QG"):
        assert torch.equal(intra[key], im[key]), key
    want = _oracle({k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()})
    _check("Akk_inv", _np(intra["Akk_inv"]), want["Akk_inv"], **TOL_FP32)
    _check("W", _np(intra["W"]), want["W"], **TOL_WU)


@pytest.mark.parametrize("path", PATHS)
def test_inverse_identity_on_gpu_output(path):
    inp = make_inputs(WORKLOADS["mha_1k"], T=256, B=1, Hq=4, Hv=4)
    _, _, im = _ours(_cuda(inp), inter=True, G=True, path=path)
    want = _oracle(inp)
    # (I + Akk) Akk_inv = I with the oracle's Akk and the GPU's inverse
    A = want["Akk"][0, :64, 0, :64]
    X = _np(im["Akk_inv"])[0, :64, 0, :64]
    assert np.abs((np.eye(64) + A) @ X - np.eye(64)).max() < 1e-4


# --------------------------------------------------------------- workloads
_ORACLE_CACHE = {}


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name, heads", [
    ("tiny", None),
    ("mha_1k", [0, 17, 63]),
    ("mha_8k", [0, 37]),
    ("gva_4k", [0, 5, 63]),
    ("varlen_16k", [0, 33]),
])
def test_workload_matches_oracle(name, heads, path):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    if name not in _ORACLE_CACHE:
        _ORACLE_CACHE[name] = _oracle(inp, heads=heads)
    want = _ORACLE_CACHE[name]
    out = _ours(_cuda(inp), inter=True, path=path)
    _compare(inp, out, want, heads=heads, inter=True)


# ------------------------------------------------------------ edge cases
def test_chunk_indices_bit_exact():
    for lens in ([1], [64], [65], [1, 63, 64, 65, 0, 129, 3], [0, 0], [4096, 1, 2000]):
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
        idx, off = ops.prepare_chunk_indices(cu, 64)
        want_idx, want_off = ref.prepare_chunk_indices(cu.cpu().numpy(), 64)
        assert np.array_equal(idx.cpu().numpy(), want_idx)
        assert np.array_equal(off.cpu().numpy(), want_off)
    cu = torch.tensor([0], dtype=torch.int32, device="cuda")
    idx, off = ops.prepare_chunk_indices(cu, 64)
    assert idx.shape == (0, 2) and off.tolist() == [0]


def test_chunk_indices_reject_bad_metadata():
    with pytest.raises(ValueError):
        ops.prepare_chunk_indices(torch.tensor([0, 10, 4], dtype=torch.int32, device="cuda"), 64)
    with pytest.raises(ValueError):
        ops.prepare_chunk_indices(torch.tensor([3, 10], dtype=torch.int32, device="cuda"), 64)
    for bad in (None, 0, -64):
        with pytest.raises(ValueError):
            ops.prepare_chunk_indices(torch.tensor([0, 4], dtype=torch.int32, device="cuda"), bad)


@pytest.mark.parametrize("path", PATHS)
def test_bad_cu_seqlens_sets_device_status(path):
    inp = _cuda(make_inputs(WORKLOADS["tiny"], lengths=(100, 156)))
    a, _ = ops.make_args(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"], None,
                         inp["cu_seqlens"])
    a.path = ops._PATHS[path]
    o = torch.zeros(1, 256, 2, 64, dtype=torch.bfloat16, device="cuda")
    a.o = o.data_ptr()
    bad = torch.tensor([0, 150, 100], dtype=torch.int32, device="cuda")  # decreasing
    a.cu_seqlens = bad.data_ptr()
    n = _lib.kda_workspace_size(a)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    assert _lib.kda_chunk_fwd(a, ws.data_ptr(), n, torch.cuda.current_stream().cuda_stream) == _lib.KDA_OK
    assert ops.device_status(ws) == _lib.KDA_ERR_BAD_SEQLENS
    assert torch.count_nonzero(o) == 0  # kernels saw the status and wrote nothing
    # a good call on the same workspace clears the status
    a.cu_seqlens = inp["cu_seqlens"].data_ptr()
    assert _lib.kda_chunk_fwd(a, ws.data_ptr(), n, torch.cuda.current_stream().cuda_stream) == _lib.KDA_OK
    assert ops.device_status(ws) == _lib.KDA_OK


@pytest.mark.parametrize("path", PATHS)
def test_caller_chunk_table_gives_the_same_results(path):
    # a chunk table built once by kda_prepare_chunk_indices and passed back in
    # (checked on the device, then used by the two-pass kernels) gives the
    # results of the call that builds its own, bit for bit
    inp = _cuda(make_inputs(WORKLOADS["tiny"], seed=71, **SMALL_CASES["varlen"]))
    table = ops.prepare_chunk_indices(inp["cu_seqlens"], 64)
    ref_out = _ours(inp, inter=True, path=path)
    out = _ours(inp, inter=True, path=path, chunk_table=table)
    assert torch.equal(ref_out[0], out[0]) and torch.equal(ref_out[1], out[1])
    for key in ref_out[2]:
        assert torch.equal(ref_out[2][key], out[2][key]), key


@pytest.mark.parametrize("path", PATHS)
def test_aqk_16_bytes_off_a_32_byte_boundary_gives_the_same_results(path):
    # Aqk rows leave in 32-byte stores when the buffer is 32-byte aligned and
    # in 16-byte stores otherwise (the API asks for 16); Akk_inv moves by the
    # same offset.  Only the store width differs, so the values are the same
    # bits as from aligned buffers, on a chain with a partial tail chunk.
    inp = _cuda(make_inputs(WORKLOADS["tiny"], seed=81, T=200, initial_state=True))
    stream = torch.cuda.current_stream().cuda_stream
    outs = []
    for shift in (0, 4):                         # fp32 elements: 0 or 16 bytes past a 256-byte base
        a, (B, T, Hq, Hv, K, V, N) = ops.make_args(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                                   inp["scale"], inp["initial_state"], inp["cu_seqlens"])
        a.path = ops._PATHS[path]
        bufs = {"o": torch.empty(B, T, Hv, V, dtype=torch.bfloat16, device="cuda"),
                "final_state": torch.empty(N, Hv, K, V, dtype=torch.float32, device="cuda"),
                "W": torch.empty(B, T, Hv, K, dtype=torch.bfloat16, device="cuda"),
                "U": torch.empty(B, T, Hv, V, dtype=torch.bfloat16, device="cuda")}
        for name in ("Aqk", "Akk_inv"):
            n = B * T * Hv * 64
            bufs[name] = torch.full((n + shift,), float("nan"), dtype=torch.float32,
                                    device="cuda")[shift:].view(B, T, Hv, 64)
        assert bufs["Aqk"].data_ptr() % 32 == (16 if shift else 0)
        for name, t in bufs.items():
            setattr(a, name, t.data_ptr())
        n = _lib.kda_workspace_size(a)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        assert _lib.kda_chunk_fwd(a, ws.data_ptr(), n, stream) == _lib.KDA_OK
        assert ops.device_status(ws) == _lib.KDA_OK
        outs.append(bufs)
    for name in outs[0]:
        assert torch.equal(outs[0][name], outs[1][name]), name
    want = _oracle(inp)
    _check("Aqk", _np(outs[1]["Aqk"]), want["Aqk"], **TOL_FP32)
    _check("Akk_inv", _np(outs[1]["Akk_inv"]), want["Akk_inv"], **TOL_FP32)


@pytest.mark.parametrize("path", PATHS)
def test_bad_caller_chunk_table_sets_device_status(path):
    inp = _cuda(make_inputs(WORKLOADS["tiny"], seed=72, lengths=(100, 30, 156)))
    idx, off = ops.prepare_chunk_indices(inp["cu_seqlens"], 64)
    stream = torch.cuda.current_stream().cuda_stream
    cases = []
    swapped = idx.clone()
    swapped[[0, 1]] = swapped[[1, 0]]            # two pairs out of order
    cases.append((swapped, off))
    shifted = off.clone()
    shifted[1:] += 1                             # offsets that skip a row
    cases.append((idx, shifted))
    for t_idx, t_off in cases:
        a, (B, T, Hq, Hv, K, V, N) = ops.make_args(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                                   inp["scale"], None, inp["cu_seqlens"])
        a.path = ops._PATHS[path]
        a.chunk_indices, a.chunk_offsets = t_idx.data_ptr(), t_off.data_ptr()
        o = torch.zeros(B, T, Hv, V, dtype=torch.bfloat16, device="cuda")
        a.o = o.data_ptr()
        n = _lib.kda_workspace_size(a)
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        assert _lib.kda_chunk_fwd(a, ws.data_ptr(), n, stream) == _lib.KDA_OK
        assert ops.device_status(ws) == _lib.KDA_ERR_BAD_CHUNK_TABLE
        assert torch.count_nonzero(o) == 0


@pytest.mark.parametrize("path", PATHS)
def test_strong_gates_within_range_match_oracle(path):
    # A per-step log-gate of -0.9 on every other channel: each full chunk then
    # decays by 57.6 on those channels, just inside KDA_MAX_CHUNK_LOG_DECAY, so
    # the operands q e^G and k e^-G span about 25 decades.
    inp = make_inputs(WORKLOADS["tiny"], seed=43, T=200, initial_state=True)
    g = inp["g"].clone()
    g[..., ::2] = -0.9
    inp["g"] = g
    want = _oracle(inp)
    out = _ours(_cuda(inp), inter=True, path=path)
    _compare(inp, out, want, inter=True)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("decay", [64.0, 200.0])
def test_gates_past_the_range_take_the_exact_path(path, decay):
    # Every other channel of value head 1 decays by `decay` over each full
    # chunk, past the range in which the tensor-core kernels' factorised decay
    # operands k e^{-G} stay finite: those kernels mark the chain and the
    # exact path recomputes it, while head 0 stays on the fast path.  The
    # oracle forms e^{G_r - G_i} directly in FP64.
    inp = make_inputs(WORKLOADS["tiny"], seed=44, T=200, K=128, V=128, initial_state=True)
    g = inp["g"].clone()
    g[:, :, 1, ::2] = -decay / 64
    inp["g"] = g
    want = _oracle(inp)
    cin = _cuda(inp)
    a, (B, T, Hq, Hv, K, V, N) = ops.make_args(cin["q"], cin["k"], cin["v"], cin["g"], cin["beta"],
                                               cin["scale"], cin["initial_state"], None)
    a.path = ops._PATHS[path]
    o = torch.full((B, T, Hv, V), float("nan"), dtype=torch.bfloat16, device="cuda")
    fin = torch.full((N, Hv, K, V), float("nan"), dtype=torch.float32, device="cuda")
    im = {"Aqk": torch.full((B, T, Hv, 64), float("nan"), dtype=torch.float32, device="cuda"),
          "Akk_inv": torch.full((B, T, Hv, 64), float("nan"), dtype=torch.float32, device="cuda"),
          "W": torch.full((B, T, Hv, K), float("nan"), dtype=torch.bfloat16, device="cuda"),
          "U": torch.full((B, T, Hv, V), float("nan"), dtype=torch.bfloat16, device="cuda"),
          "G": torch.full((B, T, Hv, K), float("nan"), dtype=torch.float32, device="cuda"),
          "QG": torch.full((B, T, Hv, K), float("nan"), dtype=torch.bfloat16, device="cuda")}
    a.o, a.final_state = o.data_ptr(), fin.data_ptr()
    for key, t in im.items():
        setattr(a, key, t.data_ptr())
    n = _lib.kda_workspace_size(a)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    assert _lib.kda_chunk_fwd(a, ws.data_ptr(), n, torch.cuda.current_stream().cuda_stream) == _lib.KDA_OK
    assert ops.device_status(ws) == _lib.KDA_OK
    _compare(inp, (o, fin, im), want, inter=True)


@pytest.mark.parametrize("path", PATHS)
def test_strong_gates_in_one_packed_sequence(path):
    # only the chain of the second sequence and head 0 passes the range (a
    # decay of 96 per full chunk on eight channels); every other chain keeps
    # the fast path, tails and an empty sequence included
    inp = make_inputs(WORKLOADS["tiny"], seed=45, lengths=(70, 130, 0, 5, 64), Hq=2, Hv=2, K=64, V=64,
                      initial_state=True, beta_dtype="bf16")
    g = inp["g"].clone()
    g[:, 70:200, 0, :8] = -1.5
    inp["g"] = g
    want = _oracle(inp)
    out = _ours(_cuda(inp), inter=True, G=True, QG=True, path=path)
    _compare(inp, out, want, inter=True)


def test_intra_primitive_with_strong_gates():
    inp = make_inputs(WORKLOADS["tiny"], seed=46, T=150, K=128, V=64)
    g = inp["g"].clone()
    g[:, :, 0, 3] = -2.0  # 128 per full chunk on one channel of head 0
    inp["g"] = g
    want = _oracle(inp)
    cin = _cuda(inp)
    intra = ops.chunk_kda_fwd_intra(cin["q"], cin["k"], cin["v"], cin["g"], cin["beta"], cin["scale"], None,
                                    return_G=True, return_QG=True)
    _check("Akk_inv", _np(intra["Akk_inv"]), want["Akk_inv"], **TOL_FP32)
    _check("Aqk", _np(intra["Aqk"]), want["Aqk"], **TOL_FP32)
    _check("W", _np(intra["W"]), want["W"], **TOL_WU)
    _check("U", _np(intra["U"]), want["U"], **TOL_WU)
    _check("G", _np(intra["G"]), want["G"], **TOL_G)
    _check("QG", _np(intra["QG"]), want["QG"], **TOL_QG)


def _ours_cp(inp, cp_chunks, inter=True):
    return ops.chunk_kda_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                             inp["initial_state"], None, output_final_state=True, return_intermediates=inter,
                             cp_chunks=cp_chunks)


def test_context_parallel_long_sequence_matches_oracle():
    # one 16k-token sequence with 8 heads (8 chains on the GPU): cut into
    # segments of 16 chunks, the 128 segment chains run in parallel, their
    # start states come from the scan over segment transitions
    host = make_inputs(WORKLOADS["long_16k_h8"])
    inp = _cuda(host)
    out = _ours_cp(inp, 16)
    heads = [0, 5]
    want = _oracle(host, heads=heads)
    _compare(host, out, want, heads=heads, inter=True)
    # and against the unsplit chains: the same numbers up to bf16 rounding order
    o0, fin0, _ = _ours(inp, inter=False)
    _check("o vs unsplit", _np(out[0]), _np(o0), rel=3e-3)
    _check("final vs unsplit", _np(out[1]), _np(fin0), rel=3e-3)


def test_context_parallel_ragged_segments_match_oracle():
    # segments of 4 chunks over 11-chunk sequences (the last segment partial,
    # the last chunk a tail of 60 tokens), two sequences with initial states
    host = make_inputs(WORKLOADS["tiny"], seed=47, B=2, T=700, Hq=2, Hv=2, K=64, V=64, initial_state=True,
                       beta_dtype="bf16")
    out = _ours_cp(_cuda(host), 4)
    _compare(host, out, _oracle(host), inter=True)


def test_context_parallel_single_segment_is_the_plain_call():
    host = make_inputs(WORKLOADS["tiny"], seed=48, T=256, initial_state=True)
    inp = _cuda(host)
    o1, f1, i1 = _ours_cp(inp, 8)
    o0, f0, i0 = _ours(inp, inter=True)
    assert torch.equal(o1, o0) and torch.equal(f1, f0)
    for key in i0:
        assert torch.equal(i1[key], i0[key]), key


@pytest.mark.parametrize("path", PATHS)
def test_zero_beta_is_pure_gated_decay(path):
    # beta = 0: no delta updates.  Akk = 0, so Akk_inv is the identity and W, U
    # vanish exactly; the state only decays, S_T = Diag(e^{sum_t g_t}) S0, and
    # o_t = scale S0^T (q_t * e^{sum_{j<=t} g_j}) in closed form.
    inp = make_inputs(WORKLOADS["tiny"], seed=47, T=200, initial_state=True)
    inp["beta"] = torch.zeros_like(inp["beta"])
    o, final, im = _ours(_cuda(inp), inter=True, path=path)
    q = inp["q"].double().numpy()[0]              # [T, H, K]
    g = inp["g"].double().numpy()[0]              # [T, H, K]
    S0 = inp["initial_state"].double().numpy()[0]  # [H, K, V]
    Gc = np.cumsum(g, axis=0)
    want_final = np.exp(Gc[-1])[:, :, None] * S0
    want_o = inp["scale"] * np.einsum("thk,hkv->thv", q * np.exp(Gc), S0)
    _check("final_state", _np(final)[0], want_final, **TOL_STATE)
    _check("o", _np(o)[0], want_o, **TOL_STATE)
    T, H = q.shape[0], q.shape[1]
    eye = np.zeros((T, H, 64))
    for t in range(T):
        eye[t, :, t % 64] = 1.0
    assert np.array_equal(_np(im["Akk_inv"])[0], eye)
    assert torch.count_nonzero(im["W"]) == 0 and torch.count_nonzero(im["U"]) == 0


def test_bounded_wait_gives_up_and_reports_timeout():
    # a wait nothing satisfies ends after its limit with KDA_ERR_TIMEOUT in the
    # status word, and the context stays usable for the next call
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert _lib.kda_check_bounded_wait(status.data_ptr(), stream) == _lib.KDA_OK
    torch.cuda.synchronize()
    assert int(status.item()) == _lib.KDA_ERR_TIMEOUT
    inp = make_inputs(WORKLOADS["tiny"], seed=48)
    _compare(inp, _ours(_cuda(inp), inter=True), _oracle(inp), inter=True)


@pytest.mark.parametrize("path", PATHS)
def test_empty_inputs(path):
    inp = _cuda(make_inputs(WORKLOADS["tiny"], T=0, initial_state=True))
    o, final, _ = _ours(inp, inter=False, path=path)
    assert o.numel() == 0 and torch.equal(final, inp["initial_state"])
    inp = _cuda(make_inputs(WORKLOADS["tiny"], lengths=(0, 0), initial_state=True))
    o, final, _ = _ours(inp, inter=False, path=path)
    assert torch.equal(final, inp["initial_state"])


@pytest.mark.parametrize("path", PATHS)
def test_nonfinite_values_stay_in_their_sequence(path):
    # Packed varlen: sequence 0 ends in a tail chunk (tokens 64-99, L = 36)
    # whose 64-row TMA boxes (v in the intra kernel, Kl in the state kernel)
    # also cover the first tokens of sequence 1.  NaN / Inf planted in v and k
    # of those tokens must not reach sequence 0: its o and final state match
    # the oracle run on sequence 0 alone.
    inp = make_inputs(WORKLOADS["tiny"], seed=61, lengths=(100, 50), Hq=2, Hv=2, K=128, V=128,
                      initial_state=True)
    bad = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    bad["v"][0, 110, 1, 5] = float("nan")
    bad["v"][0, 120, 0, :] = float("inf")
    bad["k"][0, 105, 0, 7] = float("nan")
    bad["k"][0, 126, 1, :] = float("inf")
    o, final, _ = _ours(_cuda(bad), inter=True, path=path)
    seq0 = make_inputs(WORKLOADS["tiny"], seed=61, lengths=(100, 50), Hq=2, Hv=2, K=128, V=128,
                       initial_state=True)
    for key in ("q", "k", "v", "g", "beta"):
        seq0[key] = seq0[key][:, :100]
    seq0["initial_state"] = seq0["initial_state"][:1]
    seq0["cu_seqlens"] = None
    seq0["T"] = 100
    want = _oracle(seq0)
    _check("o", _np(o[:, :100]), want["o"], **TOL_STATE)
    _check("final_state", _np(final[:1]), want["final_state"], **TOL_STATE)


@pytest.mark.parametrize("path", PATHS)
def test_replay_is_bitwise_deterministic(path):
    inp = _cuda(make_inputs(WORKLOADS["varlen_16k"], varlen_total=4096, Hq=8, Hv=8))
    first = _ours(inp, inter=True, path=path)
    for _ in range(3):
        again = _ours(inp, inter=True, path=path)
        assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])
        for key in first[2]:
            assert torch.equal(first[2][key], again[2][key]), key


@pytest.mark.parametrize("path", PATHS)
def test_two_streams_give_identical_results(path):
    a = _cuda(make_inputs(WORKLOADS["mha_1k"], seed=11, B=1, Hq=16, Hv=16))
    b = _cuda(make_inputs(WORKLOADS["gva_4k"], seed=12, T=1024, Hq=4, Hv=16))
    ref_a, ref_b = _ours(a, path=path), _ours(b, path=path)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        out_a = _ours(a, path=path)
    with torch.cuda.stream(s2):
        out_b = _ours(b, path=path)
    torch.cuda.synchronize()
    assert torch.equal(ref_a[0], out_a[0]) and torch.equal(ref_a[1], out_a[1])
    assert torch.equal(ref_b[0], out_b[0]) and torch.equal(ref_b[1], out_b[1])


@pytest.mark.parametrize("path", PATHS)
def test_poisoned_workspace_does_not_leak(path):
    # every workspace byte starts as a NaN pattern: results must equal a run on
    # a zeroed workspace, bit for bit (nothing reads workspace it did not write)
    inp = _cuda(make_inputs(WORKLOADS["tiny"], seed=5, **SMALL_CASES["varlen"]))
    outs = []
    for fill in (0x00, 0xFF):
        a, (B, T, Hq, Hv, K, V, N) = ops.make_args(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                                   inp["scale"], inp["initial_state"], inp["cu_seqlens"])
        a.path = ops._PATHS[path]
        o = torch.full((B, T, Hv, V), float("nan"), dtype=torch.bfloat16, device="cuda")
        fin = torch.full((N, Hv, K, V), float("nan"), dtype=torch.float32, device="cuda")
        a.o, a.final_state = o.data_ptr(), fin.data_ptr()
        n = _lib.kda_workspace_size(a)
        ws = torch.full((n,), fill, dtype=torch.uint8, device="cuda")
        assert _lib.kda_chunk_fwd(a, ws.data_ptr(), n, torch.cuda.current_stream().cuda_stream) == 0
        torch.cuda.synchronize()
        outs.append((o, fin))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert torch.isfinite(outs[0][0].float()).all() and torch.isfinite(outs[0][1]).all()


@pytest.mark.parametrize("path", PATHS)
def test_continuation_across_calls(path):
    inp = make_inputs(WORKLOADS["mha_1k"], seed=21, B=1, Hq=4, Hv=4, initial_state=True)
    full = _ours(_cuda(inp), inter=False, path=path)
    T1 = 384 + 17
    seq = ("q", "k", "v", "g", "beta")
    first = {k: (v[:, :T1] if k in seq else v) for k, v in inp.items()}
    second = {k: (v[:, T1:] if k in seq else v) for k, v in inp.items()}
    first["T"], second["T"] = T1, inp["T"] - T1
    r1 = _ours(_cuda(first), inter=False, path=path)
    second["initial_state"] = r1[1].cpu()
    r2 = _ours(_cuda(second), inter=False, path=path)
    _check("o", _np(r2[0]), _np(full[0])[:, T1:], **TOL_STATE)
    _check("final_state", _np(r2[1]), _np(full[1]), **TOL_STATE)
