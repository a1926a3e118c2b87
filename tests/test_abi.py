"""The C ABI without compute: the library loads, exports what include/kda.h
declares, and rejects bad arguments on the host before touching a GPU."""

import ctypes
import os
import re
import subprocess

import pytest

from chunked_gated_delta_03_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert _declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_struct_layout_matches_header(tmp_path):
    # compile a probe against include/kda.h and compare every field offset
    fields = [f[0] for f in _lib.KdaArgs._fields_]
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "kda.h"', "int main(void) {",
             '  printf("%zu\\n", sizeof(KdaArgs));']
    lines += [f'  printf("%zu\\n", offsetof(KdaArgs, {f}));' for f in fields]
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(_lib.KdaArgs)
    assert got[1:] == [getattr(_lib.KdaArgs, f).offset for f in fields]


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -16, -17, -18, -19):
        s = _lib.status_string(code)
        assert s and s != "unknown status"
    assert _lib.status_string(12345) == "unknown status"


def _args(**kw):
    a = _lib.KdaArgs()
    base = 1 << 20  # 16-byte aligned dummy addresses; never dereferenced on the host path
    a.q, a.k, a.v, a.g, a.beta, a.o = base, base, base, base, base, base
    a.B, a.T, a.Hq, a.Hv, a.K, a.V, a.chunk = 1, 128, 2, 2, 64, 64, 64
    a.scale = 0.125
    for key, val in kw.items():
        setattr(a, key, val)
    return a


@pytest.mark.parametrize("kw, code", [
    (dict(chunk=0), _lib.KDA_ERR_INVALID),
    (dict(chunk=-64), _lib.KDA_ERR_INVALID),
    (dict(chunk=32), _lib.KDA_ERR_UNSUPPORTED),
    (dict(K=96), _lib.KDA_ERR_UNSUPPORTED),
    (dict(V=256), _lib.KDA_ERR_UNSUPPORTED),
    (dict(Hv=3), _lib.KDA_ERR_INVALID),          # Hv % Hq != 0
    (dict(B=0), _lib.KDA_ERR_INVALID),
    (dict(T=-1), _lib.KDA_ERR_INVALID),
    (dict(beta_dtype=7), _lib.KDA_ERR_INVALID),
    (dict(q=0), _lib.KDA_ERR_INVALID),
    (dict(o=0), _lib.KDA_ERR_INVALID),
    (dict(q=(1 << 20) + 8), _lib.KDA_ERR_MISALIGNED),
    (dict(QG=(1 << 20) + 4), _lib.KDA_ERR_MISALIGNED),   # the optional gated-query output
    (dict(cu_seqlens=1 << 20, B=2, N=1), _lib.KDA_ERR_INVALID),  # varlen needs B == 1
])
def test_chunk_fwd_rejects_bad_arguments(lib, kw, code):
    a = _args(**kw)
    ws_bytes = 1 << 30
    assert _lib.kda_chunk_fwd(a, 1 << 24, ws_bytes, 0) == code


def test_workspace_checks(lib):
    a = _args()
    need = _lib.kda_workspace_size(a)
    assert need > 0 and need % 256 == 0
    assert _lib.kda_chunk_fwd(a, 1 << 24, need - 1, 0) == _lib.KDA_ERR_WORKSPACE
    assert _lib.kda_chunk_fwd(a, (1 << 24) + 128, need, 0) == _lib.KDA_ERR_MISALIGNED
    assert _lib.kda_chunk_fwd(a, 0, need, 0) == _lib.KDA_ERR_INVALID
    assert _lib.kda_workspace_size(_args(K=96)) == 0


def test_two_pass_workspace_accounts_for_missing_w_u(lib):
    two = dict(path=_lib.KDA_PATH_TWO_PASS)
    with_wu = _args(W=1 << 20, U=1 << 20, **two)
    without = _args(**two)
    # the two-pass state kernel reads W and U: without caller buffers they live in the workspace
    assert _lib.kda_workspace_size(without) - _lib.kda_workspace_size(with_wu) >= 2 * 128 * 2 * 64 * 2


def test_fused_workspace_is_the_header_flags_and_the_sequence_order(lib):
    # the fused path keeps every state-pass operand on chip: the workspace holds
    # the 256-byte status header, the per-chain flags of the exact path (one
    # int32 per (sequence, value head), rounded up to 256 bytes) and, in varlen
    # mode, the longest-first sequence order (one int32 per sequence, rounded up)
    up = lambda n: (n + 255) // 256 * 256
    assert _lib.kda_workspace_size(_args()) == 256 + up(1 * 2 * 4)
    assert _lib.kda_workspace_size(_args(path=_lib.KDA_PATH_FUSED, T=1 << 20, Hv=64, Hq=64)) == 256 + up(64 * 4)
    # varlen, N = 100: the fused forward needs header + flags + order;
    # kda_workspace_size also covers kda_fwd_intra on the same arguments, whose
    # chunk table takes (T/64 + N) pairs and N + 1 offsets
    varlen = _args(cu_seqlens=1 << 20, N=100)
    fused = 256 + up(100 * 2 * 4) + up(100 * 4)
    intra = 256 + up(100 * 2 * 4) + up((128 // 64 + 100) * 2 * 4) + up(101 * 4)
    assert _lib.kda_workspace_size(varlen) == max(fused, intra)
    assert _lib.kda_chunk_fwd(varlen, 1 << 24, fused - 1, 0) == _lib.KDA_ERR_WORKSPACE
    iargs = _args(cu_seqlens=1 << 20, N=100, Aqk=1 << 20, Akk_inv=1 << 20, W=1 << 20, U=1 << 20)
    assert _lib.kda_fwd_intra(iargs, 1 << 24, intra - 1, 0) == _lib.KDA_ERR_WORKSPACE


def test_workspace_size_ignores_optional_exports_and_precision(lib):
    # QG and the TF32 option change what the intra kernel writes and how it
    # forms Aqk / Akk, not the two-pass workspace; with the automatic path the
    # TF32 option selects the two-pass kernels, which need more
    two = dict(path=_lib.KDA_PATH_TWO_PASS)
    base = _lib.kda_workspace_size(_args(**two))
    assert _lib.kda_workspace_size(_args(QG=1 << 20, **two)) == base
    assert _lib.kda_workspace_size(_args(intra_tf32=1, **two)) == base
    assert _lib.kda_workspace_size(_args(intra_tf32=1)) == base
    assert _lib.kda_workspace_size(_args(QG=1 << 20)) == _lib.kda_workspace_size(_args())


@pytest.mark.parametrize("kw, code", [
    (dict(path=7), _lib.KDA_ERR_INVALID),
    (dict(path=_lib.KDA_PATH_FUSED, intra_tf32=1), _lib.KDA_ERR_UNSUPPORTED),
    (dict(cu_seqlens=1 << 20, N=2, chunk_indices=1 << 20), _lib.KDA_ERR_INVALID),     # table without offsets
    (dict(cu_seqlens=1 << 20, N=2, chunk_offsets=1 << 20), _lib.KDA_ERR_INVALID),     # offsets without table
    (dict(cu_seqlens=1 << 20, N=2, chunk_indices=(1 << 20) + 2, chunk_offsets=1 << 20), _lib.KDA_ERR_MISALIGNED),
])
def test_path_and_chunk_table_arguments(lib, kw, code):
    a = _args(**kw)
    assert _lib.kda_chunk_fwd(a, 1 << 24, 1 << 30, 0) == code


def test_intra_requires_its_outputs(lib):
    a = _args()
    assert _lib.kda_fwd_intra(a, 1 << 24, 1 << 30, 0) == _lib.KDA_ERR_INVALID


def test_prepare_chunk_indices_rejects_bad_chunk(lib):
    for chunk in (0, -64):
        assert _lib.kda_prepare_chunk_indices(1 << 20, 1, 4, chunk, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 0) \
            == _lib.KDA_ERR_INVALID


def test_context_parallel_arguments(lib):
    # intra-card context parallelism needs fixed-length input, K == V, the
    # fused path and no TF32 option; its workspace adds the segment buffers
    long = dict(T=64 * 40, Hq=2, Hv=2, K=64, V=64)
    base = _lib.kda_workspace_size(_args(**long))
    cp = _lib.kda_workspace_size(_args(cp_chunks=8, **long))
    nseg, bt = 5, 64 * 40
    assert cp >= base + 3 * nseg * 2 * 64 * 64 * 4 + 2 * bt * 2 * 64 * 2
    # one segment covers the whole sequence: the plain forward and its workspace
    assert _lib.kda_workspace_size(_args(cp_chunks=40, **long)) == base
    for kw, code in ((dict(cp_chunks=-1), _lib.KDA_ERR_INVALID),
                     (dict(cp_chunks=8, V=128), _lib.KDA_ERR_UNSUPPORTED),
                     (dict(cp_chunks=8, path=_lib.KDA_PATH_TWO_PASS), _lib.KDA_ERR_UNSUPPORTED),
                     (dict(cp_chunks=8, intra_tf32=1), _lib.KDA_ERR_UNSUPPORTED),
                     (dict(cp_chunks=8, cu_seqlens=1 << 20, N=3), _lib.KDA_ERR_UNSUPPORTED)):
        args = dict(long)
        args.update(kw)
        assert _lib.kda_chunk_fwd(_args(**args), 1 << 24, 1 << 30, 0) == code, kw
        if code == _lib.KDA_ERR_UNSUPPORTED or kw.get("cp_chunks", 0) < 0:
            assert _lib.kda_workspace_size(_args(**args)) == 0, kw
