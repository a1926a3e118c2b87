"""ctypes binding of libkda.so (include/kda.h).  Argument marshalling only.

The names mirror the C entry points.  Loading fails loudly when the shared
object has not been built: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os

from .build import LIB

KDA_OK = 0
KDA_ERR_INVALID = -1
KDA_ERR_UNSUPPORTED = -2
KDA_ERR_MISALIGNED = -3
KDA_ERR_ARCH = -4
KDA_ERR_LAUNCH = -5
KDA_ERR_WORKSPACE = -6
KDA_ERR_BAD_SEQLENS = -16
KDA_ERR_TIMEOUT = -17
KDA_ERR_GATE_RANGE = -18
KDA_ERR_BAD_CHUNK_TABLE = -19
KDA_MAX_CHUNK_LOG_DECAY = 60.0
KDA_DTYPE_BF16 = 0
KDA_DTYPE_FP32 = 1
KDA_PATH_AUTO = 0
KDA_PATH_FUSED = 1
KDA_PATH_TWO_PASS = 2

EXPORTS = ("kda_workspace_size", "kda_chunk_fwd", "kda_fwd_intra", "kda_prepare_chunk_indices",
           "kda_get_device_status", "kda_status_string", "kda_chunk_fwd_static_scratch", "kda_check_bounded_wait")
KDA_STATIC_SCRATCH_BYTES = 64 << 20


class KdaArgs(ctypes.Structure):
    """Mirror of ``struct KdaArgs`` in include/kda.h (same field order and types)."""

    _fields_ = [
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("g", ctypes.c_void_p),
        ("beta", ctypes.c_void_p),
        ("beta_dtype", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p),
        ("N", ctypes.c_int32),
        ("B", ctypes.c_int32),
        ("T", ctypes.c_int32),
        ("Hq", ctypes.c_int32),
        ("Hv", ctypes.c_int32),
        ("K", ctypes.c_int32),
        ("V", ctypes.c_int32),
        ("chunk", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("initial_state", ctypes.c_void_p),
        ("o", ctypes.c_void_p),
        ("final_state", ctypes.c_void_p),
        ("Aqk", ctypes.c_void_p),
        ("Akk_inv", ctypes.c_void_p),
        ("W", ctypes.c_void_p),
        ("U", ctypes.c_void_p),
        ("G", ctypes.c_void_p),
        ("profile_events", ctypes.c_void_p),
        ("QG", ctypes.c_void_p),
        ("intra_tf32", ctypes.c_int32),
        ("path", ctypes.c_int32),
        ("chunk_indices", ctypes.c_void_p),
        ("chunk_offsets", ctypes.c_void_p),
        ("cp_chunks", ctypes.c_int32),
    ]


class KdaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


_lib = None


def load():
    """Load libkda.so once; raise if it is missing (no CPU fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise RuntimeError(f"{LIB} is missing: build it with chunked_gated_delta_03_gb300.build.build()")
    lib = ctypes.CDLL(LIB)
    P = ctypes.POINTER(KdaArgs)
    lib.kda_workspace_size.argtypes = [P]
    lib.kda_workspace_size.restype = ctypes.c_size_t
    for name in ("kda_chunk_fwd", "kda_fwd_intra"):
        f = getattr(lib, name)
        f.argtypes = [P, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        f.restype = ctypes.c_int
    lib.kda_prepare_chunk_indices.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p]
    lib.kda_prepare_chunk_indices.restype = ctypes.c_int
    lib.kda_get_device_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
    lib.kda_get_device_status.restype = ctypes.c_int
    lib.kda_chunk_fwd_static_scratch.argtypes = [P, ctypes.c_void_p, ctypes.c_void_p]
    lib.kda_chunk_fwd_static_scratch.restype = ctypes.c_int
    lib.kda_check_bounded_wait.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.kda_check_bounded_wait.restype = ctypes.c_int
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().kda_status_string(int(code)).decode()


def kda_workspace_size(args: KdaArgs) -> int:
    return int(load().kda_workspace_size(ctypes.byref(args)))


def kda_chunk_fwd(args: KdaArgs, workspace: int, workspace_bytes: int, stream: int) -> int:
    return int(load().kda_chunk_fwd(ctypes.byref(args), workspace, workspace_bytes, stream))


def kda_chunk_fwd_static_scratch(args: KdaArgs, device_status: int, stream: int) -> int:
    """kda_chunk_fwd on the library's fixed device scratch (no workspace, no allocation)."""
    return int(load().kda_chunk_fwd_static_scratch(ctypes.byref(args), device_status, stream))


def kda_fwd_intra(args: KdaArgs, workspace: int, workspace_bytes: int, stream: int) -> int:
    return int(load().kda_fwd_intra(ctypes.byref(args), workspace, workspace_bytes, stream))


def kda_prepare_chunk_indices(cu_seqlens: int, N: int, T: int, chunk: int, chunk_indices: int,
                              chunk_offsets: int, num_chunks: int, status: int, stream: int) -> int:
    return int(load().kda_prepare_chunk_indices(cu_seqlens, N, T, chunk, chunk_indices, chunk_offsets,
                                                num_chunks, status, stream))


def kda_check_bounded_wait(device_status: int, stream: int) -> int:
    """One warp waits on a barrier nothing arrives at; the bounded wait records KDA_ERR_TIMEOUT."""
    return int(load().kda_check_bounded_wait(device_status, stream))


def kda_get_device_status(workspace: int, stream: int) -> int:
    out = ctypes.c_int32(0)
    rc = load().kda_get_device_status(workspace, stream, ctypes.byref(out))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_get_device_status")
    return int(out.value)
