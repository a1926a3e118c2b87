"""PyTorch front end of libkda: allocate outputs and workspace, pass pointers.

Every step of the computation runs in the CUDA kernels behind include/kda.h;
this module only checks dtypes and shapes, makes inputs contiguous (as the
pages' intra entry point does before dispatch, cuLA PR #131 review of
intra_fused.py) and marshals pointers and the current CUDA stream.
"""

from __future__ import annotations

import torch

from . import _lib
from ._lib import KdaArgs, KdaError

__all__ = ["chunk_kda_fwd", "chunk_kda_fwd_intra", "prepare_chunk_indices", "prepare_chunk_indices_device",
           "device_status", "KdaError"]

_CHUNK = 64


def _ptr(t):
    return 0 if t is None else t.data_ptr()


def _check_inputs(q, k, v, g, beta, cu_seqlens, initial_state):
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    dev = q.device
    for name, t in (("k", k), ("v", v), ("g", g), ("beta", beta), ("cu_seqlens", cu_seqlens),
                    ("initial_state", initial_state)):
        if t is None:
            continue
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, q on {dev}: all tensors must be on one device")
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise ValueError("q, k, v must be bfloat16")
    if g.dtype != torch.float32:
        raise ValueError("g must be float32")
    if beta.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("beta must be bfloat16 or float32")
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4:
        raise ValueError("q, k must be [B, T, Hq, K] and v [B, T, Hv, V]")
    B, T, Hq, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    if v.shape[:2] != (B, T) or tuple(g.shape) != (B, T, Hv, K) or tuple(beta.shape) != (B, T, Hv):
        raise ValueError("v [B,T,Hv,V], g [B,T,Hv,K] and beta [B,T,Hv] must match q [B,T,Hq,K]")
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1:
            raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
        if B != 1:
            raise ValueError("packed varlen inputs need B == 1")
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else B
    if initial_state is not None:
        if initial_state.dtype != torch.float32 or tuple(initial_state.shape) != (N, Hv, K, V):
            raise ValueError(f"initial_state must be float32 [{N}, {Hv}, {K}, {V}]")
    return B, T, Hq, Hv, K, V, N


_PATHS = {"auto": _lib.KDA_PATH_AUTO, "fused": _lib.KDA_PATH_FUSED, "two_pass": _lib.KDA_PATH_TWO_PASS}


def make_args(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None):
    """Fill a KdaArgs with the input pointers and sizes (outputs left NULL)."""
    B, T, Hq, Hv, K, V, N = _check_inputs(q, k, v, g, beta, cu_seqlens, initial_state)
    a = KdaArgs()
    a.q, a.k, a.v, a.g, a.beta = _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta)
    a.beta_dtype = _lib.KDA_DTYPE_FP32 if beta.dtype == torch.float32 else _lib.KDA_DTYPE_BF16
    a.cu_seqlens = _ptr(cu_seqlens)
    a.N = N if cu_seqlens is not None else 0
    a.B, a.T, a.Hq, a.Hv, a.K, a.V = B, T, Hq, Hv, K, V
    a.chunk = _CHUNK
    a.scale = float(K ** -0.5 if scale is None else scale)
    a.initial_state = _ptr(initial_state)
    return a, (B, T, Hq, Hv, K, V, N)


def _contig(*ts):
    return [None if t is None else t.contiguous() for t in ts]


def chunk_kda_fwd(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
                  output_final_state=True, return_intermediates=False, return_G=False, return_QG=False,
                  tf32=False, path="auto", chunk_table=None, cp_chunks=0):
    """Chunked KDA forward.  Returns (o, final_state, intermediates).

    ``intermediates`` is None unless ``return_intermediates`` (then a dict with
    Aqk, Akk_inv [B,T,Hv,64] fp32 and W [B,T,Hv,K], U [B,T,Hv,V] bf16) or
    ``return_G`` (adds G [B,T,Hv,K] fp32) or ``return_QG`` (adds the gated
    query QG = q * e^G [B,T,Hv,K] bf16).  ``tf32`` selects the single-pass
    TF32 intra-chunk products (faster; Akk_inv near 5e-5 instead of 1e-6
    relative L2).  ``final_state`` is None unless
    ``output_final_state``.  ``path`` picks the kernels: "auto", "fused" (one
    kernel, each (sequence, head) chain on one SM) or "two_pass" (intra-chunk
    kernel, then the state/output kernel).  ``chunk_table`` = (indices,
    offsets) from ``prepare_chunk_indices`` reuses a varlen chunk table instead
    of building it again on the device.  ``cp_chunks`` = n > 0 cuts every
    sequence into segments of n chunks that run as chains of their own (intra-card
    context parallelism: three passes and a scan over the segments; fixed-length
    input with K == V only), for batches with far fewer chains than SMs.
    """
    if path not in _PATHS:
        raise ValueError(f"path must be one of {sorted(_PATHS)}")
    q, k, v, g, beta, cu_seqlens, initial_state = _contig(q, k, v, g, beta, cu_seqlens, initial_state)
    a, (B, T, Hq, Hv, K, V, N) = make_args(q, k, v, g, beta, scale, initial_state, cu_seqlens)
    a.path = _PATHS[path]
    a.cp_chunks = int(cp_chunks)
    dev = q.device
    if chunk_table is not None:
        idx, off = (t.contiguous() for t in chunk_table)
        for name, t in (("chunk indices", idx), ("chunk offsets", off)):
            if t.dtype != torch.int32 or not t.is_cuda or t.device != dev:
                raise ValueError(f"{name} must be int32 CUDA tensors on {dev}")
        a.chunk_indices, a.chunk_offsets = idx.data_ptr(), off.data_ptr()
    o = torch.empty(B, T, Hv, V, dtype=torch.bfloat16, device=dev)
    final = torch.empty(N, Hv, K, V, dtype=torch.float32, device=dev) if output_final_state else None
    inter = {} if (return_intermediates or return_G or return_QG) else None
    if return_intermediates:
        inter["Aqk"] = torch.empty(B, T, Hv, _CHUNK, dtype=torch.float32, device=dev)
        inter["Akk_inv"] = torch.empty(B, T, Hv, _CHUNK, dtype=torch.float32, device=dev)
        inter["W"] = torch.empty(B, T, Hv, K, dtype=torch.bfloat16, device=dev)
        inter["U"] = torch.empty(B, T, Hv, V, dtype=torch.bfloat16, device=dev)
    if return_G:
        inter["G"] = torch.empty(B, T, Hv, K, dtype=torch.float32, device=dev)
    if return_QG:
        inter["QG"] = torch.empty(B, T, Hv, K, dtype=torch.bfloat16, device=dev)
    a.o, a.final_state = _ptr(o), _ptr(final)
    a.intra_tf32 = 1 if tf32 else 0
    if inter:
        a.Aqk, a.Akk_inv = _ptr(inter.get("Aqk")), _ptr(inter.get("Akk_inv"))
        a.W, a.U, a.G = _ptr(inter.get("W")), _ptr(inter.get("U")), _ptr(inter.get("G"))
        a.QG = _ptr(inter.get("QG"))
    ws_bytes = _lib.kda_workspace_size(a)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = _lib.kda_chunk_fwd(a, ws.data_ptr(), ws_bytes, torch.cuda.current_stream(dev).cuda_stream)
    if rc != _lib.KDA_OK:
        raise KdaError(rc, "kda_chunk_fwd")
    return o, final, inter


def chunk_kda_fwd_intra(q, k, v, g, beta, scale=None, cu_seqlens=None, return_G=False, return_QG=False,
                        tf32=False):
    """The standalone intra-chunk primitive: dict with Aqk, Akk_inv, W, U (and G, QG)."""
    q, k, v, g, beta, cu_seqlens = _contig(q, k, v, g, beta, cu_seqlens)
    a, (B, T, Hq, Hv, K, V, N) = make_args(q, k, v, g, beta, scale, None, cu_seqlens)
    dev = q.device
    out = {
        "Aqk": torch.empty(B, T, Hv, _CHUNK, dtype=torch.float32, device=dev),
        "Akk_inv": torch.empty(B, T, Hv, _CHUNK, dtype=torch.float32, device=dev),
        "W": torch.empty(B, T, Hv, K, dtype=torch.bfloat16, device=dev),
        "U": torch.empty(B, T, Hv, V, dtype=torch.bfloat16, device=dev),
    }
    if return_G:
        out["G"] = torch.empty(B, T, Hv, K, dtype=torch.float32, device=dev)
    if return_QG:
        out["QG"] = torch.empty(B, T, Hv, K, dtype=torch.bfloat16, device=dev)
    a.Aqk, a.Akk_inv, a.W, a.U = (_ptr(out[n]) for n in ("Aqk", "Akk_inv", "W", "U"))
    a.G = _ptr(out.get("G"))
    a.QG = _ptr(out.get("QG"))
    a.intra_tf32 = 1 if tf32 else 0
    ws_bytes = _lib.kda_workspace_size(a)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = _lib.kda_fwd_intra(a, ws.data_ptr(), ws_bytes, torch.cuda.current_stream(dev).cuda_stream)
    if rc != _lib.KDA_OK:
        raise KdaError(rc, "kda_fwd_intra")
    return out


def _check_chunk_size(chunk_size):
    # cuLA PR #135 (review of the index tests): a chunk size of None, zero or
    # below zero is rejected with ValueError.
    if chunk_size is None or isinstance(chunk_size, bool) or not isinstance(chunk_size, int) or chunk_size <= 0:
        raise ValueError("chunk_size must be a positive integer")


def prepare_chunk_indices_device(cu_seqlens, T, chunk_size=_CHUNK):
    """Varlen chunk table built on the device, with no device-to-host read.

    Returns (indices [T // chunk + N, 2], offsets [N+1], num_chunks [1],
    status [1]), all int32 on the device; rows of ``indices`` at or past
    num_chunks are unspecified, and status is nonzero for a bad cu_seqlens.
    """
    _check_chunk_size(chunk_size)
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
    cu = cu_seqlens.contiguous()
    N = cu.numel() - 1
    if N < 0:
        raise ValueError("cu_seqlens needs at least one entry")
    dev = cu.device
    idx = torch.empty(max(int(T) // chunk_size + N, 1), 2, dtype=torch.int32, device=dev)
    off = torch.empty(N + 1, dtype=torch.int32, device=dev)
    nc = torch.zeros(1, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        rc = _lib.kda_prepare_chunk_indices(cu.data_ptr(), N, int(T), chunk_size, idx.data_ptr(), off.data_ptr(),
                                            nc.data_ptr(), status.data_ptr(),
                                            torch.cuda.current_stream(dev).cuda_stream)
    if rc != _lib.KDA_OK:
        raise KdaError(rc, "kda_prepare_chunk_indices")
    return idx, off, nc, status


def prepare_chunk_indices(cu_seqlens, chunk_size=_CHUNK):
    """(indices [num_chunks, 2], offsets [N+1]) int32; reads the chunk count back.

    Raises ValueError for a bad chunk size or a cu_seqlens that does not start
    at 0 or decreases somewhere (cuLA PR #135, cula/ops/kda/index.py review).
    """
    _check_chunk_size(chunk_size)
    T = int(cu_seqlens[-1].item())
    idx, off, nc, status = prepare_chunk_indices_device(cu_seqlens, T, chunk_size)
    st = int(status.item())
    if st != _lib.KDA_OK:
        raise ValueError(f"invalid cu_seqlens: {_lib.status_string(st)}")
    return idx[: int(nc.item())], off


def device_status(workspace: torch.Tensor) -> int:
    """Status word of a workspace after the work queued on the current stream."""
    with torch.cuda.device(workspace.device):
        return _lib.kda_get_device_status(workspace.data_ptr(),
                                          torch.cuda.current_stream(workspace.device).cuda_stream)
