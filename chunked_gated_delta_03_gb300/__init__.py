"""Chunked KDA (Kimi Delta Attention) forward for GB300 (sm_103a).

The computation lives in hand-written CUDA kernels behind the C ABI of
include/kda.h (libkda.so, built by ``build.build()``); ``ops`` is a thin
PyTorch front end and ``_lib`` the ctypes binding.
"""

from .ops import (KdaError, chunk_kda_fwd, chunk_kda_fwd_intra, device_status, prepare_chunk_indices,
                  prepare_chunk_indices_device)

__all__ = ["chunk_kda_fwd", "chunk_kda_fwd_intra", "prepare_chunk_indices", "prepare_chunk_indices_device",
           "device_status", "KdaError"]
