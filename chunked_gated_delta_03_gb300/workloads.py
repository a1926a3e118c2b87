"""Seeded synthetic inputs for the KDA forward pass.

This module only draws random tensors with the shapes and distributions of the
standard workloads; it holds none of KDA's arithmetic.  Both the CUDA path and
the CPU oracle take their inputs from here.

Recipe (per workload, one ``numpy.random.Generator(PCG64(seed))``, drawn in the
order q, k, v, g, beta, initial state):
  * q, k ~ N(0, 1) in fp32, each head vector L2-normalised over K in fp32,
    then rounded to bf16.
  * v ~ N(0, 1), rounded to bf16.
  * g = -softplus(N(0, 1)) / 16 in fp32, one log-gate per value head and
    channel, shape [B, T, Hv, K].
  * beta = sigmoid(N(0, 1)), stored in bf16 or fp32.
  * initial state ~ N(0, 0.02^2) in fp32, shape [N, Hv, K, V], when the
    workload has one; otherwise none (zeros).
  * packed varlen lengths: draw U{1..4096} until the sum reaches the token
    total, cut the last length so the sum is exact, and use the first seed
    >= the workload's seed whose draw holds a length below 64 and a length
    that is not a multiple of 64.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np
import torch

__all__ = ["Workload", "WORKLOADS", "varlen_lengths", "make_inputs"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    Hq: int
    Hv: int
    K: int
    V: int
    beta_dtype: str = "fp32"        # "fp32" or "bf16"
    initial_state: bool = False
    varlen_total: int = 0           # > 0: packed varlen with this many tokens (B = 1)
    varlen_max_len: int = 4096
    intermediates: bool = False     # also return Aqk / Akk_inv / W / U
    seed: int = 0
    lengths: tuple = field(default=())  # explicit packed lengths (tests)

    @property
    def scale(self) -> float:
        return float(self.K) ** -0.5


WORKLOADS = {
    "tiny": Workload("tiny", B=1, T=256, Hq=2, Hv=2, K=64, V=64,
                     beta_dtype="fp32", seed=0),
    "mha_1k": Workload("mha_1k", B=2, T=1024, Hq=64, Hv=64, K=128, V=128,
                       beta_dtype="bf16", seed=1),
    "mha_8k": Workload("mha_8k", B=2, T=8192, Hq=64, Hv=64, K=128, V=128,
                       beta_dtype="fp32", intermediates=True, seed=2),
    "gva_4k": Workload("gva_4k", B=1, T=4096, Hq=16, Hv=64, K=128, V=128,
                       beta_dtype="bf16", initial_state=True, seed=3),
    "varlen_16k": Workload("varlen_16k", B=1, T=16384, Hq=64, Hv=64, K=128, V=128,
                           beta_dtype="bf16", initial_state=True,
                           varlen_total=16384, seed=4),
    # few long chains (8 on a 152-SM GPU): the case intra-card context
    # parallelism is for (cuLA PR #135, intra-card CP)
    "long_16k_h8": Workload("long_16k_h8", B=1, T=16384, Hq=8, Hv=8, K=128, V=128,
                            beta_dtype="bf16", initial_state=True, seed=5),
}


def _draw_lengths(seed: int, total: int, max_len: int) -> list:
    rng = np.random.default_rng(seed)
    lens = []
    while sum(lens) < total:
        lens.append(int(rng.integers(1, max_len + 1)))
    lens[-1] -= sum(lens) - total
    return [x for x in lens if x > 0]


def varlen_lengths(total: int, max_len: int = 4096, seed: int = 0):
    """(seed used, lengths) of a packed varlen draw that has a sub-chunk and a ragged sequence."""
    s = seed
    while True:
        lens = _draw_lengths(s, total, max_len)
        if any(x < 64 for x in lens) and any(x % 64 for x in lens):
            return s, lens
        s += 1


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)


def _l2norm_last(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x.astype(np.float64) ** 2, axis=-1, keepdims=True))
    return (x / np.maximum(n, 1e-12)).astype(np.float32)


def make_inputs(w: Workload, device="cpu", **overrides) -> dict:
    """Draw the inputs of workload ``w`` (fields may be overridden by keyword).

    Returns a dict of torch tensors: q, k, v (bf16), g (fp32), beta (bf16 or
    fp32), initial_state (fp32 or None), cu_seqlens (int32 or None), plus the
    plain ints B, T, Hq, Hv, K, V, N and the float scale.
    """
    if overrides:
        w = replace(w, **overrides)
    cu = None
    if w.lengths:
        lens = list(w.lengths)
        T, B = int(sum(lens)), 1
    elif w.varlen_total:
        _, lens = varlen_lengths(w.varlen_total, w.varlen_max_len, w.seed)
        T, B = w.varlen_total, 1
    else:
        lens, T, B = None, w.T, w.B
    if lens is not None:
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    N = len(lens) if lens is not None else B
    rng = np.random.default_rng(w.seed)
    f32 = np.float32
    q = _l2norm_last(rng.standard_normal((B, T, w.Hq, w.K), dtype=f32))
    k = _l2norm_last(rng.standard_normal((B, T, w.Hq, w.K), dtype=f32))
    v = rng.standard_normal((B, T, w.Hv, w.V), dtype=f32)
    z = rng.standard_normal((B, T, w.Hv, w.K), dtype=f32)
    g = (-np.logaddexp(0.0, z.astype(np.float64)) / 16.0).astype(f32)   # -softplus(z)/16
    zb = rng.standard_normal((B, T, w.Hv), dtype=f32).astype(np.float64)
    beta = (1.0 / (1.0 + np.exp(-zb))).astype(f32)                       # sigmoid
    h0 = None
    if w.initial_state:
        h0 = torch.from_numpy(0.02 * rng.standard_normal((N, w.Hv, w.K, w.V), dtype=f32))
    out = {
        "q": _bf16(q), "k": _bf16(k), "v": _bf16(v),
        "g": torch.from_numpy(g),
        "beta": _bf16(beta) if w.beta_dtype == "bf16" else torch.from_numpy(beta),
        "initial_state": h0,
        "cu_seqlens": cu,
        "B": B, "T": T, "Hq": w.Hq, "Hv": w.Hv, "K": w.K, "V": w.V, "N": N,
        "scale": w.scale,
    }
    if device != "cpu":
        for key, val in list(out.items()):
            if isinstance(val, torch.Tensor):
                out[key] = val.to(device)
    return out
