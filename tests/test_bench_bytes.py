"""The byte counts behind bench.py's roofline fractions, recomputed by hand.

mha_8k (B=2, H=64, T=8192, K=V=128, fp32 beta, Aqk/Akk_inv/W/U exported) has
2 x 128 chunks x 64 heads = 16384 chunk-heads of 64 token rows.  Per
chunk-head the intra kernel reads q, k, v (64 x 128 bf16 each), g (64 x 128
fp32) and beta (64 fp32), and writes Aqk, Akk_inv (64 x 64 fp32 each), W, U
(64 x 128 bf16 each) and the state-pass operands Qs, Kl (64 x 128 bf16 each),
the bf16 copy of Aqk (64 x 64) and gamma (128 fp32).  The state kernel reads
W, U, Qs, Kl, the bf16 Aqk and gamma and writes o (64 x 128 bf16), plus one
final state (128 x 128 fp32) per (sequence, head).
"""

import torch

import bench


def _workload(B, T, Hq, Hv, K, V, beta_dtype, intermediates, h0=False, cu=None):
    return {"B": B, "T": T, "Hq": Hq, "Hv": Hv, "K": K, "V": V,
            "beta": torch.empty(0, dtype=beta_dtype), "cu_seqlens": cu,
            "initial_state": torch.empty(0) if h0 else None, "intermediates": intermediates}


def test_mha_8k_bytes_match_the_hand_count():
    w = _workload(2, 8192, 64, 64, 128, 128, torch.float32, True)
    got = bench.algorithmic_bytes(w, N=2)
    units = 2 * 128 * 64
    tile16 = 64 * 128 * 2                       # 64 rows x 128 channels, bf16
    reads = 3 * tile16 + 64 * 128 * 4 + 64 * 4  # q, k, v, g, beta
    writes = 2 * 64 * 64 * 4 + 2 * tile16 + 2 * tile16 + 64 * 64 * 2 + 128 * 4
    assert reads + writes == 189_184
    assert got["intra"] == units * (reads + writes) == 3_099_590_656
    state = units * (4 * tile16 + 64 * 64 * 2 + 128 * 4 + tile16) + 2 * 64 * 128 * 128 * 4
    assert got["state"] == state
    # the path minimum: inputs once, o and the final state, the four exports
    path = units * (reads + tile16 + 2 * 64 * 64 * 4 + 2 * tile16) + 2 * 64 * 128 * 128 * 4
    assert got["path"] == path == 2_696_937_472


def test_bf16_beta_and_no_exports():
    # mha_1k: bf16 beta, W and U kept in the workspace for the state pass
    w = _workload(2, 1024, 64, 64, 128, 128, torch.bfloat16, False)
    got = bench.algorithmic_bytes(w, N=2)
    units = 2 * 16 * 64
    tile16 = 64 * 128 * 2
    reads = 3 * tile16 + 64 * 128 * 4 + 64 * 2
    writes = 2 * tile16 + 2 * tile16 + 64 * 64 * 2 + 128 * 4   # W, U (workspace), Qs, Kl, Aqk bf16, gamma
    assert got["intra"] == units * (reads + writes)
    assert got["path"] == units * (reads + tile16) + 2 * 64 * 128 * 128 * 4
