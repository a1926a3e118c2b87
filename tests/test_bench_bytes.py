"""The byte and FLOP counts behind bench.py's roofline fractions, recomputed by hand.

mha_8k (B=2, H=64, T=8192, K=V=128, fp32 beta, Aqk/Akk_inv/W/U exported) has
2 x 128 chunks x 64 heads = 16384 chunk-heads of 64 token rows.  The method
reads, per chunk-head, q, k, v (64 x 128 bf16 each), g (64 x 128 fp32) and beta
(64 fp32), and writes o (64 x 128 bf16) and the four exports Aqk, Akk_inv
(64 x 64 fp32 each), W, U (64 x 128 bf16 each), plus one final state
(128 x 128 fp32) per (sequence, head).  That is the path's minimum, and what
the fused kernel moves.  The two-pass design adds its own traffic on top: the
state-pass operands Qs, Kl (64 x 128 bf16 each), the bf16 copy of Aqk (64 x 64)
and gamma (128 fp32), written by the intra kernel and read back by the state
kernel together with W and U.  The roofline fraction counts the method's bytes
only; the design traffic is reported beside it.
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
    exports = 2 * 64 * 64 * 4 + 2 * tile16      # Aqk, Akk_inv (fp32), W, U (bf16)
    final = 2 * 64 * 128 * 128 * 4
    path = units * (reads + tile16 + exports) + final
    assert got["path"] == path == 2_696_937_472
    assert got["fused"] == path
    # the two-pass kernels: the method's bytes each moves, and the design's own
    assert got["intra"] == units * (reads + exports)
    assert got["state"] == units * tile16 + final
    handoff = units * (2 * tile16 + 64 * 64 * 2 + 128 * 4)   # Qs, Kl, Aqk bf16, gamma
    assert got["intra_design"] == handoff
    assert got["state_design"] == handoff + units * 2 * tile16   # and W, U read back
    # measured round-trip overhead of the two-pass design: 1.27x on the intra kernel
    assert 1.26 < (got["intra"] + got["intra_design"]) / got["intra"] < 1.29


def test_bf16_beta_and_no_exports():
    # mha_1k: bf16 beta, no exports: the two-pass design keeps W and U in the workspace
    w = _workload(2, 1024, 64, 64, 128, 128, torch.bfloat16, False)
    got = bench.algorithmic_bytes(w, N=2)
    units = 2 * 16 * 64
    tile16 = 64 * 128 * 2
    reads = 3 * tile16 + 64 * 128 * 4 + 64 * 2
    assert got["path"] == got["fused"] == units * (reads + tile16) + 2 * 64 * 128 * 128 * 4
    assert got["intra_design"] == units * (2 * tile16 + 2 * tile16 + 64 * 64 * 2 + 128 * 4)


def test_flops_match_the_hand_count():
    # per chunk-head: Aqk, Akk, W (64 x 64 x 128 each), U (64 x 64 x 128),
    # W S and Qg S (64 x 128 x 128 each), Aqk Delta (64 x 64 x 128), K^T Delta
    # (128 x 64 x 128); two FLOPs per multiply-add
    w = _workload(2, 8192, 64, 64, 128, 128, torch.float32, True)
    macs = 4 * 64 * 64 * 128 + 2 * 64 * 128 * 128 + 64 * 64 * 128 + 128 * 64 * 128
    assert bench.algorithmic_flops(w) == 16384 * 2 * macs == 188_978_561_024
