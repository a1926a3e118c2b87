"""Write tests/golden/tiny_oracle_digest.json from the FP64 oracle alone.

The pages print no worked values (their golden test keeps "output digests" of
the removed native kernels, cuLA PR #131), so this fixture is a digest of the
oracle's own outputs on the seeded tiny workload (B=1, H=2, T=256 = four
chunks of 64, K=V=64, fp32 beta, zero initial state): it pins the oracle and
the input recipe against silent change.  Run from the repository root:

    python tests/golden/make_golden.py
"""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from chunked_gated_delta_03_gb300.workloads import WORKLOADS, make_inputs  # noqa: E402
from oracle import kda_ref as ref  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle_digest.json")
KEYS = ("o", "final_state", "Aqk", "Akk", "Akk_inv", "W", "U", "G", "QG")


def digest():
    inp = make_inputs(WORKLOADS["tiny"])
    f64 = lambda t: t.double().numpy()
    out = ref.kda_chunked(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["g"]), f64(inp["beta"]),
                          inp["scale"], None, None, chunk_size=64)
    d = {"workload": "tiny: B=1 H=2 T=256 K=V=64, fp32 beta, zero initial state, default seed"}
    for key in KEYS:
        x = out[key]
        d[key] = {
            "shape": list(x.shape),
            "sum": float(x.sum()),
            "l2": float((x ** 2).sum() ** 0.5),
            "first": [float(v) for v in x.reshape(-1)[:8]],
            "last": [float(v) for v in x.reshape(-1)[-8:]],
        }
    return d


if __name__ == "__main__":
    with open(OUT, "w") as f:
        json.dump(digest(), f, indent=1)
    print("wrote", OUT)
