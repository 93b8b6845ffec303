"""Write the stored oracle values for the small forward case.

Calls only the oracle (and the seeded input generator).  Case: forward,
non-causal MHA, B=1, H=2, Hkv=2, L=128, D=64, fp16 inputs drawn from
N(0, 1) with seed 0, scale 1/sqrt(64) -- the smallest configuration the
pages' forward kernel is written for (one 128-row tile per head).

Run from the repository root:  python tests/golden/make_golden.py
"""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import fa_oracle as orc  # noqa: E402
from tiled_attention_fa_gb300.inputs import make_qkv  # noqa: E402


def main():
    q, k, v, _ = make_qkv(1, 128, 2, 2, 64, "fp16", seed=0, with_do=False)
    o, lse = orc.forward(q.double().numpy(), k.double().numpy(), v.double().numpy(), False)
    rows = []
    for h in range(2):
        for i in (0, 1, 63, 64, 127):
            rows.append({"h": h, "i": i, "o": [float(x) for x in o[0, i, h]],
                         "lse": float(lse[0, h, i])})
    out = {
        "case": "forward non-causal B1 H2 Hkv2 L128 D64 fp16 seed0",
        "source": "oracle/fa_oracle.py forward(); inputs tiled_attention_fa_gb300/inputs.py make_qkv",
        "rows": rows,
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "fwd_b1_h2_l128_d64_seed0.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
