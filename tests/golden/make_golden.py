"""Write tests/golden/prefill_small.json from the fp64 oracle.

The pages print no worked numeric example, so this fixture pins the oracle to
its own earlier output (a regression guard): inputs are drawn from a fixed
seed, and the expected output comes from ``oracle.prefill`` only.  Re-run only
when a change to the oracle's arithmetic is justified by a reading of the page
"Gated MLA（矩阵吸收版）", and say which in the commit message.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402


def main():
    rng = np.random.default_rng(20260)
    B, T, H, dq, dv, r = 2, 6, 2, 3, 4, 5
    q = rng.standard_normal((B, T, H, dq)).round(6)
    c = rng.standard_normal((B, T, r)).round(6)
    w_uk = (rng.standard_normal((H, dq, r)) * 0.5).round(6)
    w_uv = (rng.standard_normal((H, dv, r)) * 0.5).round(6)
    gate = rng.standard_normal((B, T, H * dv)).round(6)
    scale = 0.75
    out = oracle.prefill(q, c, w_uk, w_uv, gate, scale)
    fx = dict(note="toy causal absorbed Gated-MLA case; expected output written by oracle.prefill",
              scale=scale, q=q.tolist(), c=c.tolist(), w_uk=w_uk.tolist(), w_uv=w_uv.tolist(),
              gate=gate.tolist(), out=out.tolist())
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "prefill_small.json")
    with open(path, "w") as f:
        json.dump(fx, f, indent=None)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
