"""Write tests/golden/tiny_rational.json from the oracle alone.

The pages print no KDA worked example, so this fixture is a regression
guard for the oracle itself: a tiny packed case with exactly representable
inputs (multiples of 1/8, decays alpha in {1/2, 3/4, 1}), its token-recurrence
outputs and final states.  Re-run only when the oracle's arithmetic changes
for a reason that cites the passage or reading behind the change.
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def case():
    rng = np.random.default_rng(2024)
    lens = [3, 1, 4]
    T, H, dk, dv = sum(lens), 2, 4, 3
    eighth = lambda *s: rng.integers(-8, 9, s) / 8.0
    q, k, v = eighth(T, H, dk), eighth(T, H, dk), eighth(T, H, dv)
    alpha = rng.choice([0.5, 0.75, 1.0], (T, H, dk))
    beta = rng.choice([0.0, 0.25, 0.5, 1.0], (T, H))
    s0 = eighth(len(lens), H, dv, dk)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return dict(q=q, k=k, v=v, g=np.log(alpha), beta=beta, cu_seqlens=cu, initial_state=s0), alpha


def main():
    c, alpha = case()
    out, fin = oracle.run(**c)
    doc = {
        "what": "tiny packed KDA case, token recurrence in fp64 (oracle output)",
        "inputs": {"q": c["q"].tolist(), "k": c["k"].tolist(), "v": c["v"].tolist(),
                   "alpha": alpha.tolist(), "beta": c["beta"].tolist(),
                   "cu_seqlens": c["cu_seqlens"].tolist(), "initial_state": c["initial_state"].tolist()},
        "out": out.tolist(),
        "final_state": fin.tolist(),
    }
    with open(os.path.join(HERE, "tiny_rational.json"), "w") as fh:
        json.dump(doc, fh, indent=1)


if __name__ == "__main__":
    main()
