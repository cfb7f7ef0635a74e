"""Writes tests/golden/tiny_decode_fp32.json from the oracle alone.

The pages print no worked example for the KDA step, so the stored values are
the oracle's own output on the tiny fp32 workload (1 sequence, 2 heads,
d_k = d_v = 16, 8 decode steps from a zero state and a zero conv tail).  They
guard the oracle against unintended change; the GPU tests compare against the
oracle directly.  Run from the repository root:  python tests/golden/make_golden.py
"""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from hybrid_linear_attention_03_gb300 import inputs as I  # noqa: E402  (seeded inputs only)
from oracle import kda_oracle as ko  # noqa: E402


def main():
    wl = I.TINY_DECODE
    w = {k: v.double().numpy() for k, v in wl.weights().items()}
    pool = ko.OraclePool(wl.H, wl.dk, wl.dv, wl.W, wl.eps_l2, wl.eps_rms)
    outs = []
    for step in range(wl.extra["steps"]):
        inp = {k: v.double().numpy() for k, v in wl.tokens(100 + step, 1).items()}
        outs.append(pool.run(0, inp, w)[0].tolist())
    S, tail = pool.get(0)
    doc = {
        "what": "oracle output, tiny fp32 decode workload (8 steps, H=2, d=16)",
        "workload": wl.name,
        "seed": wl.seed,
        "out": outs,
        "state": S.tolist(),
        "tail": tail.tolist(),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_decode_fp32.json")
    with open(path, "w") as f:
        json.dump(doc, f)
    print("wrote", path)


if __name__ == "__main__":
    main()
