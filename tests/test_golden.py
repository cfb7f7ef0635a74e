"""The oracle still reproduces its stored tiny-workload output (regression
guard; the stored file is written by tests/golden/make_golden.py from the
oracle alone)."""

import json
import os

import numpy as np

from hybrid_linear_attention_03_gb300 import inputs as I
from oracle import kda_oracle as ko

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "tiny_decode_fp32.json")


def test_tiny_decode_matches_golden():
    with open(GOLDEN) as f:
        doc = json.load(f)
    wl = I.TINY_DECODE
    w = {k: v.double().numpy() for k, v in wl.weights().items()}
    pool = ko.OraclePool(wl.H, wl.dk, wl.dv, wl.W, wl.eps_l2, wl.eps_rms)
    for step in range(wl.extra["steps"]):
        inp = {k: v.double().numpy() for k, v in wl.tokens(100 + step, 1).items()}
        out = pool.run(0, inp, w)
        np.testing.assert_allclose(out[0], np.array(doc["out"][step]), rtol=0, atol=1e-12)
    S, tail = pool.get(0)
    np.testing.assert_allclose(S, np.array(doc["state"]), rtol=0, atol=1e-12)
    np.testing.assert_array_equal(tail, np.array(doc["tail"]))
