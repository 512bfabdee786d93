"""The oracle reproduces its stored recipe-1 fixture (tests/golden/make_golden.py).

Indices must match exactly; floating-point values to 1e-6 relative (BLAS summation
order may differ between machines); the paper's own criterion -- CA-SGD loss within
0.5% of FP32/FP64 SGD -- is checked on the stored final losses as well.
"""
import json
import os

import numpy as np

import oracle
import synth_inputs as si

FIX = os.path.join(os.path.dirname(__file__), "golden", "recipe1_oracle.json")


def test_recipe1_fixture_matches():
    d = json.load(open(FIX))
    p = si.make_problem(1)
    r = p.recipe
    for tag, w0 in (("from_zero", np.zeros(r.n, np.float32)),
                    ("from_random", si.random_weights(r.n, seed=5))):
        parts = oracle.outer_step(p.X, p.y, w0, r.b, r.s, r.eta, r.loss, 0, 0,
                                  mode="emulate", return_parts=True)
        assert [int(v) for v in parts["idx"]] == d[tag]["idx"]
        for key in ("r", "alpha", "w"):
            want = np.array(d[tag][key])
            assert np.allclose(parts[key], want, rtol=1e-6, atol=1e-9), key


def test_recipe1_final_loss_gap_within_half_percent():
    d = json.load(open(FIX))
    gap = abs(d["final_loss_emulate"] - d["final_loss_fp64_sgd"]) / d["final_loss_fp64_sgd"]
    assert gap < 0.005
