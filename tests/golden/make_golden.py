"""Writes tests/golden/recipe1_oracle.json from the CPU oracle alone.

Inputs come from `synth_inputs` (recipe 1: logistic, X 4096x64, b=16, s=4,
eta=0.1, 20 outer iterations, seed 0); every stored value is computed by `oracle`.
It serves as a regression fixture: a later change to the oracle's arithmetic
shows up as a mismatch here.  Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth_inputs as si  # noqa: E402


def main():
    p = si.make_problem(1)
    r = p.recipe
    w_nz = si.random_weights(r.n, seed=5)
    out = {"recipe": r.name, "seed": 0}
    for tag, w0 in (("from_zero", np.zeros(r.n, np.float32)), ("from_random", w_nz)):
        parts = oracle.outer_step(p.X, p.y, w0, r.b, r.s, r.eta, r.loss, 0, 0,
                                  mode="emulate", return_parts=True)
        out[tag] = {
            "idx": [int(v) for v in parts["idx"]],
            "r": [float(v) for v in parts["r"]],
            "alpha": [float(v) for v in parts["alpha"]],
            "w": [float(v) for v in parts["w"]],
        }
    w_ca, _ = oracle.train(p.X, p.y, r.b, r.s, r.eta, r.loss, 0, r.iters, mode="emulate")
    w_sgd = oracle.plain_sgd(p.X, p.y, r.b, r.iters * r.s, r.eta, r.loss, 0, mode="fp64")
    out["final_loss_emulate"] = oracle.full_loss(p.X, p.y, w_ca, r.loss)
    out["final_loss_fp64_sgd"] = oracle.full_loss(p.X, p.y, w_sgd, r.loss)
    with open(os.path.join(HERE, "recipe1_oracle.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
