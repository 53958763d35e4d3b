"""Write tiny_step.json: worked examples of whole training steps computed by
the fp64 oracle alone (no GPU code), frozen so that any later change to the
oracle's arithmetic shows up as a failing test and has to be justified.

The pages print no worked example of a training step, so these values are
the oracle's own; they guard it against accidental change, while the pins
of tests/test_oracle_pins.py tie it to facts outside it.

Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import mlp_oracle as om  # noqa: E402

CASES = [
    # name, loss, optimizer, clipping threshold
    ("ce_adamw", "ce", "adamw", 0.0),
    ("ce_adam_clip", "ce", "adam", 0.05),
    ("mse_sgd_clip", "mse", "sgd", 0.05),
    ("mse_adamw", "mse", "adamw", 0.0),
]
DIMS = [8, 6, 5, 4]
ACTS = (om.ACT_RELU, om.ACT_GELU_TANH)
B = 7
HYPER = (1e-2, 0.9, 0.999, 1e-8, 0.05)


def inputs():
    rng = np.random.default_rng(2024)
    params = []
    for l in range(len(DIMS) - 1):
        params.append(rng.standard_normal((DIMS[l + 1], DIMS[l])) * np.sqrt(2.0 / DIMS[l]))
        params.append(rng.standard_normal(DIMS[l + 1]) * 0.1)
    x = rng.standard_normal((B, DIMS[0]))
    labels = rng.integers(0, DIMS[-1], B)
    targets = rng.standard_normal((B, DIMS[-1]))
    return params, x, labels, targets


def compute():
    params, x, labels, targets = inputs()
    out = {"dims": DIMS, "acts": list(ACTS), "batch": B, "hyper": list(HYPER), "cases": {}}
    for name, loss, optim, max_norm in CASES:
        y = targets if loss == "mse" else labels
        zero = [np.zeros_like(p) for p in params]
        L, newp, newm, newv, grads, ex = om.train_step(params, zero, zero, 1, x, y, ACTS, *HYPER, optim=optim,
                                                       max_norm=max_norm, loss=loss)
        out["cases"][name] = {
            "loss": L, "clip": ex["clip"],
            "grads": [g.ravel().tolist() for g in grads],
            "params": [p.ravel().tolist() for p in newp],
        }
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_step.json"), "w") as f:
        json.dump(compute(), f, indent=None, separators=(",", ":"))
        f.write("\n")
