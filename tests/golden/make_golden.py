"""Writes tests/golden/worked_examples.json from the float64 oracle only.

The pages print no worked example for these operations, so the fixtures are
small hand-checkable cases taken through the oracle (run:
``python tests/golden/make_golden.py``).  ``tests/test_golden.py`` pins each
stored value independently with a 40-digit evaluation of the closed form, and
checks that the oracle still reproduces the file.

Definitions: "Engineering a CUDA Machine Learning Framework from Scratch",
sec. 3.1 (softmax by three passes), sec. 3.2 (LayerNorm moments), sec. 2.1 /
2.2 (fused loss gradient, analytic backward); "gpu-ml-learning" README,
Module 3 (cross-entropy).
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def main():
    x = np.array([[1.0, 2.0, 3.0]], np.float32)
    one = np.ones(3, np.float32)
    zero = np.zeros(3, np.float32)
    cases = {}
    cases["softmax_123"] = dict(
        cite="three-pass softmax, sec. 3.1 'Online FlashSoftmax'",
        x=x.tolist(), y=oracle.softmax(x).tolist())
    for lab in (0, 2):
        loss, dl, _ = oracle.xent(x, np.array([lab], np.int32))
        cases[f"xent_123_label{lab}"] = dict(
            cite="softmax cross-entropy, Module 3; fused gradient, sec. 2.1",
            x=x.tolist(), label=lab, loss=loss.tolist(), dlogits=dl.tolist())
    for eps in (0.0, 1e-5):
        y, mean, rstd = oracle.ln_fwd(x, one, zero, eps)
        cases[f"ln_fwd_123_eps{eps:g}"] = dict(
            cite="LayerNorm, sec. 3.2 'Welford Single-Pass Normalization'",
            x=x.tolist(), eps=eps, y=y.tolist(), mean=mean.tolist(), rstd=rstd.tolist())
    y, mean, rstd = oracle.ln_fwd(x, one, zero, 0.0)
    dy = np.array([[1.0, 0.0, 0.0]], np.float32)
    dx, dg, db, _, _ = oracle.ln_bwd(dy, x, mean, rstd, one)
    cases["ln_bwd_123_dy100"] = dict(
        cite="analytic LayerNorm backward, sec. 2.2",
        x=x.tolist(), dy=dy.tolist(), mean=mean.tolist(), rstd=rstd.tolist(),
        dx=dx.tolist(), dgamma=dg.tolist(), dbeta=db.tolist())
    with open(os.path.join(HERE, "worked_examples.json"), "w") as f:
        json.dump(cases, f, indent=1, sort_keys=True)
        f.write("\n")


if __name__ == "__main__":
    main()
