"""Writes the golden fixtures of this directory from the float64 oracle.

The pages print no worked numerical example of LLA or Parallax, so every stored value here is
written by this script, which calls only ``oracle/`` (and the seeded input generators of
``local_linear_attention_gb300.workloads``, which hold none of the method's arithmetic). The
fixtures pin the oracle against accidental change (``tests/test_golden.py`` recomputes them) and
give the GPU path fixed expected values.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import torch  # noqa: E402

from local_linear_attention_gb300 import workloads as W  # noqa: E402
from oracle import (lla_forward_oracle, parallax_backward_oracle,  # noqa: E402
                    parallax_forward_oracle)

ROWS = [0, 1, 2, 3, 16, 17, 64, 127]  # first token, tiny prefixes, T = d + 1, the last row


def tiny_inputs():
    w = W.WORKLOADS[1]
    q, k, v = W.make_inputs(w)
    r = W.make_probe(w.B, w.H, w.T, w.d, w.dtype, seed=w.seed + 100)
    return w, q, k, v, r


def backward_inputs():
    q, k, v = W.make_iid(1, 1, 8, 16, 16, "f32", seed=77)
    r = W.make_probe(1, 1, 8, 16, "f32", seed=78)
    g = torch.Generator().manual_seed(79)
    do = torch.randn(1, 1, 8, 16, generator=g)
    return q, k, v, r, do


def fixtures():
    w, q, k, v, r = tiny_inputs()
    lam, h = w.points[0]
    out = {}
    out["lla_forward_tiny.json"] = {
        "what": ("causal LLA forward (intercept of the weighted ridge regression), workload 1 "
                 "(tiny: B1 H1 T128 d=dv=16 fp32, i.i.d. N(0,1), seed 0, h=4, lambda=1e-2)"),
        "definition": "'Parallax' blog, s.2 Canonical Formulation",
        "generator": "oracle.lla_forward_oracle via tests/golden/make_golden.py",
        "h": h, "lambda": lam, "rows": ROWS,
        "values": lla_forward_oracle(q, k, v, h, lam, rows=ROWS).tolist(),
    }
    out["parallax_forward_tiny.json"] = {
        "what": "causal Parallax forward with probe N(0,1/d) (seed 100) on workload 1",
        "definition": "'Parallax' blog, s.2 Parallax and Appendix B with eta = 0",
        "generator": "oracle.parallax_forward_oracle via tests/golden/make_golden.py",
        "h": h, "rows": ROWS,
        "values": parallax_forward_oracle(q, k, v, r, h, rows=ROWS).tolist(),
    }
    bq, bk, bv, br, bdo = backward_inputs()
    dq, dk, dv, dr = parallax_backward_oracle(bq, bk, bv, br, bdo, 1.5)
    out["parallax_backward_tiny.json"] = {
        "what": ("gradients of the causal Parallax forward, B1 H1 T8 d=dv=16 fp32: q, k, v from "
                 "make_iid seed 77, probe from make_probe seed 78, dO ~ N(0,1) seed 79, h = 1.5"),
        "definition": ("the gradient of the 'Parallax' blog's forward (s.2, Appendix B with "
                       "eta = 0), split as its Appendix F describes"),
        "generator": "oracle.parallax_backward_oracle via tests/golden/make_golden.py",
        "h": 1.5,
        "values": {"dq": dq.tolist(), "dk": dk.tolist(), "dv": dv.tolist(), "dr": dr.tolist()},
    }
    return out


def main():
    for name, fx in fixtures().items():
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(fx, f, indent=1)
            f.write("\n")


if __name__ == "__main__":
    main()
