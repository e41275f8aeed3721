"""Writes oracle_tiny.json: the fp64 oracle on a tiny seeded case.

The stored values come from the oracle alone (this script imports only the
oracle and the seeded input generator).  They freeze the oracle: a later
change to its arithmetic shows up as a mismatch in test_golden.py and has to
name the passage of the method that justifies it.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from hyper_connection_gated_gb300 import inputs  # noqa: E402

SHAPE = inputs.Shape(HC=2, HS=8, r=4)
M = 3


def case():
    w = {k: inputs.bf16_bits_to_f64(v) for k, v in inputs.weights(SHAPE, seed=11).items()}
    a = inputs.activations(M, SHAPE, seed=11)
    return dict(R=inputs.bf16_bits_to_f64(a["R"]), y=inputs.bf16_bits_to_f64(a["y"]),
                inj=a["inj"].astype(np.float64), Wnorm=w["Wnorm"], Wd=w["Wd"], Wi=w["Wi"],
                Wu=w["Wu"], eps=SHAPE.eps)


def main():
    out = oracle.forward(**case())
    doc = {"shape": {"HC": SHAPE.HC, "HS": SHAPE.HS, "r": SHAPE.r, "M": M, "seed": 11,
                     "eps": SHAPE.eps},
           "outputs": {k: np.asarray(out[k]).tolist()
                       for k in ("R2", "rrms", "lora", "inj_next", "x")}}
    with open(os.path.join(HERE, "oracle_tiny.json"), "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    main()
