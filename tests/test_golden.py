"""The oracle still reproduces its frozen tiny case (tests/golden/oracle_tiny.json)."""
import json
import os

import numpy as np

import oracle

from .golden import make_golden


def test_oracle_matches_frozen_tiny_case():
    with open(os.path.join(os.path.dirname(__file__), "golden", "oracle_tiny.json")) as f:
        doc = json.load(f)
    out = oracle.forward(**make_golden.case())
    for k, v in doc["outputs"].items():
        np.testing.assert_allclose(out[k], np.array(v), rtol=1e-13, atol=1e-15, err_msg=k)
