"""Regression check of the oracle against its stored small case (written by
tests/golden/make_golden.py, which calls only the oracle)."""
import json
import os

import numpy as np

import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_small_case():
    d = json.load(open(os.path.join(HERE, "oracle_small_case.json")))
    c = {k: (np.array(v) if isinstance(v, list) else v) for k, v in d["inputs"].items()}
    o, hT = oracle.gdn2_forward(**c)
    np.testing.assert_allclose(o, np.array(d["o"]), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(hT, np.array(d["final_state"]), rtol=1e-13, atol=1e-15)
