"""Writes tests/golden/oracle_small_case.json: a small fixed case and the
oracle's FP64 result on it.  Calls only the oracle (no CUDA code).  The case
is a regression fixture for the oracle itself: the independent checks of its
arithmetic are the pins in tests/test_oracle_pins.py.

Inputs are short decimal values (exactly what the JSON holds) in the layout of
the FlashInfer docs' chunk_gated_delta_rule2 parameters: two packed sequences
(lengths 3 and 2), H = 1 key head, HV = 2 value heads, K = 3, V = 2.
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def case():
    rng = np.random.default_rng(2024)
    T, H, HV, K, V, N = 5, 1, 2, 3, 2, 2
    r = lambda *s: np.round(rng.uniform(-1, 1, s), 2)
    return dict(
        q=r(T, H, K), k=r(T, H, K), v=r(T, HV, V),
        g=-np.round(rng.uniform(0, 0.5, (T, HV, K)), 2),
        beta=np.round(rng.uniform(0, 2, (T, HV, K)), 2),
        w=np.round(rng.uniform(0, 1, (T, HV, V)), 2),
        initial_state=r(N, HV, K, V), cu_seqlens=[0, 3, 5], scale=0.5)


def main():
    c = case()
    o, hT = oracle.gdn2_forward(**c)
    out = {"source": "FlashInfer docs, chunk_gated_delta_rule2 recurrence; oracle FP64",
           "inputs": {k: (np.asarray(v).tolist() if not isinstance(v, float) else v) for k, v in c.items()},
           "o": o.tolist(), "final_state": hT.tolist()}
    with open(os.path.join(HERE, "oracle_small_case.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
