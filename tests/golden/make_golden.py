"""Writes tests/golden/oracle_samples.json: sampled outputs of the fp64 oracle on small seeded
cases, so that any later change to the oracle's arithmetic shows up as a failing pin.

Calls only the oracle and the seeded input generator. Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from gqa_attention_long_gb300.inputs import layer_inputs  # noqa: E402

CASES = [dict(seed=0, S=256, Smax=512, rope_delta=0),
         dict(seed=5, S=3, Smax=128, rope_delta=-2),
         dict(seed=9, S=130, Smax=256, rope_delta=40)]


def main():
    rng = np.random.default_rng(2024)
    out_cases = []
    for c in CASES:
        x = layer_inputs(c["seed"], c["S"], c["Smax"])
        f = lambda t: t.double().numpy()  # noqa: E731
        r = oracle.expert_attention_layer(f(x.q_raw), f(x.k_raw), f(x.v_raw), f(x.q_gamma),
                                          f(x.k_gamma), f(x.k_cache), f(x.v_cache),
                                          c["S"], c["Smax"], c["rope_delta"])
        idx = np.stack([rng.integers(0, 16, 48), rng.integers(0, 64, 48), rng.integers(0, 128, 48)], 1)
        val = r["out"][idx[:, 0], idx[:, 1], idx[:, 2]]
        out_cases.append(dict(c, idx=idx.tolist(), val=[float(v) for v in val]))
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_samples.json")
    with open(path, "w") as fh:
        json.dump({"_about": "fp64 oracle outputs at sampled (head, token, channel) indices; "
                             "written by tests/golden/make_golden.py from the oracle only",
                   "cases": out_cases}, fh, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
