"""Writes tests/golden/oracle_samples.json and tests/golden/decode_samples.json: sampled outputs
of the fp64 oracle (the expert attention layer, and the text model's decode step) on small
seeded cases, so that any later change to the oracle's arithmetic shows up as a failing pin.

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
from gqa_attention_long_gb300.inputs import decode_inputs, layer_inputs  # noqa: E402

CASES = [dict(seed=0, S=256, Smax=512, rope_delta=0),
         dict(seed=5, S=3, Smax=128, rope_delta=-2),
         dict(seed=9, S=130, Smax=256, rope_delta=40)]
DECODE_CASES = [dict(seed=3, pos=0, Smax=128, rope_delta=0),
                dict(seed=4, pos=200, Smax=256, rope_delta=-17),
                dict(seed=6, pos=383, Smax=384, rope_delta=1000)]


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

    drng = np.random.default_rng(2025)
    dec_cases = []
    for c in DECODE_CASES:
        x = decode_inputs(c["seed"], c["pos"], c["Smax"])
        f = lambda t: t.double().numpy()  # noqa: E731
        r = oracle.text_decode_attention(f(x.q_raw), f(x.k_raw), f(x.v_raw), f(x.q_gamma),
                                         f(x.k_gamma), f(x.k_cache), f(x.v_cache), c["pos"],
                                         c["rope_delta"])
        idx = np.stack([drng.integers(0, 64, 48), drng.integers(0, 128, 48)], 1)
        val = r["out"][idx[:, 0], idx[:, 1]]
        dec_cases.append(dict(c, idx=idx.tolist(), val=[float(v) for v in val]))
    dpath = os.path.join(os.path.dirname(os.path.abspath(__file__)), "decode_samples.json")
    with open(dpath, "w") as fh:
        json.dump({"_about": "fp64 decode-step oracle outputs at sampled (query head, channel) "
                             "indices; written by tests/golden/make_golden.py from the oracle only",
                   "cases": dec_cases}, fh, indent=1)
    print("wrote", dpath)


if __name__ == "__main__":
    main()
