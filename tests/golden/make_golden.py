"""Writes the stored fixtures under tests/golden/.

Calls only the seeded input generator and the CPU oracle (never the CUDA
path):
  * input_checksums.json — SHA-256 of the generated q, k, v bytes of the small
    workloads, so a change of the generator is caught;
  * oracle_tiny.json — the oracle's output on a tiny seeded fp32 case,
    a regression record of the oracle itself (the pins in
    test_oracle_pins.py, not this file, tie the oracle to the mathematics).

Run:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from exact_tiled_attention_04_gb300 import inputs as I  # noqa: E402


def checksums():
    out = {}
    for name in ("single_head_n512", "tail_n1000"):
        q, k, v = I.make(I.WORKLOADS[name])
        out[name] = {t: hashlib.sha256(x.tobytes()).hexdigest() for t, x in zip("qkv", (q, k, v))}
    return out


def tiny():
    w = I.custom(1, 2, 5, 4, "f32", seed=7)
    q, k, v = I.make(w)
    o, lse = oracle.attention_f64(q, k, v, float(w.scale), threads=1)
    return {"workload": [w.B, w.H, w.N, w.d, w.dtype, w.seed],
            "scale": float(w.scale),
            "o": [float(x) for x in o.reshape(-1)],
            "lse": [float(x) for x in lse.reshape(-1)]}


if __name__ == "__main__":
    with open(os.path.join(HERE, "input_checksums.json"), "w") as f:
        json.dump(checksums(), f, indent=1, sort_keys=True)
    with open(os.path.join(HERE, "oracle_tiny.json"), "w") as f:
        json.dump(tiny(), f, indent=1)
    print("wrote fixtures")
