"""Write tests/golden/oracle_trajectories.json: short trajectories computed by the CPU
oracle alone (no other code), stored as exact bit patterns.

They freeze the oracle's arithmetic: any later change to it shows up as a diff here and
must be justified by the method's sources. Run: python tests/golden/write_golden.py
"""
import hashlib
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from oracle import HParams, Q8Opts  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_trajectories.json")
CASES = {
    "fp32_n2049_wd01": dict(mode="fp32", n=2049, steps=4, hp=HParams(weight_decay=0.01), q8=None),
    "bf16m_n777": dict(mode="bf16m", n=777, steps=4, hp=HParams(weight_decay=0.01), q8=None),
    "q8_rne_n4100": dict(mode="q8", n=4100, steps=4, hp=HParams(), q8=Q8Opts()),
    "q8_sr_p999_n4100": dict(mode="q8", n=4100, steps=4, hp=HParams(weight_decay=0.1),
                             q8=Q8Opts(stochastic_rounding=True, seed=42, percentile=99.9)),
    "q8v_sr_n3000": dict(mode="q8v", n=3000, steps=4, hp=HParams(weight_decay=0.01),
                         q8=Q8Opts(stochastic_rounding=True, seed=7, percentile=100.0)),
}


def inputs(n, steps, seed):
    """Small hand-rolled generator so the fixture does not depend on numpy's streams."""
    x = (np.arange(n * (steps + 1), dtype=np.float64) * 0.6180339887498949 + seed) % 1.0
    x = (x - 0.5) * 2.0
    p = (x[:n] * 0.03).astype(np.float32)
    grads = [(x[n * (t + 1):n * (t + 2)] * 1e-2).astype(np.float32) for t in range(steps)]
    return p, grads


def run(case):
    n, steps, mode = case["n"], case["steps"], case["mode"]
    p, grads = inputs(n, steps, seed=0.25)
    nb = oracle.n_blocks(n)
    if mode == "fp32":
        st = [np.zeros(n, np.float32), np.zeros(n, np.float32)]
    elif mode == "bf16m":
        st = [np.zeros(n, np.uint16), np.zeros(n, np.uint16)]
    elif mode == "q8v":
        st = [np.zeros(n, np.float32), np.zeros(n, np.uint8), np.zeros(nb, np.float32)]
    else:
        st = [np.zeros(n, np.int8), np.zeros(n, np.uint8), np.zeros(nb, np.float32), np.zeros(nb, np.float32)]
    for t in range(1, steps + 1):
        oracle.step_list(mode, [p], [grads[t - 1]], [st], t, case["hp"], case["q8"] or Q8Opts())
    return {"param": p, **{f"state{i}": a for i, a in enumerate(st)}}


def digest(arrays):
    out = {}
    for k, a in arrays.items():
        out[k] = {"dtype": str(a.dtype), "n": int(a.size), "sha256": hashlib.sha256(a.tobytes()).hexdigest(),
                  "head": a[:4].view(np.uint8).tobytes().hex()}
    return out


def main():
    data = {name: digest(run(case)) for name, case in CASES.items()}
    with open(OUT, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
    print("wrote", OUT)


if __name__ == "__main__":
    main()
