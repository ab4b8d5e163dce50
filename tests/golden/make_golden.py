"""Writes the oracle fixtures of this directory. Calls only the oracle and the seeded input
generator; nothing here comes from the CUDA path. The pages print no worked-example values
(their numbers are parity summaries such as cosine similarities), so the stored values are
the oracle's own, kept to catch any later drift of the oracle (an edit, a compiler, a
platform): for each output of a small workload, its sum, its sum of squares and eight
elements at fixed flat indices, with 17 significant digits.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from kimi_delta_attention_15_gb300 import inputs as I  # noqa: E402

WORKLOADS = ("fixed_T17_H1", "varlen_17_33_65_H4")
KEYS = ("o", "hT", "dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "dA_log", "ddt_bias")


def digest(x):
    x = np.asarray(x, dtype=np.float64).ravel()
    idx = [int(i) for i in np.linspace(0, x.size - 1, 8).round()] if x.size else []
    return {"size": int(x.size), "sum": float(x.sum()), "sumsq": float((x * x).sum()),
            "at": {str(i): float(x[i]) for i in idx}}


def golden(name):
    w = next(x for x in I.WORKLOADS if x.name == name)
    inp = I.make_inputs(w)
    out = dict(oracle.forward(inp))
    out.update(oracle.backward(inp))
    return {k: digest(out[k]) for k in KEYS if out.get(k) is not None}


def main():
    for name in WORKLOADS:
        path = os.path.join(HERE, f"oracle_{name}.json")
        with open(path, "w") as f:
            json.dump({"workload": name, "writer": "tests/golden/make_golden.py", "outputs": golden(name)}, f,
                      indent=1, sort_keys=True, default=repr)
            f.write("\n")
        print("wrote", path)


if __name__ == "__main__":
    main()
