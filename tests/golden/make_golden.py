"""Writes tests/golden/oracle_tiny_varlen.txt: the fp64 oracle's backward on
one tiny seeded case, as a regression fixture of the oracle itself.

The case: three packed sequences of 9, 0 and 12 tokens (an empty one in the
middle), H = 2 heads, K = 3, V = 2 (K != V), a nonzero h0 and dh_T and a gate
bias; inputs from the shared seeded recipe (linear_attention_backward_gb300.
workloads, seed 7) and the bias from torch.Generator(11).  Only oracle/
computes the values.  Rerun this script only for a deliberate change to the
oracle's arithmetic, and name the passage that justifies it.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from linear_attention_backward_gb300 import workloads as wl  # noqa: E402

FIXTURE = os.path.join(HERE, "oracle_tiny_varlen.txt")
KEYS = ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias", "dh0")


def case():
    w = wl.custom("golden", H=2, K=3, V=2, dtype="fp32", with_h0=True, with_dhT=True,
                  varlen=(3, 0, 12))
    x = wl.make_inputs(w, seed=7, lengths=[9, 0, 12])
    x["dt_bias"] = torch.randn(2, 3, generator=torch.Generator().manual_seed(11)) * 0.5
    return x


def oracle_grads(x):
    f64 = lambda t: t.double().reshape(-1, *t.shape[2:]).numpy()
    return oracle.backward(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]), f64(x["beta"]),
                           x["A_log"].double().numpy(), x["h0"].double().numpy(), f64(x["dO"]),
                           x["dhT"].double().numpy(), cu_seqlens=wl.seq_bounds(x),
                           dt_bias=x["dt_bias"].double().numpy())


def read_fixture(path=FIXTURE):
    out, key, shape, vals = {}, None, None, []
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("tensor "):
            if key is not None:
                out[key] = np.array(vals, dtype=np.float64).reshape(shape)
            _, key, dims = line.split(" ", 2)
            shape = tuple(int(d) for d in dims.split("x"))
            vals = []
        else:
            vals.append(float.fromhex(line))
    if key is not None:
        out[key] = np.array(vals, dtype=np.float64).reshape(shape)
    return out


def main():
    oracle.build()
    g = oracle_grads(case())
    with open(FIXTURE, "w") as f:
        f.write("# fp64 oracle backward on the tiny varlen case of tests/golden/make_golden.py\n")
        f.write("# (lengths 9, 0, 12; H=2 K=3 V=2; h0, dh_T, gate bias; seed 7, bias seed 11).\n")
        f.write("# Values are exact fp64 in C99 hex notation, row-major, one per line.\n")
        for k in KEYS:
            a = np.asarray(g[k], dtype=np.float64)
            f.write(f"tensor {k} {'x'.join(str(d) for d in a.shape)}\n")
            for v in a.ravel():
                f.write(float(v).hex() + "\n")
    print("wrote", FIXTURE)


if __name__ == "__main__":
    main()
