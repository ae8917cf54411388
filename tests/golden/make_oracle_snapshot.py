"""Writes tests/golden/oracle_snapshot_small.json: a small case's inputs and the
fp64 oracle's outputs and gradients, as a regression snapshot of the oracle.

It calls only ``oracle/`` (inputs come from numpy's seeded generator). The
snapshot is not a pin: it records what the oracle computes today, so that any
later change to the oracle's arithmetic shows up in
tests/test_oracle_snapshot.py and has to be justified.

    python tests/golden/make_oracle_snapshot.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402

OUT = os.path.join(HERE, "oracle_snapshot_small.json")


def make_inputs():
    rng = np.random.default_rng(20260601)
    B, T, H, HV, K, V = 1, 21, 1, 2, 4, 3
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, HV, V))
    g = -np.log1p(np.exp(-rng.normal(3.0, 1.0, (B, T, HV, K))))  # logsigmoid
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, HV))))
    h0 = 0.1 * rng.standard_normal((1, HV, K, V))
    do = rng.standard_normal((B, T, HV, V))
    dht = rng.standard_normal((1, HV, K, V))
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, do=do, dht=dht, scale=K ** -0.5)


def run(x):
    return oracle.run(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], x["do"], x["dht"], None,
                      chunk=8)


def main():
    x = make_inputs()
    r = run(x)
    keys = ["o", "ht", "dq", "dk", "dv", "dg", "dbeta", "dh0"]
    doc = {
        "what": "regression snapshot of the fp64 oracle (not a pin); written by make_oracle_snapshot.py",
        "inputs": {n: (np.asarray(a).tolist() if n != "scale" else a) for n, a in x.items()},
        "shapes": {n: list(np.asarray(a).shape) for n, a in x.items() if n != "scale"},
        "outputs": {n: np.asarray(r[n]).tolist() for n in keys},
    }
    with open(OUT, "w") as f:
        json.dump(doc, f, indent=None, separators=(",", ":"))
        f.write("\n")


if __name__ == "__main__":
    main()
