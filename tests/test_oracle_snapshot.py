"""Regression check of the fp64 oracle against its stored snapshot
(tests/golden/oracle_snapshot_small.json, written by
tests/golden/make_oracle_snapshot.py from the oracle alone). This is not a pin:
it makes any change to the oracle's arithmetic visible. A change that is meant
must come with the passage or reading that justifies it, and with a rewritten
snapshot."""
import json
import os

import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_its_snapshot():
    with open(os.path.join(HERE, "golden", "oracle_snapshot_small.json")) as f:
        doc = json.load(f)
    x = {n: (np.asarray(a, dtype=np.float64).reshape(doc["shapes"][n]) if n != "scale" else a)
         for n, a in doc["inputs"].items()}
    r = oracle.run(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], x["do"], x["dht"], None,
                   chunk=8)
    for key, ref in doc["outputs"].items():
        ref = np.asarray(ref, dtype=np.float64)
        err = np.abs(np.asarray(r[key]) - ref).max() / max(np.abs(ref).max(), 1e-300)
        assert err < 1e-13, (key, err)
