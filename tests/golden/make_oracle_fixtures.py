"""Write oracle_small.json: the float64 oracle's outputs on three small seeded cases.

These are regression fixtures for the oracle itself: any later change to its arithmetic
shows up as a failing comparison, and has to be justified by the passage of the pages it
follows.  The values come from `oracle` alone; the inputs come from the seeded generators in
`contrastive_embedding_loss_gb300.synth`.  No library output is involved.

Run: python tests/golden/make_oracle_fixtures.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from contrastive_embedding_loss_gb300 import synth  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.json")

CASES = [
    # name, kind, generator, generator args, prefixes, scale, bias
    ("clip_n12_d192", "clip", "paired", (12, 192, 1.0, 11), (64, 128, 192), 1 / 0.07, 0.0),
    ("siglip_n10_d128", "siglip", "paired", (10, 128, 1.0, 12), (64, 128), 10.0, -10.0),
    ("rows_q6_k15_d128", "rows", "queries_keys", (6, 15, 128, 1.0, 13), (64, 128), 20.0, 0.0),
]


def inputs(gen, args):
    return getattr(synth, gen)(*args)


def summary(x):
    """Sum, sum of squares and four fixed entries of a gradient matrix."""
    n, d = x.shape
    picks = [(0, 0), (0, d - 1), (n - 1, 0), (n - 1, d - 1)]
    return {"sum": float(x.sum()), "sumsq": float((x * x).sum()), "entries": [[i, j, float(x[i, j])] for i, j in picks]}


def main():
    out = {
        "source": "float64 oracle (oracle/), inputs from contrastive_embedding_loss_gb300.synth; written by "
                  "tests/golden/make_oracle_fixtures.py",
        "cases": [],
    }
    for name, kind, gen, args, pre, sc, bias in CASES:
        A, B = inputs(gen, args)
        r = oracle.fwd_bwd(kind, A, B, pre, sc, bias)
        out["cases"].append({
            "name": name, "kind": kind, "generator": gen, "args": list(args), "prefixes": list(pre), "scale": sc,
            "bias": bias, "loss": [float(v) for v in r["loss"]], "dA": summary(r["dA"]), "dB": summary(r["dB"]),
        })
    with open(OUT, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
