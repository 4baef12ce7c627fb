"""Writes tests/golden/oracle_small.json: the oracle's values on a small seeded case.

The stored values come from oracle/ alone (never from the GPU path); the inputs
come from the seeded generator.  The pages print no worked example, so this
fixture is a regression lock on the oracle across machines and edits: a change
to it must be justified by a reading of the method, and the fixture rewritten
with this script.

Run:  python tests/golden/make_fixtures.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from speculative_decoding_mla_gb300 import synth  # noqa: E402

CASES = {
    "causal_b2": dict(prefixes=[37, 100], drafts=[3, 5], heads=4, tree=None, seed=101),
    "tree_b2": dict(prefixes=[64, 9], drafts=[12, 7], heads=2, tree=3, seed=102),
}
DIMS = [0, 1, 255, 511]


def make(spec):
    pool = sum(spec["prefixes"]) + sum(spec["drafts"]) + 11
    return synth.make_case("golden", spec["prefixes"], spec["drafts"], num_heads=spec["heads"], pool_slots=pool,
                           tree_depth=spec["tree"], seed=spec["seed"])


def main():
    out = {"generator": "speculative_decoding_mla_gb300.synth.make_case", "dims": DIMS, "cases": {}}
    for name, spec in CASES.items():
        case = make(spec)
        o, l = oracle.verify(case)
        T, H = l.shape
        out["cases"][name] = {
            "spec": spec,
            "lse": [[float(x) for x in row] for row in l],
            "out_dims": [[[float(o[t, h, d]) for d in DIMS] for h in range(H)] for t in range(T)],
        }
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
