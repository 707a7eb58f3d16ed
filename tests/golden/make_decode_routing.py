"""Writes decode_routing.json: the router-logit sub-seed of the MoE decode
workload (3 tokens, top-8 of 128 experts) whose routing covers exactly 20
distinct experts.  Calls only the oracle's routing and the seeded generators.

The workload asks for 24 token entries over 20 distinct experts; the pages do
not say how that count is reached, so sub-seeds 0, 1, 2, ... are drawn until
the oracle's top-8 routing gives exactly 20 distinct experts.

Run from the repository root:  python tests/golden/make_decode_routing.py
"""
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))

import numpy as np  # noqa: E402

import synth  # noqa: E402
from oracle import moe  # noqa: E402

T, E, K, DISTINCT = 3, 128, 8, 20


def main():
    for sub in range(100000):
        ids, w = moe.route_topk(synth.decode_logits(T, E, sub), K)
        if len(set(ids.reshape(-1).tolist())) == DISTINCT:
            out = dict(tokens=T, experts=E, top_k=K, distinct=DISTINCT, sub_seed=sub,
                       ids=ids.tolist())
            path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "decode_routing.json")
            with open(path, "w") as f:
                json.dump(out, f, indent=1)
                f.write("\n")
            print(path, sub)
            return
    raise SystemExit("no sub-seed found")


if __name__ == "__main__":
    main()
