"""Top-k router on the GPU: ids bit-exact (same FP32 comparisons as the
oracle), softmax weights within a few FP32 ulps."""
import json
import os

import numpy as np
import pytest

import synth
from helpers import ROOT, ensure_lib, to_np
from oracle import moe as om

pytestmark = pytest.mark.gpu


def _route(logits, k):
    import torch
    import moe_expert_gb300 as mx
    ensure_lib()
    ids, w = mx.route_topk(torch.from_numpy(np.ascontiguousarray(logits)).cuda(), k)
    torch.cuda.synchronize()
    return to_np(ids), to_np(w)


@pytest.mark.parametrize("T,E,k", [(1, 8, 1), (37, 128, 8), (8192, 128, 8), (5, 1000, 16), (3, 33, 4)])
def test_route_matches_oracle(T, E, k):
    logits = synth.router_logits(synth.rng(T + E), T, E)
    ids, w = _route(logits, k)
    rid, rw = om.route_topk(logits, k)
    assert np.array_equal(ids.astype(np.int64), rid)
    assert np.all(np.abs(w - rw) <= 4e-6 * rw + 1e-9)


def test_route_ties_go_to_lower_id():
    logits = np.zeros((2, 64), np.float32)
    logits[0, [5, 9, 40]] = 1.0
    logits[1, :] = 0.5
    ids, w = _route(logits, 4)
    assert ids[0].tolist() == [5, 9, 40, 0]
    assert ids[1].tolist() == [0, 1, 2, 3]
    assert np.allclose(w[1], 0.25, rtol=0, atol=1e-7)


def test_decode_workload_routing_covers_20_experts():
    ref = json.load(open(os.path.join(ROOT, "tests", "golden", "decode_routing.json")))
    logits = synth.decode_logits(ref["tokens"], ref["experts"], ref["sub_seed"])
    ids, _ = _route(logits, ref["top_k"])
    assert ids.tolist() == ref["ids"]
    assert len(set(ids.reshape(-1).tolist())) == ref["distinct"] == 20
