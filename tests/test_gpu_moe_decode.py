"""Grouped MoE decode layer on the GPU, checked stage by stage.

(i)   Hq is bit-exact to the oracle's q8_1 of the GPU's own FP32 H.
(ii)  H is the SwiGLU of the GPU's own g, u within a few FP32 ulps.
(iii) g, u (gate/up GEMV) within 1e-5 * sum|w*x| + 1e-6 of the oracle.
(iv)  out (down GEMV + combine on the GPU's Hq) within 1e-5 * sum|w*x| + 1e-6
      of the oracle run on that Hq.
(v)   end to end against the oracle's own chain: Hq agrees except where the
      FP32 rounding of g, u moves a value across a q8_1 rounding boundary;
      out agrees to a relative 1e-3 of its scale.
"""
import json
import os

import numpy as np
import pytest

import synth
from helpers import ROOT, assert_within, ensure_lib, to_np
from oracle import moe as om
from oracle import q8_1 as oq

pytestmark = pytest.mark.gpu


def build_layer(E, hidden, inter, experts, seed=0, dn_fmt="iq4_nl"):
    import moe_expert_gb300 as mx
    ensure_lib()
    gu = mx.PackedWeight("q8_0", E, 2 * inter, hidden).zero_()
    dn = mx.PackedWeight(dn_fmt, E, hidden, inter).zero_()
    gub, dnb = {}, {}
    for e in sorted(set(int(v) for v in experts)):
        gub[e] = synth.expert_blocks("gate_up", e, hidden, inter, "q8_0", seed=seed)
        dnb[e] = synth.expert_blocks("down", e, hidden, inter, dn_fmt, seed=seed)
        gu.pack_matrix(e, gub[e])
        dn.pack_matrix(e, dnb[e])
    return gu, dn, gub, dnb


def run_checks(E, hidden, inter, x, ids, w, dn_fmt="iq4_nl", seed=0):
    import torch
    import moe_expert_gb300 as mx
    T, k = ids.shape
    gu, dn, gub, dnb = build_layer(E, hidden, inter, ids.reshape(-1), seed=seed, dn_fmt=dn_fmt)
    xt = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    it = torch.from_numpy(np.ascontiguousarray(ids.astype(np.int32))).cuda()
    wt = torch.from_numpy(np.ascontiguousarray(w.astype(np.float32))).cuda()
    out, dbg = mx.moe_decode(gu, dn, xt, it, wt, debug=True)
    out_plain = mx.moe_decode(gu, dn, xt, it, wt)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    out, out_plain = to_np(out), to_np(out_plain)
    g = {k_: to_np(v) for k_, v in dbg.items()}
    # the debug call and the plain call compute the same bits
    assert np.array_equal(out.view(np.uint32), out_plain.view(np.uint32))

    w32 = w.astype(np.float32)
    # (iii) gate/up against the oracle (identical q8_1 of x on both sides)
    ref = om.moe_decode(gub, dnb, x, ids, w32, down_fmt=dn_fmt, h_override=g["h"])
    assert_within(g["gu"], ref["gu"], ref["gu_A"], "gate/up")
    # (ii) SwiGLU of the GPU's own g, u
    gg, uu = g["gu"][:, :inter].astype(np.float64), g["gu"][:, inter:].astype(np.float64)
    h64 = gg / (1 + np.exp(-gg)) * uu
    ulp = np.spacing(np.abs(g["h"]).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(g["h"] - h64) <= 4 * ulp + 1e-30)
    # (i) Hq bit-exact to q8_1 of the GPU's H
    assert np.array_equal(g["hq"], ref["Hq"])
    assert np.array_equal(g["hds"][..., 0].view(np.uint32), ref["Hd"].view(np.uint32))
    assert np.array_equal(g["hds"][..., 1].view(np.uint32), ref["Hs"].view(np.uint32))
    # (iv) down + combine on the GPU's Hq
    assert_within(out, ref["out"], ref["out_A"], "down+combine")
    # (v) end to end against the oracle's own H
    own = om.moe_decode(gub, dnb, x, ids, w32, down_fmt=dn_fmt)
    flips = int((own["Hq"] != g["hq"]).sum())
    assert flips <= max(2, own["Hq"].size // 2000), flips
    scale = np.abs(own["out"]).max()
    assert np.abs(out - own["out"]).max() <= 1e-3 * scale
    return flips


@pytest.mark.parametrize("T,k,E,hidden,inter,dn_fmt", [
    (1, 1, 4, 64, 32, "iq4_nl"),
    (3, 4, 16, 512, 256, "iq4_nl"),
    (2, 8, 32, 2560, 96, "q8_0"),
    (8, 8, 64, 1024, 512, "iq4_nl"),
])
def test_decode_small(T, k, E, hidden, inter, dn_fmt):
    g = synth.rng(T * 100 + E)
    x = synth.activations(g, T, hidden)
    ids, w = om.route_topk(synth.router_logits(g, T, E), k)
    run_checks(E, hidden, inter, x, ids, w, dn_fmt=dn_fmt, seed=3)


def test_decode_wide_layer():
    """hidden 4096 and inter 2048: eight K slices in gate/up (one warp per
    slice) and four in down (two-team down kernel), the variants the
    2560 x 1536 workload does not reach."""
    T, k, E, hidden, inter = 2, 4, 8, 4096, 2048
    g = synth.rng(77)
    x = synth.activations(g, T, hidden)
    ids, w = om.route_topk(synth.router_logits(g, T, E), k)
    run_checks(E, hidden, inter, x, ids, w, seed=5)


def test_decode_repeated_expert_and_single_expert_chain():
    """All 8 slots on one expert (more entries than a group pass holds when
    T = 2) equals the single-expert chain."""
    T, k, E, hidden, inter = 2, 8, 4, 256, 64
    x = synth.activations(synth.rng(4), T, hidden)
    ids = np.full((T, k), 1)
    w = np.full((T, k), 1.0 / k)
    run_checks(E, hidden, inter, x, ids, w, seed=4)


def test_decode_workload_full_size():
    ref = json.load(open(os.path.join(ROOT, "tests", "golden", "decode_routing.json")))
    T, E, k = ref["tokens"], ref["experts"], ref["top_k"]
    hidden, inter = 2560, 1536
    ids, w = om.route_topk(synth.decode_logits(T, E, ref["sub_seed"]), k)
    assert len(set(ids.reshape(-1).tolist())) == 20
    x = synth.decode_tokens(T, hidden)
    flips = run_checks(E, hidden, inter, x, ids, w, seed=0)
    print("Hq flips vs the oracle's own chain:", flips)
