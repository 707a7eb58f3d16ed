"""The residual add fused into the MoE combine (moex_moe_decode_residual,
moex_moe_prefill_residual), on the GPU through the C ABI.

Decode adds the residual after the slot-order combine with one FP32
addition, so its output is checked bitwise against fp32(residual + the
plain layer's output).  Prefill starts the output at the residual and adds
the weighted expert outputs in any order, so it is checked against the
plain layer plus the residual within 1e-5 * (sum|w*x| + |residual|) + 1e-6,
with the error scale from the oracle.  Both are run with a separate residual
and in place (residual == out).
"""
import numpy as np
import pytest

import synth
from helpers import ensure_lib, to_np
from oracle import moe as om
from oracle import prefill as op

pytestmark = pytest.mark.gpu


def _stack(mx, kind, fmt, E, hidden, inter, seed):
    rows, K = (2 * inter, hidden) if kind == "gate_up" else (hidden, inter)
    W = mx.PackedWeight(fmt, E, rows, K)
    blocks = {}
    for e in range(E):
        blocks[e] = synth.expert_blocks(kind, e, hidden, inter, fmt, seed=seed)
        W.pack_matrix(e, blocks[e])
    return W, blocks


def test_decode_residual_bitwise():
    import torch
    import moe_expert_gb300 as mx
    ensure_lib()
    T, k, E, hidden, inter = 3, 4, 16, 512, 256
    g = synth.rng(61)
    x = synth.activations(g, T, hidden)
    ids, w = om.route_topk(synth.router_logits(g, T, E), k)
    res = synth.activations(g, T, hidden)
    gu, _ = _stack(mx, "gate_up", "q8_0", E, hidden, inter, 61)
    dn, _ = _stack(mx, "down", "iq4_nl", E, hidden, inter, 61)
    xt = torch.from_numpy(x).cuda()
    it = torch.from_numpy(ids.astype(np.int32)).cuda()
    wt = torch.from_numpy(w.astype(np.float32)).cuda()
    plain = to_np(mx.moe_decode(gu, dn, xt, it, wt))
    want = (res + plain).astype(np.float32)
    rt = torch.from_numpy(res).cuda()
    got = to_np(mx.moe_decode(gu, dn, xt, it, wt, residual=rt))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    inplace = rt.clone()
    mx.moe_decode(gu, dn, xt, it, wt, out=inplace, residual=inplace)
    assert np.array_equal(to_np(inplace).view(np.uint32), want.view(np.uint32))
    assert mx.device_status() == 0


def test_prefill_residual_within_tolerance():
    import torch
    import moe_expert_gb300 as mx
    ensure_lib()
    T, k, E, hidden, inter = 80, 2, 4, 256, 128
    g = synth.rng(67)
    xb = synth.bf16_activations(g, T, hidden)
    ids, w = om.route_topk(synth.router_logits(g, T, E), k)
    res = synth.activations(g, T, hidden)
    gu, gub = _stack(mx, "gate_up", "iq4_nl", E, hidden, inter, 67)
    dn, dnb = _stack(mx, "down", "iq4_nl", E, hidden, inter, 67)
    xt = torch.from_numpy(xb.view(np.int16)).cuda()
    it = torch.from_numpy(ids.astype(np.int32)).cuda()
    wt = torch.from_numpy(w.astype(np.float32)).cuda()
    plain = to_np(mx.moe_prefill(gu, dn, xt, it, wt)).astype(np.float64)
    scale = op.moe_prefill(gub, dnb, xb, ids, w.astype(np.float32).astype(np.float64))["out_A"]
    bound = 1e-5 * (scale + np.abs(res)) + 1e-6
    rt = torch.from_numpy(res).cuda()
    got = to_np(mx.moe_prefill(gu, dn, xt, it, wt, residual=rt)).astype(np.float64)
    assert np.all(np.abs(got - (plain + res)) <= bound)
    inplace = rt.clone()
    mx.moe_prefill(gu, dn, xt, it, wt, out=inplace, residual=inplace)
    assert np.all(np.abs(to_np(inplace).astype(np.float64) - (plain + res)) <= bound)
    assert mx.device_status() == 0
