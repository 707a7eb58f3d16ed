"""Edge cases on the GPU, through the C ABI, against the oracle.

* GEMV with extreme FP16 weight scales (zero, negative zero, the smallest
  and largest subnormals, 65504) and activation columns that are all zero or
  carry +-3e4 outliers next to N(0,1) values: q8_1 bit-exact, outputs within
  1e-5 * sum|w*x| + 1e-6.
* Routing ids outside [0, E) in the decode and prefill layers: the device
  flags them (MOEX_EDEVICE, bit 1 of the status word), the entry is left out
  of the layer (the oracle gives it weight 0), and the next clean call leaves
  the status word clear.
"""
import numpy as np
import pytest

import synth
from helpers import assert_within, ensure_lib, to_np
from oracle import gemv as og
from oracle import moe as om
from oracle import prefill as op
from oracle import q8_1 as oq

pytestmark = pytest.mark.gpu

BAD_ROUTE = 1


def _set_scale(blocks, row, bits, every=1):
    blocks[row, ::every, 0:2] = np.array([bits], dtype="<u2").view(np.uint8)


@pytest.mark.parametrize("fmt", ["q8_0", "iq4_nl"])
def test_gemv_extreme_scales_and_outliers(fmt):
    import torch
    import moe_expert_gb300 as mx
    ensure_lib()
    rows, K, C = 40, 512, 3
    g = synth.rng(77)
    blocks = synth.weight_blocks(fmt, g, rows, K).copy()
    _set_scale(blocks, 0, 0x0000)           # zero
    _set_scale(blocks, 1, 0x7BFF)           # 65504
    _set_scale(blocks, 2, 0x0001)           # 2^-24, smallest subnormal
    _set_scale(blocks, 3, 0x03FF)           # largest subnormal
    _set_scale(blocks, 4, 0x8000, every=2)  # negative zero in every other block
    _set_scale(blocks, 5, 0xFBFF, every=3)  # -65504
    x = synth.activations(g, C, K)
    x[0] = 0.0                              # all-zero column
    x[1, 100], x[1, 301], x[1, 511] = 3e4, -3e4, 3e4
    W = mx.PackedWeight.from_gguf(fmt, blocks)
    xq, xds = mx.quantize_q8_1(torch.from_numpy(x).cuda())
    y = to_np(mx.qgemv(W, xq, xds))
    rq, rd, rs = oq.quantize_q8_1(x)
    assert np.array_equal(to_np(xq), rq)
    assert np.array_equal(to_np(xds)[..., 0].view(np.uint32), rd.astype(np.float32).view(np.uint32))
    ref, A = og.gemv(fmt, blocks, rq, rd)
    assert_within(y, ref, A, f"{fmt} extreme scales")
    assert np.all(y[:, 0] == 0.0)           # zero-scale row
    assert np.all(y[0] == 0.0)              # zero column
    assert mx.device_status() == 0


def _decode_weights(E, hidden, inter, seed):
    import moe_expert_gb300 as mx
    gu = mx.PackedWeight("q8_0", E, 2 * inter, hidden)
    dn = mx.PackedWeight("iq4_nl", E, hidden, inter)
    gub, dnb = {}, {}
    for e in range(E):
        gub[e] = synth.expert_blocks("gate_up", e, hidden, inter, "q8_0", seed=seed)
        dnb[e] = synth.expert_blocks("down", e, hidden, inter, "iq4_nl", seed=seed)
        gu.pack_matrix(e, gub[e])
        dn.pack_matrix(e, dnb[e])
    return gu, dn, gub, dnb


def test_decode_invalid_ids_flagged_and_left_out():
    import torch
    import moe_expert_gb300 as mx
    ensure_lib()
    T, k, E, hidden, inter = 2, 4, 8, 256, 64
    g = synth.rng(91)
    x = synth.activations(g, T, hidden)
    ids, w = om.route_topk(synth.router_logits(g, T, E), k)
    gu, dn, gub, dnb = _decode_weights(E, hidden, inter, seed=91)
    bad = ids.copy()
    bad[0, 0], bad[1, 2] = -1, E
    xt = torch.from_numpy(x).cuda()
    wt = torch.from_numpy(w.astype(np.float32)).cuda()
    out = to_np(mx.moe_decode(gu, dn, xt, torch.from_numpy(bad.astype(np.int32)).cuda(), wt))
    assert mx.device_status() & BAD_ROUTE
    # the oracle with those two slots on a valid expert at weight 0
    ids0, w0 = ids.copy(), w.astype(np.float32).astype(np.float64)
    w0[0, 0] = w0[1, 2] = 0.0
    ref = om.moe_decode(gub, dnb, x, ids0, w0, down_fmt="iq4_nl")
    scale = np.abs(ref["out"]).max()
    assert np.abs(out - ref["out"]).max() <= 1e-3 * scale
    # a clean call afterwards
    out2 = to_np(mx.moe_decode(gu, dn, xt, torch.from_numpy(ids.astype(np.int32)).cuda(), wt))
    assert mx.device_status() == 0
    full = om.moe_decode(gub, dnb, x, ids, w.astype(np.float32).astype(np.float64), down_fmt="iq4_nl")
    assert np.abs(out2 - full["out"]).max() <= 1e-3 * np.abs(full["out"]).max()


def test_prefill_invalid_ids_flagged_and_left_out():
    import torch
    import moe_expert_gb300 as mx
    ensure_lib()
    T, k, E, hidden, inter = 96, 2, 4, 256, 64
    g = synth.rng(93)
    xb = synth.bf16_activations(g, T, hidden)
    ids, w = om.route_topk(synth.router_logits(g, T, E), k)
    gu = mx.PackedWeight("iq4_nl", E, 2 * inter, hidden)
    dn = mx.PackedWeight("iq4_nl", E, hidden, inter)
    gub, dnb = {}, {}
    for e in range(E):
        gub[e] = synth.expert_blocks("gate_up", e, hidden, inter, "iq4_nl", seed=93)
        dnb[e] = synth.expert_blocks("down", e, hidden, inter, "iq4_nl", seed=93)
        gu.pack_matrix(e, gub[e])
        dn.pack_matrix(e, dnb[e])
    bad = ids.copy()
    bad[3, 1], bad[50, 0], bad[95, 1] = E, -7, 1 << 30
    xt = torch.from_numpy(xb.view(np.int16)).cuda()
    wt = torch.from_numpy(w.astype(np.float32)).cuda()
    ws = torch.zeros(mx.moe_prefill_workspace_bytes(T, k, E, hidden, inter), dtype=torch.uint8, device="cuda")
    out = to_np(mx.moe_prefill(gu, dn, xt, torch.from_numpy(bad.astype(np.int32)).cuda(), wt, ws=ws))
    assert mx.device_status() & BAD_ROUTE
    off = mx.moe_prefill_workspace_layout(T, k, E, hidden, inter)
    totals = to_np(ws)[off[5]:off[5] + 16].view(np.int32)
    assert totals[2] == T * k - 3          # placed rows
    ids0, w0 = ids.copy(), w.astype(np.float32).astype(np.float64)
    w0[3, 1] = w0[50, 0] = w0[95, 1] = 0.0
    ref = op.moe_prefill(gub, dnb, xb, ids0, w0)
    assert np.abs(out - ref["out"]).max() <= 1e-3 * np.abs(ref["out"]).max()
    out2 = to_np(mx.moe_prefill(gu, dn, xt, torch.from_numpy(ids.astype(np.int32)).cuda(), wt, ws=ws))
    assert mx.device_status() == 0
    full = op.moe_prefill(gub, dnb, xb, ids, w.astype(np.float32).astype(np.float64))
    assert np.abs(out2 - full["out"]).max() <= 1e-3 * np.abs(full["out"]).max()
