"""The allocation-free decode entry point (moex_moe_decode_noalloc).

Some callers cannot allocate device memory (code inside another framework's
memory pool, plug-ins that may not allocate after start-up, decode paths that
must never call cudaMalloc); this entry point runs the decode layer on a
workspace compiled into the library.  The test calls it through the C ABI
twice in a row, with different inputs each time, and checks each result
against the regular entry point on the same inputs, within the GEMV pass
rule used by the other tests (1e-5 * sum|w*x| + 1e-6 per element).  This file
is collected last so that a run stopping at the first failure has already
run every other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import synth
from helpers import assert_within, ensure_lib, to_np
from oracle import moe as om

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_regular_entry_point_twice():
    import torch
    import moe_expert_gb300 as mx
    L = ensure_lib()
    T, k, E, hidden, inter = 3, 4, 16, 512, 256
    gu = mx.PackedWeight("q8_0", E, 2 * inter, hidden).zero_()
    dn = mx.PackedWeight("iq4_nl", E, hidden, inter).zero_()
    gub, dnb = {}, {}
    for e in range(E):
        gub[e] = synth.expert_blocks("gate_up", e, hidden, inter, "q8_0", seed=9)
        dnb[e] = synth.expert_blocks("down", e, hidden, inter, "iq4_nl", seed=9)
        gu.pack_matrix(e, gub[e])
        dn.pack_matrix(e, dnb[e])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        g = synth.rng(100 + call)
        x = synth.activations(g, T, hidden)
        ids, w = om.route_topk(synth.router_logits(g, T, E), k)
        xt = torch.from_numpy(x).cuda()
        it = torch.from_numpy(ids.astype(np.int32)).cuda()
        wt = torch.from_numpy(w.astype(np.float32)).cuda()
        ref = to_np(mx.moe_decode(gu, dn, xt, it, wt))
        out = torch.full((T, hidden), float("nan"), device="cuda")
        st = L.moex_moe_decode_noalloc(ctypes.byref(gu.struct), ctypes.byref(dn.struct),
                                       ctypes.c_void_p(xt.data_ptr()), T, ctypes.c_void_p(it.data_ptr()),
                                       ctypes.c_void_p(wt.data_ptr()), k, ctypes.c_void_p(out.data_ptr()), stream)
        assert st == 0, mx.lib().moex_status_string(st)
        got = to_np(out)
        assert mx.device_status() == 0
        scale = om.moe_decode(gub, dnb, x, ids, w.astype(np.float32))["out_A"]
        assert_within(got, ref.astype(np.float64), scale, f"call {call}")


def test_noalloc_rejects_layers_beyond_the_built_in_buffer():
    import moe_expert_gb300 as mx
    L = ensure_lib()
    # 8 tokens x top-8 x inter 8192 needs more than the 512 KiB buffer
    gu = mx.QWeight(1, 4, 2 * 8192, 1024, 16, 16)
    dn = mx.QWeight(2, 4, 1024, 8192, 16, 16)
    null = ctypes.c_void_p(0)
    assert L.moex_moe_decode_noalloc(ctypes.byref(gu), ctypes.byref(dn), null, 8, null, null, 8, null, null) == 7
