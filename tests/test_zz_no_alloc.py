"""The allocation-free decode entry point (moex_moe_decode_noalloc).

Some callers cannot allocate device memory (code inside another framework's
memory pool, plug-ins that may not allocate after start-up, decode paths that
must never call cudaMalloc); this entry point runs the decode layer on a
workspace compiled into the library.  The test calls it through the C ABI
twice in a row, with different inputs each time.  Both entry points run the
same deterministic kernels, so each result must be bitwise equal to the
regular entry point's on the same inputs; the first call is also checked
against the oracle, within the pass rule of the decode tests (1e-5 * sum|w*x|
+ 1e-6 per element, on the GPU's own H).  This file is collected last so that
a run stopping at the first failure has already run every other test; it also
passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import synth
from helpers import assert_within, ensure_lib, to_np
from oracle import moe as om

pytestmark = pytest.mark.gpu

MOEX_EINVAL, MOEX_ENOSPACE = 1, 7


def _noalloc(L, gu, dn, x, ids, w, out, T, k, stream):
    p = lambda t: ctypes.c_void_p(t.data_ptr() if t is not None else 0)  # noqa: E731
    return L.moex_moe_decode_noalloc(ctypes.byref(gu), ctypes.byref(dn), p(x), T, p(ids), p(w), k, p(out), stream)


def test_noalloc_decode_bitwise_equal_to_regular_entry_point_twice():
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
        ref_out, dbg = mx.moe_decode(gu, dn, xt, it, wt, debug=True)
        ref = to_np(ref_out)
        out = torch.full((T, hidden), float("nan"), device="cuda")
        st = _noalloc(L, gu.struct, dn.struct, xt, it, wt, out, T, k, stream)
        assert st == 0, mx.lib().moex_status_string(st)
        got = to_np(out)
        assert mx.device_status() == 0
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), f"call {call}: not bitwise equal"
        if call == 0:
            o = om.moe_decode(gub, dnb, x, ids, w.astype(np.float32), h_override=to_np(dbg["h"]))
            assert np.array_equal(to_np(dbg["hq"]), o["Hq"])
            assert_within(got, o["out"], o["out_A"], "no-alloc decode against the oracle")


def test_noalloc_rejects_layers_beyond_the_built_in_buffer():
    import torch
    import moe_expert_gb300 as mx
    L = ensure_lib()
    # 8 tokens x top-8 x inter 8192 needs more than the 512 KiB buffer; every
    # pointer is a valid, aligned device buffer, so only the size is at fault
    buf = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    ptr = buf.data_ptr()
    gu = mx.QWeight(1, 4, 2 * 8192, 1024, ptr, ptr)
    dn = mx.QWeight(2, 4, 1024, 8192, ptr, ptr)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert mx.moe_decode_workspace_bytes(8, 8, 1024, 8192) > 512 * 1024
    assert _noalloc(L, gu, dn, buf, buf, buf, buf, 8, 8, stream) == MOEX_ENOSPACE
    # a malformed call gets moex_moe_decode's status, not the size verdict
    assert _noalloc(L, gu, dn, None, buf, buf, buf, 8, 8, stream) == MOEX_EINVAL
    assert _noalloc(L, gu, dn, buf, buf, buf, buf, 9, 8, stream) == MOEX_EINVAL
