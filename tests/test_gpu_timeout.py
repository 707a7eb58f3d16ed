"""The failure path of the bounded device waits, driven on purpose.

Every spin or mbarrier wait in the kernels gives up after a time limit, sets a
bit of the device status word and lets the kernel return, so a stalled
pipeline is reported instead of hanging the GPU.  moex_debug_qgemv_starved
launches the ring GEMV with its copy producer switched off (it issues no copy
at all) and a 1 ms limit: every consumer's wait for its first stage runs out.
The test checks that the call returns, that moex_device_status reports
MOEX_ETIMEOUT with the copy-pipeline bit and clears the word, and that the
next regular call on the same context is correct and leaves the word clear.
Nothing faults, traps or hangs: no copy is ever issued, and each wait ends
after 1 ms.
"""
import ctypes
import time

import numpy as np
import pytest

import synth
from helpers import assert_within, ensure_lib, to_np
from oracle import gemv as og
from oracle import q8_1 as oq

pytestmark = pytest.mark.gpu

MOEX_ETIMEOUT = 5
DEV_TIMEOUT_PIPE = 2


@pytest.mark.parametrize("fmt", ["q8_0", "iq4_nl"])
def test_starved_pipeline_times_out_and_the_next_call_is_clean(fmt):
    import torch
    import moe_expert_gb300 as mx
    L = ensure_lib()
    rows, K = 4 * 152 + 13, 2560  # several rows per CTA and a ragged tail
    blocks = synth.weight_blocks(fmt, synth.rng(7), rows, K)
    W = mx.PackedWeight.from_gguf(fmt, blocks)
    x = synth.activations(synth.rng(8), 1, K)
    xq, xds = mx.quantize_q8_1(torch.from_numpy(x).cuda())
    y = torch.zeros((1, rows), dtype=torch.float32, device="cuda")
    assert mx.device_status() == 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t0 = time.perf_counter()
    st = L.moex_debug_qgemv_starved(ctypes.byref(W.struct), ctypes.c_void_p(xq.data_ptr()),
                                    ctypes.c_void_p(xds.data_ptr()), 1, ctypes.c_void_p(y.data_ptr()), rows,
                                    1_000_000, stream)
    assert st == 0
    flags = ctypes.c_uint32(0)
    st = L.moex_device_status(stream, ctypes.byref(flags))
    waited = time.perf_counter() - t0
    assert st == MOEX_ETIMEOUT, mx.lib().moex_status_string(st)
    assert flags.value & DEV_TIMEOUT_PIPE
    assert waited < 1.0  # the 1 ms limit ended the waits, not the 2 s default
    # the word was cleared, and the context still runs a correct GEMV
    assert mx.device_status() == 0
    got = to_np(mx.qgemv(W, xq, xds))
    assert mx.device_status() == 0
    q, d, _ = oq.quantize_q8_1(x)
    ref, A = og.gemv(fmt, blocks, q, d)
    assert_within(got, ref, A, f"{fmt} after the starved call")


def test_starved_hook_validates_its_arguments():
    import torch
    import moe_expert_gb300 as mx
    L = ensure_lib()
    W = mx.PackedWeight("q8_0", 1, 64, 256).zero_()
    xq = torch.zeros((2, 256), dtype=torch.int8, device="cuda")
    xds = torch.zeros((2, 8, 2), dtype=torch.float32, device="cuda")
    y = torch.zeros((2, 64), dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.moex_debug_qgemv_starved(ctypes.byref(W.struct), p(xq), p(xds), 2, p(y), 64, 1_000_000, s) == 1
    assert L.moex_debug_qgemv_starved(ctypes.byref(W.struct), p(xq), p(xds), 1, p(y), 64, 10, s) == 1
    assert L.moex_debug_qgemv_starved(ctypes.byref(W.struct), p(xq), p(xds), 1, p(y), 64, 3_000_000_000, s) == 1
    assert mx.device_status() == 0
