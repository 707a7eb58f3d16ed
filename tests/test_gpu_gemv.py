"""Multi-column GEMV on the GPU against the oracle.

Integer block dots: bit-exact.  Float outputs: |gpu - ref| <= 1e-5 * sum|w*x|
+ 1e-6 per element.  Column invariance: every column of a multi-column call is
bitwise equal to a one-column call.  Shapes span several 8-row stages, ragged
row tails, partial K slices (K not a multiple of 512), 1..8 and 11 columns,
and the full-size benchmark workloads.
"""
import numpy as np
import pytest

import synth
from helpers import assert_within, ensure_lib, to_np
from oracle import gemv as og
from oracle import q8_1 as oq

pytestmark = pytest.mark.gpu


def _run(fmt, rows, K, ncols, seed=0):
    import torch
    import moe_expert_gb300 as mx
    ensure_lib()
    g = synth.rng(seed)
    blocks = synth.weight_blocks(fmt, g, rows, K)
    x = synth.activations(g, ncols, K)
    W = mx.PackedWeight.from_gguf(fmt, blocks)
    xq, xds = mx.quantize_q8_1(torch.from_numpy(x).cuda())
    y = mx.qgemv(W, xq, xds)
    torch.cuda.synchronize()
    rq, rd, _ = oq.quantize_q8_1(x)
    assert np.array_equal(to_np(xq), rq)
    ref, A = og.gemv(fmt, blocks, rq, rd)
    return W, xq, xds, to_np(y), ref, A, blocks, rq


SMALL = [
    ("q8_0", 8, 32, 1),
    ("q8_0", 300, 512, 3),
    ("iq4_nl", 301, 1536, 5),
    ("q8_0", 1000, 2560, 8),
    ("iq4_nl", 77, 96, 2),
    ("iq4_nl", 1000, 2560, 7),
    ("q8_0", 517, 4096, 4),
    ("iq4_nl", 257, 7680, 6),
    ("q8_0", 33, 2048, 11),
    ("iq4_nl", 1, 64, 1),
]


@pytest.mark.parametrize("fmt,rows,K,ncols", SMALL)
def test_gemv_small(fmt, rows, K, ncols):
    import moe_expert_gb300 as mx
    _, _, _, y, ref, A, _, _ = _run(fmt, rows, K, ncols, seed=rows + K)
    assert_within(y, ref, A, f"{fmt} {rows}x{K} c{ncols}")
    assert mx.device_status() == 0


@pytest.mark.parametrize("fmt", ["q8_0", "iq4_nl"])
def test_block_dots_bit_exact(fmt):
    import moe_expert_gb300 as mx
    W, xq, xds, y, ref, A, blocks, rq = _run(fmt, 200, 2560, 3, seed=5)
    dots = to_np(mx.qgemv_block_dots(W, xq))
    from oracle import formats
    _, wq = formats.decode(fmt, blocks)
    assert np.array_equal(dots.astype(np.int64), og.block_dots(wq, rq))


@pytest.mark.parametrize("fmt,rows,K", [("q8_0", 129, 2560), ("iq4_nl", 129, 2560), ("iq4_nl", 129, 1536),
                                         ("q8_0", 129, 96),
                                         # more than one round of 16-row tiles a CTA, ragged last round
                                         ("q8_0", 10500, 2560), ("iq4_nl", 13001, 2560), ("q8_0", 60001, 480)])
def test_columns_bitwise_equal_single_column_calls(fmt, rows, K):
    import torch
    import moe_expert_gb300 as mx
    W, xq, xds, y, ref, A, _, _ = _run(fmt, rows, K, 8, seed=9)
    assert_within(y, ref, A, f"{fmt} {rows}x{K} c8")
    for c in range(8):
        y1 = to_np(mx.qgemv(W, xq[c:c + 1].contiguous(), xds[c:c + 1].contiguous()))
        assert np.array_equal(y1[0].view(np.uint32), y[c].view(np.uint32)), c
    for n in [2, 3, 5]:
        yn = to_np(mx.qgemv(W, xq[:n].contiguous(), xds[:n].contiguous()))
        assert np.array_equal(yn.view(np.uint32), y[:n].view(np.uint32)), n


def test_repeat_calls_identical():
    import moe_expert_gb300 as mx
    W, xq, xds, y, _, _, _, _ = _run("iq4_nl", 640, 2560, 4, seed=3)
    for _ in range(3):
        y2 = to_np(mx.qgemv(W, xq, xds))
        assert np.array_equal(y2.view(np.uint32), y.view(np.uint32))


# -------------------------------------------------------- full-size workloads

def test_config_q8_0_512x2048_one_column():
    _, _, _, y, ref, A, _, _ = _run("q8_0", 512, 2048, 1, seed=0)
    assert_within(y, ref, A, "q8_0 512x2048")


@pytest.mark.parametrize("ncols", [1, 2, 4, 8])
def test_config_q8_0_8192x2560(ncols):
    _, _, _, y, ref, A, _, _ = _run("q8_0", 8192, 2560, ncols, seed=0)
    assert_within(y, ref, A, f"q8_0 8192x2560 c{ncols}")


@pytest.mark.parametrize("ncols", [1, 2, 3, 4, 8])
def test_config_iq4_nl_12288x2560(ncols):
    _, _, _, y, ref, A, _, _ = _run("iq4_nl", 12288, 2560, ncols, seed=0)
    assert_within(y, ref, A, f"iq4_nl 12288x2560 c{ncols}")


@pytest.mark.parametrize("fmt,ncols", [("q8_0", 3), ("iq4_nl", 11)])
def test_strided_output_leaves_padding(fmt, ncols):
    """y with a leading dimension above rows: column c at y + c*ldy; the
    padding between columns is never written."""
    import torch
    import moe_expert_gb300 as mx
    rows, K, pad = 300, 1024, 37
    W, xq, xds, y, ref, A, _, _ = _run(fmt, rows, K, ncols, seed=21)
    big = torch.full((ncols, rows + pad), float("nan"), dtype=torch.float32, device="cuda")
    mx.qgemv(W, xq, xds, big[:, :rows])
    got = to_np(big)
    assert np.array_equal(got[:, :rows].view(np.uint32), y.view(np.uint32))
    assert np.all(np.isnan(got[:, rows:]))


# -------------------------------------------------------- vocabulary-sized head

@pytest.mark.parametrize("ncols", [1, 8])
def test_q8_0_vocab_head_sampled_rows(ncols):
    """A vocabulary-sized Q8_0 output head, 128256 x 2560 (349 MB of blocks),
    beyond the register-staged kernel's row limit: every row is computed on
    the GPU, and the oracle checks 600 sampled rows (first, last, random)."""
    import torch
    import moe_expert_gb300 as mx
    ensure_lib()
    rows, K = 128256, 2560
    blocks, x = synth.dense_case("q8_0", rows, K, ncols, seed=31)
    W = mx.PackedWeight.from_gguf("q8_0", blocks)
    xq, xds = mx.quantize_q8_1(torch.from_numpy(x).cuda())
    y = to_np(mx.qgemv(W, xq, xds))
    assert mx.device_status() == 0
    rq, rd, _ = oq.quantize_q8_1(x)
    g = np.random.default_rng(5)
    sample = np.unique(np.concatenate([[0, 1, rows - 1], g.integers(0, rows, 597)]))
    ref, A = og.gemv("q8_0", blocks[sample], rq, rd)
    assert_within(y[:, sample], ref, A, f"q8_0 head c{ncols}")
    assert np.all(np.isfinite(y))
