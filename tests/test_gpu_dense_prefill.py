"""Dense prefill product on the tensor cores (moex_dense_prefill) against the
oracle: y = fp16(W) . fp16(x)^T with FP32 sums, each element within
1e-5 * sum|w*x| + 1e-6.  Shapes span several token and feature tiles, a
ragged last token tile, a single token, an output stride above the row
count (padding untouched), and the full-size 12288 x 2560 matrix over 8192
tokens checked on sampled rows and tokens."""
import numpy as np
import pytest

import synth
from helpers import assert_within, ensure_lib, to_np
from oracle import prefill as op

pytestmark = pytest.mark.gpu


def _run(T, R, K, seed, ldy_pad=0):
    import torch
    import moe_expert_gb300 as mx
    ensure_lib()
    g = synth.rng(seed)
    blocks = synth.iq4_nl_blocks(g, R, K)
    xb = synth.bf16_activations(g, T, K)
    W = mx.PackedWeight.from_gguf("iq4_nl", blocks)
    xt = torch.from_numpy(xb.view(np.int16)).cuda()
    big = torch.full((T, R + ldy_pad), float("nan"), dtype=torch.float32, device="cuda")
    mx.dense_prefill(W, xt, y=big[:, :R])
    y = to_np(big)
    assert mx.device_status() == 0
    if ldy_pad:
        assert np.all(np.isnan(y[:, R:]))
    return blocks, xb, y[:, :R]


@pytest.mark.parametrize("T,R,K", [
    (300, 256, 512),     # two token tiles (192 + 108), two feature tiles
    (1, 128, 64),        # one token, one k-step
    (193, 384, 1536),    # ragged: a one-row last tile; odd feature-tile count
])
def test_dense_prefill_small(T, R, K):
    blocks, xb, y = _run(T, R, K, seed=T + R, ldy_pad=13)
    ref, A = op.dense_prefill(blocks, xb)
    assert_within(y, ref, A, f"dense {T}x{R}x{K}")


def test_dense_prefill_full_size_sampled():
    T, R, K = 8192, 12288, 2560
    blocks, xb, y = _run(T, R, K, seed=7)
    g = np.random.default_rng(3)
    toks = np.unique(np.concatenate([[0, 191, 192, T - 1], g.integers(0, T, 28)]))
    rows = np.unique(np.concatenate([[0, 127, 128, R - 1], g.integers(0, R, 124)]))
    ref, A = op.dense_prefill(blocks, xb[toks], rows=rows)
    assert_within(y[np.ix_(toks, rows)], ref, A, "dense 8192x12288x2560")
    assert np.all(np.isfinite(y))


def _run_fmt(fmt, T, R, K, seed):
    import torch
    import moe_expert_gb300 as mx
    ensure_lib()
    g = synth.rng(seed)
    blocks = synth.weight_blocks(fmt, g, R, K)
    xb = synth.bf16_activations(g, T, K)
    W = mx.PackedWeight.from_gguf(fmt, blocks)
    y = to_np(mx.dense_prefill(W, torch.from_numpy(xb.view(np.int16)).cuda()))
    assert mx.device_status() == 0
    return blocks, xb, y


@pytest.mark.parametrize("T,R,K", [(300, 256, 512), (193, 384, 1536), (70, 128, 192)])
def test_dense_prefill_q8_0(T, R, K):
    """Q8_0 weights: raw stages of two k-steps, Wh = fp16_rn(d * q)."""
    blocks, xb, y = _run_fmt("q8_0", T, R, K, seed=T * 3 + R)
    ref, A = op.dense_prefill(blocks, xb, fmt="q8_0")
    assert_within(y, ref, A, f"dense q8_0 {T}x{R}x{K}")
