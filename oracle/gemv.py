"""Block-quantized weight x q8_1 activation GEMV (oracle; test infrastructure only).

What is computed (#242 What it does: a dot split into a weight-side load and an
activation-side apply; #1424 What changed: Q8_0 weights on q8_1 activations for
1-8 columns):

    I[c, r, b] = sum_{i<32} qw[r, 32b+i] * qx[c, 32b+i]           (int32, exact)
    y[c, r]    = sum_b fp32(dw[r, b]) * dx[c, b] * I[c, r, b]      (here float64)

where qw are the weight quants (Q8_0: int8; IQ4_NL: codebook values) and
(qx, dx) the q8_1 activation block.  Every GPU summation order of these terms
is a correct answer; the pass rule used by the tests is

    |y_gpu - y_ref| <= 1e-5 * A[c, r] + 1e-6,
    A[c, r] = sum_b |dw * dx| * sum_i |qw_i * qx_i|,

the per-element form of #1424's "max relative error < 1e-5" against a CPU
double reference.  With at most a few hundred blocks and three FP32 roundings
per block the FP32 error is below (nb + 3) * 2^-24 * A, under that bound for
any K up to ~160k.
"""
from __future__ import annotations

import numpy as np

from . import formats

QK = 32


def block_dots(wq: np.ndarray, xq: np.ndarray) -> np.ndarray:
    """I[c, r, b] = sum_i wq[r, 32b+i] * xq[c, 32b+i], int64 (exact).

    wq: integer quants [R, K]; xq: integer quants [C, K]."""
    R, K = wq.shape
    C = xq.shape[0]
    nb = K // QK
    w = wq.astype(np.int64).reshape(R, nb, QK)
    x = xq.astype(np.int64).reshape(C, nb, QK)
    return np.einsum('rbi,cbi->crb', w, x)


def block_abs_dots(wq: np.ndarray, xq: np.ndarray) -> np.ndarray:
    """sum_i |wq * xq| per block, int64 [C, R, nb]."""
    return block_dots(np.abs(wq.astype(np.int64)), np.abs(xq.astype(np.int64)))


def gemv_planes(dw: np.ndarray, wq: np.ndarray, dx: np.ndarray, xq: np.ndarray):
    """y [C, R] float64 and the error scale A [C, R] from decoded planes.

    dw [R, nb] weight scales, wq [R, K] weight quants, dx [C, nb] activation
    scales, xq [C, K] activation quants."""
    I = block_dots(wq, xq).astype(np.float64)                  # [C, R, nb]
    Iabs = block_abs_dots(wq, xq).astype(np.float64)
    scale = dw.astype(np.float64)[None, :, :] * dx.astype(np.float64)[:, None, :]
    y = np.sum(scale * I, axis=2)
    A = np.sum(np.abs(scale) * Iabs, axis=2)
    return y, A


def gemv(fmt: str, blocks: np.ndarray, xq: np.ndarray, dx: np.ndarray):
    """y [C, R] (float64) and error scale A [C, R] for a weight matrix given as
    GGUF blocks [R, nb, bytes] and q8_1 activations (xq int8 [C, K], dx [C, nb])."""
    dw, wq = formats.decode(fmt, blocks)
    return gemv_planes(dw, wq, np.asarray(dx), np.asarray(xq))


def tolerance(A: np.ndarray) -> np.ndarray:
    """Per-element pass bound 1e-5 * A + 1e-6."""
    return 1e-5 * A + 1e-6
