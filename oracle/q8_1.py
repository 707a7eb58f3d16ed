"""The q8_1 activation quantiser (oracle; test infrastructure only).

Activations reach the integer GEMV as q8_1 blocks (#1525 Change:
``quantize_mmq_q8_1`` rows for the down product; #1424 What changed: "an int8
plane plus float scales").  Per block of 32 FP32 values x_i:

    amax = max_i |x_i|
    d    = amax / 127            (one IEEE FP32 division)
    q_i  = round(x_i / d)        (one IEEE FP32 division, then round half away
                                  from zero -- C ``roundf``)
    s    = d * float(sum_i q_i)  (one FP32 multiply)

Readings (the pages are silent on these steps):
* ``round`` is C ``roundf``: half away from zero.
* a block with amax == 0 gives d = 0, q = 0, s = 0 (no 0/0).
* d and s are stored as FP32 (the pages' "float scales").
* NaN / Inf inputs are undefined.
"""
from __future__ import annotations

import numpy as np

QK = 32


def round_half_away(r32: np.ndarray) -> np.ndarray:
    """C roundf of FP32 values, computed exactly in float64 (|r| + 0.5 is exact
    in float64 for any FP32 r, so floor() sees the true sum)."""
    r = r32.astype(np.float64)
    return np.sign(r) * np.floor(np.abs(r) + 0.5)


def quantize_q8_1(x: np.ndarray):
    """q8_1 of FP32 activations x [ncols, K] (K a multiple of 32).

    Returns (q int8 [ncols, K], d float32 [ncols, K/32], s float32 [ncols, K/32]).
    """
    x = np.asarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    C, K = x.shape
    assert K % QK == 0
    nb = K // QK
    xb = x.reshape(C, nb, QK)
    amax = np.max(np.abs(xb), axis=2)                       # exact in FP32
    d = (amax / np.float32(127.0)).astype(np.float32)       # FP32 division
    nz = amax > 0
    dsafe = np.where(nz, d, np.float32(1.0)).astype(np.float32)
    ratio = (xb / dsafe[:, :, None]).astype(np.float32)    # FP32 division
    q = round_half_away(ratio)
    q = np.where(nz[:, :, None], q, 0.0)
    assert np.all(np.abs(q) <= 127)
    q = q.astype(np.int8)
    qsum = q.astype(np.int64).sum(axis=2).astype(np.float32)  # exact (|sum| <= 4064)
    s = (d * qsum).astype(np.float32)                        # FP32 multiply
    s = np.where(nz, s, np.float32(0.0)).astype(np.float32)
    d = np.where(nz, d, np.float32(0.0)).astype(np.float32)
    return q.reshape(C, K), d, s

