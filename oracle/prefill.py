"""The grouped MoE prefill layer on FP16 operands (oracle; test infrastructure only).

What is computed (#2356 Summary: prompt rows sorted by expert, IQ4_NL weights
dequantised to FP16 for the tensor cores with FP32 sums; #1525 Change: each
dequantised value is one expression rounded by ``__float2half_rn``, SwiGLU
between the two products, the top-k outputs combined):

    ids, w  = top-k of the router logits, softmax over the k (as in decode)
    order   = the (token, slot) entries sorted by expert, ties by entry index
    Xh      = fp16_rn(x)                          x given as BF16
    Wh      = fp16_rn(fp32(d) * kvalues[idx])     one rounding of an exact product
    g, u    = Wh_gu[e] . Xh[t]                    here in float64
    H       = fp16_rn(silu(g) * u)                H is FP16, the second GEMM's input
    o       = Wh_dn[e] . H                        float64
    out[t]  = sum_{k ascending} w[t, k] * o[(t, k)]

Readings (pages silent): H is rounded to FP16 once from the exact value; the
sort is stable by token, which does not change any result.

The integer route of the same layer (``moe_prefill_q8``; #1525 Change: the
prompt path's SwiGLU fused with the q8_1 quantisation of H, ``swiglu_quant``
writing q8_1 rows for the down product, ``quantize_mmq_q8_1``) keeps the
first product on FP16 operands and replaces the second:

    H       = silu(g) * u                         FP32, no FP16 rounding
    Hq, Hd  = q8_1(H)                             per 32-feature block
    o       = sum_b fp32(dw[r,b]) * Hd[b] * I_b   the block-integer GEMV of gemv.py
    out[t]  = sum_{k ascending} w[t, k] * o[(t, k)]

Reading (pages silent): H reaches the quantiser as the FP32 value of
silu(g) * u, exactly as the decode layer's H does.
"""
from __future__ import annotations

import numpy as np

from . import formats
from . import gemv as _gemv
from . import moe as _moe
from . import q8_1 as _q8_1


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns to FP32 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def fp16_rn(x: np.ndarray) -> np.ndarray:
    """Round to FP16, nearest even, straight from the given precision.
    Magnitudes past the FP16 range become inf, as IEEE rounding gives."""
    with np.errstate(over="ignore"):
        return np.asarray(x).astype(np.float16)


def dequant_fp16(fmt: str, blocks: np.ndarray) -> np.ndarray:
    """fp16_rn(fp32(d) * q) as float16 [rows, K].  The FP32 product is exact
    (11-bit scale significand times a 7-bit integer), so this is one rounding."""
    d, q = formats.decode(fmt, blocks)
    rows, nb = d.shape
    prod32 = (np.repeat(d.astype(np.float32), 32, axis=1) * q.astype(np.float32))
    return fp16_rn(prod32.reshape(rows, nb * 32))


def sort_entries(ids: np.ndarray, n_experts: int):
    """Entries t*k+slot sorted by expert, ties by entry index (stable).

    Returns (order int64 [T*k], offsets int64 [n_experts+1])."""
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    order = np.argsort(flat, kind='stable')
    counts = np.bincount(flat, minlength=n_experts)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    return order, offsets


class ExpertCache:
    """Dequantised FP16 experts, built on first use (kept as float16, handed
    out as float64; every FP16 value is exact in float64)."""

    def __init__(self, fmt: str, blocks_of):
        self.fmt, self.blocks_of, self.cache = fmt, blocks_of, {}

    def __getitem__(self, e: int) -> np.ndarray:
        if e not in self.cache:
            self.cache[e] = dequant_fp16(self.fmt, self.blocks_of[e])
        return self.cache[e].astype(np.float64)


def dense_prefill(blocks, x_bf16: np.ndarray, fmt: str = "iq4_nl", rows=None):
    """The dense prefill product (#1525 Change: dense weights dequantised to
    FP16 for the prompt product, one rounding per value, FP32 sums; here
    the sums are float64): y[t][r] = sum_i Wh[r, i] * Xh[t, i] with
    Wh = fp16_rn(fp32(d) * kv) and Xh = fp16_rn(bf16 x).

    blocks: GGUF blocks [R, K/32, *]; ``rows`` restricts the output to those
    weight rows.  Returns (y [T, len(rows)] float64, error scale
    A = |Wh| . |Xh|^T)."""
    b = blocks if rows is None else blocks[np.asarray(rows)]
    wh = dequant_fp16(fmt, b).astype(np.float64)
    xh = fp16_rn(bf16_bits_to_f32(x_bf16)).astype(np.float64)
    return xh @ wh.T, np.abs(xh) @ np.abs(wh).T


def moe_prefill(gate_up, down, x_bf16: np.ndarray, ids: np.ndarray, w: np.ndarray,
                tokens=None, fmt: str = "iq4_nl", h_override=None, down_fmt=None):
    """Prefill output rows for ``tokens`` (default: every token).

    gate_up[e]: GGUF blocks [2*inter, hidden/32, *]; down[e]: [hidden, inter/32, *].
    x_bf16: uint16 [T, hidden].  ids, w: [T, k].
    ``h_override(t, slot)`` may return an FP16 H row that replaces the oracle's
    (the tests use it to check the second product on the GPU's own H).

    Returns dict: tokens, out [n, hidden] float64, out_A (error scale),
    g, u, H (float16) [n, k, inter] and gu_A [n, k, 2*inter]."""
    T, hidden = x_bf16.shape
    k = ids.shape[1]
    if tokens is None:
        tokens = list(range(T))
    Wgu = ExpertCache(fmt, gate_up)
    Wdn = ExpertCache(down_fmt or fmt, down)
    inter = Wgu[int(ids[tokens[0], 0])].shape[0] // 2
    n = len(tokens)
    G = np.zeros((n, k, inter))
    U = np.zeros((n, k, inter))
    Hs = np.zeros((n, k, inter), dtype=np.float16)
    gu_A = np.zeros((n, k, 2 * inter))
    O = np.zeros((n, k, hidden))
    O_A = np.zeros((n, k, hidden))
    Xh = fp16_rn(bf16_bits_to_f32(x_bf16[np.asarray(tokens)])).astype(np.float64)   # [n, hidden]
    # every (token, slot) entry of each expert, experts in ascending order (the
    # rows sorted by expert of #2356), so each expert's weights are expanded once
    ent = {}
    for i, t in enumerate(tokens):
        for s in range(k):
            ent.setdefault(int(ids[t, s]), []).append((i, s))
    for e in sorted(ent):
        ii = np.array([i for i, _ in ent[e]])
        ss = np.array([s for _, s in ent[e]])
        wg = Wgu[e]
        gu = Xh[ii] @ wg.T                                   # [m, 2*inter], float64 sums
        gu_A[ii, ss] = np.abs(Xh[ii]) @ np.abs(wg).T
        G[ii, ss], U[ii, ss] = gu[:, :inter], gu[:, inter:]
        if h_override is not None:
            h = np.stack([np.asarray(h_override(tokens[i], s), dtype=np.float16) for i, s in ent[e]])
        else:
            h = fp16_rn(_moe.silu(gu[:, :inter]) * gu[:, inter:])
        Hs[ii, ss] = h
        wd = Wdn[e]
        hf = h.astype(np.float64)
        O[ii, ss] = hf @ wd.T
        O_A[ii, ss] = np.abs(hf) @ np.abs(wd).T
    # the top-k combine, slots in ascending order
    out = np.zeros((n, hidden))
    out_A = np.zeros((n, hidden))
    for i, t in enumerate(tokens):
        for s in range(k):
            out[i] += float(w[t, s]) * O[i, s]
            out_A[i] += abs(float(w[t, s])) * O_A[i, s]
    return dict(tokens=tokens, out=out, out_A=out_A, g=G, u=U, H=Hs, gu_A=gu_A)


def moe_prefill_q8(gate_up, down, x_bf16: np.ndarray, ids: np.ndarray, w: np.ndarray,
                   tokens=None, fmt: str = "iq4_nl", h_override=None, down_fmt=None):
    """The integer route of the prefill layer for ``tokens`` (default: every
    token): the first product as in ``moe_prefill`` (FP16 operands, float64
    sums), H = silu(g) * u taken to FP32, q8_1 of H per 32-feature block,
    then the down product as block-integer dots (the GEMV of #1424 / #242)
    and the top-k combine in slot order.

    ``h_override(t, slot)`` may return an FP32 H row that replaces the
    oracle's before its quantisation (the tests quantise the GPU's own H).

    Returns dict: tokens, out [n, hidden] float64, out_A (error scale of the
    combine), g, u, H (float64) [n, k, inter], Hq int8 [n, k, inter], Hd
    float32 [n, k, inter/32], gu_A [n, k, 2*inter]."""
    T, hidden = x_bf16.shape
    k = ids.shape[1]
    if tokens is None:
        tokens = list(range(T))
    Wgu = ExpertCache(fmt, gate_up)
    inter = Wgu[int(ids[tokens[0], 0])].shape[0] // 2
    n = len(tokens)
    G = np.zeros((n, k, inter))
    U = np.zeros((n, k, inter))
    gu_A = np.zeros((n, k, 2 * inter))
    Hq = np.zeros((n, k, inter), dtype=np.int8)
    Hd = np.zeros((n, k, inter // 32), dtype=np.float32)
    O = np.zeros((n, k, hidden))
    O_A = np.zeros((n, k, hidden))
    Xh = fp16_rn(bf16_bits_to_f32(x_bf16[np.asarray(tokens)])).astype(np.float64)
    ent = {}
    for i, t in enumerate(tokens):
        for s in range(k):
            ent.setdefault(int(ids[t, s]), []).append((i, s))
    for e in sorted(ent):
        ii = np.array([i for i, _ in ent[e]])
        ss = np.array([s for _, s in ent[e]])
        wg = Wgu[e]
        gu = Xh[ii] @ wg.T
        gu_A[ii, ss] = np.abs(Xh[ii]) @ np.abs(wg).T
        G[ii, ss], U[ii, ss] = gu[:, :inter], gu[:, inter:]
        if h_override is not None:
            h32 = np.stack([np.asarray(h_override(tokens[i], s), dtype=np.float32) for i, s in ent[e]])
        else:
            h32 = (_moe.silu(gu[:, :inter]) * gu[:, inter:]).astype(np.float32)
        q, d, _ = _q8_1.quantize_q8_1(h32)
        Hq[ii, ss] = q
        Hd[ii, ss] = d
        y, A = _gemv.gemv(down_fmt or fmt, down[e], q, d)
        O[ii, ss] = y
        O_A[ii, ss] = A
    out = np.zeros((n, hidden))
    out_A = np.zeros((n, hidden))
    for i, t in enumerate(tokens):
        for s in range(k):
            out[i] += float(w[t, s]) * O[i, s]
            out_A[i] += abs(float(w[t, s])) * O_A[i, s]
    H = _moe.silu(G) * U
    return dict(tokens=tokens, out=out, out_A=out_A, g=G, u=U, H=H, Hq=Hq, Hd=Hd, gu_A=gu_A)
