"""Routing, SwiGLU and the grouped MoE decode layer (oracle; test infrastructure only).

The layer (#242 What it does: ``native_gu_kernel`` / ``native_down_kernel`` run
every entry of an expert group; #1525 Change: ``mmq::swiglu_quant`` with split
gate/up, ``moe_combine4`` summing the top-k outputs):

    xq[t]   = q8_1(x[t])
    gu[j]   = W_gu[e_j] . xq[t_j]          rows 0..I-1 are gate, I..2I-1 up
    H[j]    = silu(g) * u,  silu(g) = g / (1 + exp(-g))
    Hq[j]   = q8_1(H[j])
    o[j]    = W_dn[e_j] . Hq[j]
    out[t]  = sum_{k ascending} w[t, k] * o[(t, k)]

Readings (pages silent): split gate/up layout (the GGUF one, first of the two
#1525 lists); plain SiLU with no clamp; router weights = softmax over the k
selected logits (max subtracted); top-k ties go to the lower expert id; the k
slots are ordered by descending logit.
"""
from __future__ import annotations

import numpy as np

from . import gemv as _gemv
from . import q8_1 as _q8_1


def route_topk(logits: np.ndarray, k: int):
    """Top-k experts per token and softmax weights over the selected logits.

    logits: FP32 [T, E].  Returns ids int64 [T, k] (descending logit, ties to
    the lower id) and w float64 [T, k]."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), dtype=np.int64)
    for t in range(T):
        # stable sort on -logit keeps equal logits in ascending id order
        order = np.argsort(-logits[t].astype(np.float64), kind='stable')
        ids[t] = order[:k]
    sel = np.take_along_axis(logits, ids, axis=1).astype(np.float64)
    m = sel.max(axis=1, keepdims=True)
    e = np.exp(sel - m)
    w = e / e.sum(axis=1, keepdims=True)
    return ids, w


def silu(g: np.ndarray) -> np.ndarray:
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def swiglu(gu: np.ndarray, inter: int) -> np.ndarray:
    """H = silu(g) * u for stacked [..., 2*inter] gate/up outputs (split)."""
    gu = np.asarray(gu, dtype=np.float64)
    return silu(gu[..., :inter]) * gu[..., inter:2 * inter]


def entry_groups(ids: np.ndarray):
    """Group the T*k (token, slot) entries by expert.

    Returns a list of (expert, [entry indices]) with experts ascending and
    entries ascending inside each group; entry j = t*k + slot."""
    flat = np.asarray(ids).reshape(-1)
    groups = []
    for e in sorted(set(int(v) for v in flat)):
        groups.append((e, [j for j in range(flat.size) if int(flat[j]) == e]))
    return groups


def moe_decode(gate_up, down, x: np.ndarray, ids: np.ndarray, w: np.ndarray,
               gate_up_fmt: str = "q8_0", down_fmt: str = "iq4_nl",
               h_override=None):
    """The grouped MoE decode layer.

    gate_up[e]: GGUF blocks [2*inter, hidden/32, *]; down[e]: [hidden, inter/32, *]
    (any indexable of experts).  x FP32 [T, hidden]; ids [T, k]; w [T, k].

    ``h_override`` (float32 [T*k, inter]) replaces H before its quantisation;
    the tests use it to quantise the GPU's own H and check each later stage on
    identical inputs.

    Returns a dict with xq, xd, gu [T*k, 2I], gu_A (error scale), H [T*k, I]
    (float64), Hq, Hd, o [T*k, hidden], o_A, out [T, hidden] and out_A
    (error scale of the combine of o)."""
    x = np.asarray(x, dtype=np.float32)
    T, hidden = x.shape
    k = ids.shape[1]
    n = T * k
    xq, xd, _ = _q8_1.quantize_q8_1(x)
    first = gate_up[int(ids.reshape(-1)[0])]
    inter = first.shape[0] // 2
    gu = np.zeros((n, 2 * inter))
    gu_A = np.zeros((n, 2 * inter))
    for e, entries in entry_groups(ids):
        toks = [j // k for j in entries]
        y, A = _gemv.gemv(gate_up_fmt, gate_up[e], xq[toks], xd[toks])
        gu[entries] = y
        gu_A[entries] = A
    H = swiglu(gu, inter)
    H32 = H.astype(np.float32) if h_override is None else np.asarray(h_override, np.float32)
    Hq, Hd, Hs = _q8_1.quantize_q8_1(H32)
    o = np.zeros((n, hidden))
    o_A = np.zeros((n, hidden))
    for e, entries in entry_groups(ids):
        y, A = _gemv.gemv(down_fmt, down[e], Hq[entries], Hd[entries])
        o[entries] = y
        o_A[entries] = A
    wf = np.asarray(w, dtype=np.float64).reshape(n)
    out = np.zeros((T, hidden))
    out_A = np.zeros((T, hidden))
    for t in range(T):
        for s in range(k):
            j = t * k + s
            out[t] += wf[j] * o[j]
            out_A[t] += abs(wf[j]) * o_A[j]
    return dict(xq=xq, xd=xd, gu=gu, gu_A=gu_A, H=H, Hq=Hq, Hd=Hd, Hs=Hs,
                o=o, o_A=o_A, out=out, out_A=out_A)
