"""Python binding of the moex C-ABI library (libmoex.so).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C entry points declared in include/moex.h.  PyTorch supplies
device memory (torch tensors) and the current CUDA stream.  There is no CPU
fallback: if the library is missing, every call raises.

The function names follow the C ABI without the ``moex_`` prefix.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoex.so")

FMT = {"q8_0": 1, "iq4_nl": 2}
QK = 32
BLOCK_BYTES = {"q8_0": 34, "iq4_nl": 18}

STATUS = {0: "MOEX_OK", 1: "MOEX_EINVAL", 2: "MOEX_EALIGN", 3: "MOEX_EUNSUPPORTED", 4: "MOEX_ECUDA",
          5: "MOEX_ETIMEOUT", 6: "MOEX_EDEVICE", 7: "MOEX_ENOSPACE"}


class MoexError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class QWeight(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("n_mats", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("K", ctypes.c_int64), ("qs", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_QWP = ctypes.POINTER(QWeight)

# name -> (restype, argtypes); mirrors include/moex.h
SIGNATURES = {
    "moex_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moex_version": (ctypes.c_int, []),
    "moex_weight_plane_bytes": (ctypes.c_int, [ctypes.c_int, _I64, _I64, _I64, ctypes.POINTER(_SZ),
                                               ctypes.POINTER(_SZ)]),
    "moex_weight_pack": (ctypes.c_int, [_QWP, _P, _P]),
    "moex_quantize_q8_1": (ctypes.c_int, [_P, _I64, ctypes.c_int, _I64, _P, _P, _P]),
    "moex_qgemv": (ctypes.c_int, [_QWP, _P, _P, ctypes.c_int, _P, _I64, _P]),
    "moex_qgemv_block_dots": (ctypes.c_int, [_QWP, _P, ctypes.c_int, _P, _P]),
    "moex_debug_qgemv_starved": (ctypes.c_int, [_QWP, _P, _P, ctypes.c_int, _P, _I64, ctypes.c_uint64, _P]),
    "moex_route_topk": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P]),
    "moex_moe_decode_workspace_bytes": (_SZ, [ctypes.c_int, ctypes.c_int, _I64, _I64]),
    "moex_moe_decode": (ctypes.c_int, [_QWP, _QWP, _P, ctypes.c_int, _P, _P, ctypes.c_int, _P, _P, _SZ, _P]),
    "moex_moe_decode_debug": (ctypes.c_int, [_QWP, _QWP, _P, ctypes.c_int, _P, _P, ctypes.c_int, _P, _P, _SZ,
                                             _P, _P, _P, _P, _P]),
    "moex_device_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "moex_moe_prefill_workspace_bytes": (_SZ, [ctypes.c_int, ctypes.c_int, ctypes.c_int, _I64, _I64]),
    "moex_moe_prefill_workspace_layout": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, _I64, _I64,
                                                         ctypes.POINTER(_SZ)]),
    "moex_moe_prefill": (ctypes.c_int, [_QWP, _QWP, _P, ctypes.c_int, _P, _P, ctypes.c_int, _P, _P, _SZ, _P]),
    "moex_moe_decode_noalloc": (ctypes.c_int, [_QWP, _QWP, _P, ctypes.c_int, _P, _P, ctypes.c_int, _P, _P]),
    "moex_moe_prefill_q8_workspace_bytes": (_SZ, [ctypes.c_int, ctypes.c_int, ctypes.c_int, _I64, _I64]),
    "moex_moe_prefill_q8_workspace_layout": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, _I64, _I64,
                                                            ctypes.POINTER(_SZ)]),
    "moex_moe_prefill_q8": (ctypes.c_int, [_QWP, _QWP, _P, ctypes.c_int, _P, _P, ctypes.c_int, _P, _P, _SZ, _P]),
    "moex_moe_prefill_q8_debug": (ctypes.c_int, [_QWP, _QWP, _P, ctypes.c_int, _P, _P, ctypes.c_int, _P, _P, _SZ, _P,
                                                 _P]),
    "moex_dense_prefill_workspace_bytes": (_SZ, [ctypes.c_int, _I64, _I64]),
    "moex_dense_prefill": (ctypes.c_int, [_QWP, _P, ctypes.c_int, _P, _I64, _P, _SZ, _P]),
    "moex_moe_decode_residual": (ctypes.c_int, [_QWP, _QWP, _P, ctypes.c_int, _P, _P, ctypes.c_int, _P, _P, _P, _SZ,
                                                _P]),
    "moex_moe_prefill_residual": (ctypes.c_int, [_QWP, _QWP, _P, ctypes.c_int, _P, _P, ctypes.c_int, _P, _P, _P, _SZ,
                                                 _P]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m moe_expert_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != 0:
        raise MoexError(status, what)


def _torch():
    import torch
    return torch


_raw_stream = None


def _stream(stream=None) -> ctypes.c_void_p:
    """The handle of `stream`, else of torch's current stream on the current
    device (read without building a Stream object when torch offers that)."""
    global _raw_stream
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    torch = _torch()
    if _raw_stream is None:
        _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None) or False
    if _raw_stream:
        return ctypes.c_void_p(_raw_stream(torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def qs_row_bytes(fmt: str, K: int) -> int:
    return K if fmt == "q8_0" else K // 2


def sc_row_bytes(K: int) -> int:
    return ((K // QK) * 2 + 15) // 16 * 16


class PackedWeight:
    """A stack of n_mats rows x K weight matrices in device planes."""

    def __init__(self, fmt: str, n_mats: int, rows: int, K: int, device="cuda"):
        torch = _torch()
        if K % QK:
            raise ValueError("K must be a multiple of 32")
        self.fmt, self.n_mats, self.rows, self.K = fmt, n_mats, rows, K
        qb, sb = ctypes.c_size_t(), ctypes.c_size_t()
        _check(lib().moex_weight_plane_bytes(FMT[fmt], n_mats, rows, K, ctypes.byref(qb), ctypes.byref(sb)),
               "moex_weight_plane_bytes")
        self.qs = torch.empty(qb.value, dtype=torch.uint8, device=device)
        self.scales = torch.empty(sb.value, dtype=torch.uint8, device=device)
        self.struct = QWeight(FMT[fmt], n_mats, rows, K, self.qs.data_ptr(), self.scales.data_ptr())

    @property
    def nbytes(self) -> int:
        """Algorithmic weight bytes (34 or 18 per 32 values)."""
        return self.n_mats * self.rows * (self.K // QK) * BLOCK_BYTES[self.fmt]

    def pack(self, gguf_blocks, stream=None) -> "PackedWeight":
        """Fills the planes from GGUF blocks (numpy uint8 or a device tensor)."""
        torch = _torch()
        if isinstance(gguf_blocks, np.ndarray):
            src = torch.from_numpy(np.ascontiguousarray(gguf_blocks).reshape(-1)).to(self.qs.device)
        else:
            src = gguf_blocks.reshape(-1)
        expect = self.n_mats * self.rows * (self.K // QK) * BLOCK_BYTES[self.fmt]
        if src.numel() != expect:
            raise ValueError(f"expected {expect} block bytes, got {src.numel()}")
        _check(lib().moex_weight_pack(ctypes.byref(self.struct), _ptr(src), _stream(stream)), "moex_weight_pack")
        torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
        return self

    def pack_matrix(self, m: int, gguf_blocks, stream=None) -> "PackedWeight":
        """Fills matrix m of the stack from its GGUF blocks [rows, K/32, bytes]."""
        torch = _torch()
        src = torch.from_numpy(np.ascontiguousarray(gguf_blocks).reshape(-1)).to(self.qs.device)
        expect = self.rows * (self.K // QK) * BLOCK_BYTES[self.fmt]
        if src.numel() != expect:
            raise ValueError(f"expected {expect} block bytes, got {src.numel()}")
        qoff = m * self.rows * qs_row_bytes(self.fmt, self.K)
        soff = m * self.rows * sc_row_bytes(self.K)
        one = QWeight(FMT[self.fmt], 1, self.rows, self.K, self.qs.data_ptr() + qoff,
                      self.scales.data_ptr() + soff)
        _check(lib().moex_weight_pack(ctypes.byref(one), _ptr(src), _stream(stream)), "moex_weight_pack")
        torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
        return self

    def zero_(self) -> "PackedWeight":
        self.qs.zero_()
        self.scales.zero_()
        return self

    @classmethod
    def from_gguf(cls, fmt: str, blocks: np.ndarray, n_mats: Optional[int] = None, device="cuda"):
        """blocks: uint8 [rows, K/32, bytes] or [n_mats, rows, K/32, bytes]."""
        if blocks.ndim == 3:
            blocks = blocks[None]
        n, rows, nb = blocks.shape[0], blocks.shape[1], blocks.shape[2]
        w = cls(fmt, n if n_mats is None else n_mats, rows, nb * QK, device=device)
        return w.pack(blocks)


def quantize_q8_1(x, q=None, ds=None, stream=None):
    """q8_1 of FP32 activations x [ncols, K] (CUDA).  Returns (q int8 [ncols, K],
    ds float32 [ncols, K/32, 2])."""
    torch = _torch()
    ncols, K = x.shape
    if q is None:
        q = torch.empty((ncols, K), dtype=torch.int8, device=x.device)
    if ds is None:
        ds = torch.empty((ncols, K // QK, 2), dtype=torch.float32, device=x.device)
    _check(lib().moex_quantize_q8_1(_ptr(x), K, ncols, x.stride(0), _ptr(q), _ptr(ds), _stream(stream)),
           "moex_quantize_q8_1")
    return q, ds


def qgemv(W: PackedWeight, xq, xds, y=None, stream=None):
    """y [ncols, rows] = W . x for q8_1 activations (xq int8 [ncols, K], xds [ncols, K/32, 2])."""
    torch = _torch()
    ncols = xq.shape[0]
    if y is None:
        y = torch.empty((ncols, W.rows), dtype=torch.float32, device=xq.device)
    _check(lib().moex_qgemv(ctypes.byref(W.struct), _ptr(xq), _ptr(xds), ncols, _ptr(y), y.stride(0),
                            _stream(stream)), "moex_qgemv")
    return y


def qgemv_block_dots(W: PackedWeight, xq, stream=None):
    """Per-block integer dots int32 [ncols, rows, K/32] (diagnostic)."""
    torch = _torch()
    ncols = xq.shape[0]
    dots = torch.empty((ncols, W.rows, W.K // QK), dtype=torch.int32, device=xq.device)
    _check(lib().moex_qgemv_block_dots(ctypes.byref(W.struct), _ptr(xq), ncols, _ptr(dots), _stream(stream)),
           "moex_qgemv_block_dots")
    return dots


def route_topk(logits, k: int, ids=None, w=None, stream=None):
    """Top-k expert ids (int32 [T, k]) and softmax weights (float32 [T, k])."""
    torch = _torch()
    T, E = logits.shape
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if w is None:
        w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check(lib().moex_route_topk(_ptr(logits), T, E, k, _ptr(ids), _ptr(w), _stream(stream)), "moex_route_topk")
    return ids, w


def moe_decode_workspace_bytes(T: int, k: int, hidden: int, inter: int) -> int:
    return int(lib().moex_moe_decode_workspace_bytes(T, k, hidden, inter))


def moe_decode(gate_up: PackedWeight, down: PackedWeight, x, ids, w, out=None, ws=None, debug=False,
               stream=None, residual=None):
    """The grouped MoE decode layer.  x [T, hidden] FP32, ids/w [T, k].

    Returns out [T, hidden]; with debug=True returns (out, dict of the
    intermediates gu [T*k, 2I], h [T*k, I], hq [T*k, I], hds [T*k, I/32, 2]).
    With residual [T, hidden] FP32 (may be out) the layer writes
    residual + combine (moex_moe_decode_residual)."""
    torch = _torch()
    T, hidden = x.shape
    k = ids.shape[1]
    inter = down.K
    if out is None:
        out = torch.empty((T, hidden), dtype=torch.float32, device=x.device)
    nbytes = moe_decode_workspace_bytes(T, k, hidden, inter)
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    st = _stream(stream)
    if residual is not None:
        if debug:
            raise ValueError("residual and debug are separate entry points")
        _check(lib().moex_moe_decode_residual(ctypes.byref(gate_up.struct), ctypes.byref(down.struct), _ptr(x), T,
                                              _ptr(ids), _ptr(w), k, _ptr(residual), _ptr(out), _ptr(ws),
                                              ws.numel(), st), "moex_moe_decode_residual")
        return out
    if not debug:
        _check(lib().moex_moe_decode(ctypes.byref(gate_up.struct), ctypes.byref(down.struct), _ptr(x), T,
                                     _ptr(ids), _ptr(w), k, _ptr(out), _ptr(ws), ws.numel(), st),
               "moex_moe_decode")
        return out
    n = T * k
    dbg = dict(gu=torch.full((n, 2 * inter), float("nan"), device=x.device),
               h=torch.full((n, inter), float("nan"), device=x.device),
               hq=torch.zeros((n, inter), dtype=torch.int8, device=x.device),
               hds=torch.full((n, inter // QK, 2), float("nan"), device=x.device))
    _check(lib().moex_moe_decode_debug(ctypes.byref(gate_up.struct), ctypes.byref(down.struct), _ptr(x), T,
                                       _ptr(ids), _ptr(w), k, _ptr(out), _ptr(ws), ws.numel(),
                                       _ptr(dbg["gu"]), _ptr(dbg["h"]), _ptr(dbg["hq"]), _ptr(dbg["hds"]), st),
           "moex_moe_decode_debug")
    return out, dbg


def moe_prefill_workspace_bytes(T: int, k: int, E: int, hidden: int, inter: int) -> int:
    return int(lib().moex_moe_prefill_workspace_bytes(T, k, E, hidden, inter))


def moe_prefill_workspace_layout(T: int, k: int, E: int, hidden: int, inter: int):
    """Byte offsets of the prefill workspace parts (see include/moex.h)."""
    off = (ctypes.c_size_t * 9)()
    _check(lib().moex_moe_prefill_workspace_layout(T, k, E, hidden, inter, off), "moex_moe_prefill_workspace_layout")
    return [int(v) for v in off]


def moe_prefill(gate_up: PackedWeight, down: PackedWeight, x_bf16, ids, w, out=None, ws=None, stream=None,
                residual=None):
    """The grouped MoE prefill layer.  x_bf16: BF16 (or raw uint16/int16 bit
    patterns) [T, hidden]; ids / w [T, k].  Returns out [T, hidden] FP32;
    with residual [T, hidden] FP32 (may be out), residual + the layer
    (moex_moe_prefill_residual)."""
    torch = _torch()
    T, hidden = x_bf16.shape
    k = ids.shape[1]
    E, inter = gate_up.n_mats, down.K
    if out is None:
        out = torch.empty((T, hidden), dtype=torch.float32, device=x_bf16.device)
    if ws is None:
        ws = torch.empty(moe_prefill_workspace_bytes(T, k, E, hidden, inter), dtype=torch.uint8,
                         device=x_bf16.device)
    if residual is not None:
        _check(lib().moex_moe_prefill_residual(ctypes.byref(gate_up.struct), ctypes.byref(down.struct), _ptr(x_bf16),
                                               T, _ptr(ids), _ptr(w), k, _ptr(residual), _ptr(out), _ptr(ws),
                                               ws.numel(), _stream(stream)), "moex_moe_prefill_residual")
        return out
    _check(lib().moex_moe_prefill(ctypes.byref(gate_up.struct), ctypes.byref(down.struct), _ptr(x_bf16), T,
                                  _ptr(ids), _ptr(w), k, _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "moex_moe_prefill")
    return out


def moe_prefill_q8_workspace_bytes(T: int, k: int, E: int, hidden: int, inter: int) -> int:
    return int(lib().moex_moe_prefill_q8_workspace_bytes(T, k, E, hidden, inter))


def moe_prefill_q8_workspace_layout(T: int, k: int, E: int, hidden: int, inter: int):
    """Byte offsets of the integer-route workspace parts (see include/moex.h)."""
    off = (ctypes.c_size_t * 10)()
    _check(lib().moex_moe_prefill_q8_workspace_layout(T, k, E, hidden, inter, off),
           "moex_moe_prefill_q8_workspace_layout")
    return [int(v) for v in off]


def moe_prefill_q8(gate_up: PackedWeight, down: PackedWeight, x_bf16, ids, w, out=None, ws=None, h_dbg=None,
                   stream=None):
    """The grouped MoE prefill layer on its integer route (q8_1 rows of H, a
    block-integer down product).  Arguments as moe_prefill; with h_dbg (FP32
    [T*k, inter]) the layer also writes H in sorted-row order."""
    torch = _torch()
    T, hidden = x_bf16.shape
    k = ids.shape[1]
    E, inter = gate_up.n_mats, down.K
    if out is None:
        out = torch.empty((T, hidden), dtype=torch.float32, device=x_bf16.device)
    if ws is None:
        ws = torch.empty(moe_prefill_q8_workspace_bytes(T, k, E, hidden, inter), dtype=torch.uint8,
                         device=x_bf16.device)
    args = (ctypes.byref(gate_up.struct), ctypes.byref(down.struct), _ptr(x_bf16), T, _ptr(ids), _ptr(w), k,
            _ptr(out), _ptr(ws), ws.numel())
    if h_dbg is None:
        _check(lib().moex_moe_prefill_q8(*args, _stream(stream)), "moex_moe_prefill_q8")
    else:
        _check(lib().moex_moe_prefill_q8_debug(*args, _ptr(h_dbg), _stream(stream)), "moex_moe_prefill_q8_debug")
    return out


def dense_prefill(W: PackedWeight, x_bf16, y=None, ws=None, stream=None):
    """Dense prefill product on the tensor cores: y [T, rows] FP32 =
    fp16(W) . fp16(x)^T for an IQ4_NL matrix and BF16 rows x [T, K]."""
    torch = _torch()
    T = x_bf16.shape[0]
    if y is None:
        y = torch.empty((T, W.rows), dtype=torch.float32, device=x_bf16.device)
    if ws is None:
        ws = torch.empty(lib().moex_dense_prefill_workspace_bytes(T, W.rows, W.K), dtype=torch.uint8,
                         device=x_bf16.device)
    _check(lib().moex_dense_prefill(ctypes.byref(W.struct), _ptr(x_bf16), T, _ptr(y), y.stride(0), _ptr(ws), ws.numel(),
                                    _stream(stream)), "moex_dense_prefill")
    return y


def moe_decode_noalloc(gate_up: PackedWeight, down: PackedWeight, x, ids, w, out=None, stream=None):
    """moe_decode on the library's built-in workspace, for callers that
    cannot allocate device memory (see include/moex.h)."""
    torch = _torch()
    T, hidden = x.shape
    k = ids.shape[1]
    if out is None:
        out = torch.empty((T, hidden), dtype=torch.float32, device=x.device)
    _check(lib().moex_moe_decode_noalloc(ctypes.byref(gate_up.struct), ctypes.byref(down.struct), _ptr(x), T,
                                         _ptr(ids), _ptr(w), k, _ptr(out), _stream(stream)),
           "moex_moe_decode_noalloc")
    return out


def device_status(stream=None) -> int:
    """Synchronises the stream, returns and clears the device status bits."""
    flags = ctypes.c_uint32(0)
    lib().moex_device_status(_stream(stream), ctypes.byref(flags))
    return int(flags.value)
