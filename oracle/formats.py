"""Q8_0 and IQ4_NL weight blocks (oracle; test infrastructure only).

Both formats hold 32 values per block with one FP16 scale.  The pages name the
formats but never print a byte layout; the reading taken here is the GGUF one
that the pages refer to ("GGUF-block -> planes repack", #1424 What changed):

* Q8_0, 34 bytes: FP16 scale ``d`` (little endian), then 32 int8 quants.
  Value i = fp32(d) * q[i].
* IQ4_NL, 18 bytes: FP16 scale ``d``, then 16 bytes of 4-bit codebook
  indices.  Byte j holds element j in its low nibble and element j+16 in its
  high nibble.  Value i = fp32(d) * kvalues[idx[i]].

The IQ4_NL codebook is the 16-entry int8 table ``kvalues_iq4nl`` named in #2356
(Summary: "a byte -> two kvalues_iq4nl table"); its entries are the ones the
IQ4_NL benchmark workload lists.
"""
from __future__ import annotations

import numpy as np

QK = 32

KVALUES_IQ4NL = np.array(
    [-127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113],
    dtype=np.int64)

BLOCK_BYTES = {"q8_0": 34, "iq4_nl": 18}


def fp16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """FP16 bit patterns (uint16) to float64; every FP16 value is exact."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def block_scales(blocks: np.ndarray) -> np.ndarray:
    """FP16 scale of each block as float64, shape blocks.shape[:-1]."""
    b = np.ascontiguousarray(blocks[..., 0:2])
    bits = b[..., 0].astype(np.uint16) | (b[..., 1].astype(np.uint16) << 8)
    return fp16_bits_to_f64(bits)


def q8_0_quants(blocks: np.ndarray) -> np.ndarray:
    """int8 quants of Q8_0 blocks as int64, shape [..., 32]."""
    assert blocks.shape[-1] == 34
    return np.ascontiguousarray(blocks[..., 2:34]).view(np.int8).astype(np.int64)


def iq4_nl_indices(blocks: np.ndarray) -> np.ndarray:
    """Codebook indices of IQ4_NL blocks, shape [..., 32] (element j is the low
    nibble of byte j, element j+16 its high nibble)."""
    assert blocks.shape[-1] == 18
    qs = blocks[..., 2:18].astype(np.int64)
    idx = np.empty(qs.shape[:-1] + (QK,), dtype=np.int64)
    idx[..., 0:16] = qs & 0x0F
    idx[..., 16:32] = qs >> 4
    return idx


def iq4_nl_quants(blocks: np.ndarray) -> np.ndarray:
    """Integer codebook values kvalues[idx] of IQ4_NL blocks, [..., 32]."""
    return KVALUES_IQ4NL[iq4_nl_indices(blocks)]


def block_quants(fmt: str, blocks: np.ndarray) -> np.ndarray:
    if fmt == "q8_0":
        return q8_0_quants(blocks)
    if fmt == "iq4_nl":
        return iq4_nl_quants(blocks)
    raise ValueError(fmt)


def decode(fmt: str, blocks: np.ndarray):
    """(d float64 [rows, nb], q int64 [rows, K]) of a [rows, nb, bytes] matrix."""
    rows, nb = blocks.shape[0], blocks.shape[1]
    d = block_scales(blocks)
    q = block_quants(fmt, blocks).reshape(rows, nb * QK)
    return d, q


def dequantize(fmt: str, blocks: np.ndarray) -> np.ndarray:
    """Dequantised weights fp32(d) * q as float64 [rows, K] (exact)."""
    d, q = decode(fmt, blocks)
    rows, nb = d.shape
    return (np.repeat(d, QK, axis=1) * q).reshape(rows, nb * QK)
