"""Seeded synthetic inputs for the block-quantized GEMV and grouped-MoE workloads.

This module only draws random numbers and lays them out as GGUF-style byte
blocks.  It holds none of the arithmetic of the method: no dequantisation,
no activation quantiser, no dot products, no routing.  Both the CPU oracle
and the CUDA path read their inputs from here, and nothing else is shared
between them.

Recipe (every generator takes a numpy ``Generator(PCG64(seed))`` and draws
in the order written in its docstring):

* Q8_0 block (34 bytes): little-endian FP16 scale ``fp16(|N(0,1)| * 0.01)``
  followed by 32 int8 quants drawn uniformly from [-127, 127].
* IQ4_NL block (18 bytes): the same FP16 scale followed by 16 uniformly
  random bytes.  A uniform byte holds two independent uniform 4-bit
  codebook indices, so no nibble order is assumed here.
* Activations: FP32 N(0,1).
* Router logits: FP32 N(0,1).
* BF16 activations: N(0,1) drawn in FP32, rounded to BF16 (nearest even) and
  returned as raw uint16 bit patterns.

The pages measure on real GGUF models that are not available here; these
draws take the shapes and value distributions of the benchmark configs
instead.
"""
from __future__ import annotations

import numpy as np

QK = 32  # values per quantisation block


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _fp16_scales(g: np.random.Generator, shape) -> np.ndarray:
    """|N(0,1)| * 0.01 rounded to FP16, as uint16 bit patterns."""
    s = np.abs(g.standard_normal(size=shape, dtype=np.float64)) * 0.01
    return s.astype(np.float16).view(np.uint16)


def q8_0_blocks(g: np.random.Generator, rows: int, K: int) -> np.ndarray:
    """Q8_0 weight matrix as GGUF blocks, uint8 [rows, K/32, 34].

    Draw order: scales [rows, K/32], then quants [rows, K].
    """
    assert K % QK == 0
    nb = K // QK
    d = _fp16_scales(g, (rows, nb))
    q = g.integers(-127, 128, size=(rows, K), dtype=np.int16).astype(np.int8)
    out = np.empty((rows, nb, 34), dtype=np.uint8)
    out[:, :, 0:2] = d.astype('<u2').view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 2:34] = q.view(np.uint8).reshape(rows, nb, QK)
    return out


def iq4_nl_blocks(g: np.random.Generator, rows: int, K: int) -> np.ndarray:
    """IQ4_NL weight matrix as GGUF blocks, uint8 [rows, K/32, 18].

    Draw order: scales [rows, K/32], then index bytes [rows, K/32, 16].
    """
    assert K % QK == 0
    nb = K // QK
    d = _fp16_scales(g, (rows, nb))
    qs = g.integers(0, 256, size=(rows, nb, 16), dtype=np.int16).astype(np.uint8)
    out = np.empty((rows, nb, 18), dtype=np.uint8)
    out[:, :, 0:2] = d.astype('<u2').view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 2:18] = qs
    return out


def weight_blocks(fmt: str, g: np.random.Generator, rows: int, K: int) -> np.ndarray:
    if fmt == "q8_0":
        return q8_0_blocks(g, rows, K)
    if fmt == "iq4_nl":
        return iq4_nl_blocks(g, rows, K)
    raise ValueError(fmt)


def activations(g: np.random.Generator, ncols: int, K: int) -> np.ndarray:
    """FP32 N(0,1) activations, [ncols, K] (each column contiguous)."""
    return g.standard_normal(size=(ncols, K), dtype=np.float32)


def router_logits(g: np.random.Generator, T: int, E: int) -> np.ndarray:
    """FP32 N(0,1) router logits, [T, E]."""
    return g.standard_normal(size=(T, E), dtype=np.float32)


def bf16_activations(g: np.random.Generator, T: int, H: int) -> np.ndarray:
    """BF16 bit patterns (uint16 [T, H]) of N(0,1) FP32 draws, nearest-even."""
    x = g.standard_normal(size=(T, H), dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


# ---------------------------------------------------------------------------
# The benchmark workloads.  Sub-seeds are fixed so that any one tensor can be
# regenerated alone (for example one expert of a 128-expert layer).
# ---------------------------------------------------------------------------

SEED = 0


def dense_case(fmt: str, rows: int, K: int, ncols: int, seed: int = SEED):
    """(weight blocks, activations [ncols, K]) for a dense GEMV case."""
    g = rng(seed)
    w = weight_blocks(fmt, g, rows, K)
    x = activations(g, ncols, K)
    return w, x


def expert_blocks(kind: str, e: int, hidden: int, inter: int, fmt: str,
                  seed: int = SEED) -> np.ndarray:
    """Blocks of expert ``e``: kind "gate_up" -> [2*inter, hidden/32, *] with
    gate rows first then up rows; kind "down" -> [hidden, inter/32, *]."""
    base = {"gate_up": 1_000_000, "down": 2_000_000}[kind]
    g = rng(seed * 7919 + base + e)
    if kind == "gate_up":
        return weight_blocks(fmt, g, 2 * inter, hidden)
    return weight_blocks(fmt, g, hidden, inter)


def decode_tokens(T: int, hidden: int, seed: int = SEED) -> np.ndarray:
    return activations(rng(seed * 7919 + 3_000_000), T, hidden)


def decode_logits(T: int, E: int, sub_seed: int, seed: int = SEED) -> np.ndarray:
    return router_logits(rng(seed * 7919 + 4_000_000 + sub_seed), T, E)


def prefill_tokens(T: int, hidden: int, seed: int = SEED) -> np.ndarray:
    return bf16_activations(rng(seed * 7919 + 5_000_000), T, hidden)


def prefill_logits(T: int, E: int, seed: int = SEED) -> np.ndarray:
    return router_logits(rng(seed * 7919 + 6_000_000), T, E)
