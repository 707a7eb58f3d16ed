"""The IQ4_NL codebook tables compiled into the kernels, checked on the host.

The kernels decode 4-bit indices with `prmt` byte selection from constant
tables in csrc/common.cuh.  This test emulates `prmt` (default mode: selector
nibble bits 0-2 pick one of 8 bytes, bit 3 replicates that byte's sign bit)
and checks every decoding against the codebook fixture for every index: the
GEMV's rebuilt lookup, the split lookup of the one- and two-column dots, and
the prefill dequantiser's biased lookup (codebook value + 128).
"""

import os
import re

from helpers import ROOT


def _codebook():
    with open(os.path.join(ROOT, "tests", "golden", "iq4nl_codebook.txt")) as f:
        rows = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    return [int(v) for v in rows[0].split()]


def _constants(name="common.cuh", prefix="IQ4NL_"):
    with open(os.path.join(ROOT, "moe_expert_gb300", "csrc", name)) as f:
        src = f.read()
    return {m.group(1): int(m.group(2), 16)
            for m in re.finditer(r"constexpr uint32_t (%s\w+) = 0x([0-9A-Fa-f]+)u;" % prefix, src)}


def _prmt_byte(a, b, nib):
    tab = a | (b << 32)
    byte = (tab >> (8 * (nib & 7))) & 0xFF
    if nib & 8:
        byte = 0xFF if byte & 0x80 else 0x00
    return byte


def _s8(v):
    return v - 256 if v & 0x80 else v


def test_iq4nl_rebuilt_lookup_matches_codebook():
    cb, k = _codebook(), _constants()
    for idx in range(16):
        lo7 = _prmt_byte(k["IQ4NL_LO7_0"], k["IQ4NL_LO7_1"], idx)
        hi = _prmt_byte(k["IQ4NL_HI_0"], k["IQ4NL_HI_1"], idx ^ 8)
        sgn = (lo7 + 0x7F) & 0x80
        assert _s8(lo7 | hi | sgn) == cb[idx], idx


def test_iq4nl_split_lookup_sums_to_codebook():
    cb, k = _codebook(), _constants()
    for idx in range(16):
        lo = _s8(_prmt_byte(k["IQ4NL_LO_0"], k["IQ4NL_LO_1"], idx))
        hi = _s8(_prmt_byte(k["IQ4NL_HIP1_0"], k["IQ4NL_HIP1_1"], idx ^ 8))
        assert lo + hi == cb[idx], idx
        # each part alone stays an int8 that dp4a reads as signed
        assert -128 <= lo <= 127 and -128 <= hi <= 127


def test_iq4nl_biased_lookup_is_codebook_plus_128():
    cb, k = _codebook(), _constants("moe_prefill.cu", "IQ4B_")
    for idx in range(16):
        lo = _prmt_byte(k["IQ4B_LO_0"], k["IQ4B_LO_1"], idx)
        hi7 = _prmt_byte(k["IQ4B_HI_0"], k["IQ4B_HI_1"], idx ^ 8)
        b7 = (hi7 + 0x7F) & 0x80
        assert (lo | hi7 | b7) == cb[idx] + 128, idx
