"""Pins of the CPU oracle against things other than itself.

Each test checks an oracle function against a closed form, brute force on tiny
inputs (pure-Python loops and exact rationals), a hand-derived fixture under
tests/golden/, or an invariant of the mathematics.  A plausible mistake in the
oracle (dropped term, wrong sign or index, transposed operand, wrong nibble
order, round-half-even instead of half-away) fails at least one of them; the
mutation tests at the end plant such mistakes in the oracle and check that.
"""
import itertools
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from oracle import formats, gemv, moe, prefill, q8_1

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- fixtures

def read_codebook():
    with open(os.path.join(GOLDEN, "iq4nl_codebook.txt")) as f:
        rows = [l for l in f if l.strip() and not l.startswith("#")]
    return [int(v) for v in rows[0].split()]


def read_q8_1_cases():
    cases, cur = [], {}
    with open(os.path.join(GOLDEN, "q8_1_hand.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            cur[key.strip()] = val.split()
            if key.strip() == "s":
                cases.append(cur)
                cur = {}
    return cases


def read_dequant_cases():
    cases, cur = [], {}
    with open(os.path.join(GOLDEN, "dequant_hand.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            cur[key.strip()] = val.split()
            if key.strip() == "values":
                cases.append(cur)
                cur = {}
    return cases


def expand(vals, n=32):
    out = []
    for v in vals:
        if v == "...":
            out += [out[-1]] * (n - len(out))
        else:
            out.append(float(v))
    out += [0.0] * (n - len(out))
    return out


# ---------------------------------------------------------------- formats

def test_codebook_matches_fixture():
    assert list(formats.KVALUES_IQ4NL) == read_codebook()
    # monotone, 8 negative then 8 positive entries, all within int8
    kv = read_codebook()
    assert kv == sorted(kv) and all(-128 <= v <= 127 for v in kv)


@pytest.mark.parametrize("case", read_dequant_cases(), ids=lambda c: c["fmt"][0] + ":" + "".join(c["hex"])[:12])
def test_dequant_hand_fixture(case):
    fmt = case["fmt"][0]
    raw = bytes.fromhex("".join(case["hex"]))
    blocks = np.frombuffer(raw, dtype=np.uint8).reshape(1, 1, -1)
    got = formats.dequantize(fmt, blocks)[0]
    want = expand(case["values"])
    assert got.tolist() == want


def _fp16_exact(bits):
    return Fraction(struct.unpack("<e", struct.pack("<H", bits))[0])


@pytest.mark.parametrize("fmt", ["q8_0", "iq4_nl"])
def test_dequant_brute_force(fmt):
    g = synth.rng(11)
    blocks = synth.weight_blocks(fmt, g, 3, 64)
    got = formats.dequantize(fmt, blocks)
    kv = read_codebook()
    for r in range(3):
        for b in range(2):
            blk = bytes(blocks[r, b])
            d = _fp16_exact(blk[0] | (blk[1] << 8))
            for i in range(32):
                if fmt == "q8_0":
                    q = struct.unpack("b", blk[2 + i:3 + i])[0]
                else:
                    byte = blk[2 + (i % 16)]
                    q = kv[(byte & 15) if i < 16 else (byte >> 4)]
                assert Fraction(got[r, 32 * b + i]) == d * q


def test_dequant_one_hot_and_zero_block():
    # one index j set, other elements weighted zero -> y = d * kvalues[j]
    kv = read_codebook()
    for j in range(16):
        blk = np.zeros((1, 1, 18), dtype=np.uint8)
        blk[0, 0, 0:2] = np.frombuffer(struct.pack("<e", 0.25), dtype=np.uint8)
        blk[0, 0, 2] = j          # element 0 has index j
        w = formats.dequantize("iq4_nl", blk)[0]
        sel = np.zeros(32)
        sel[0] = 1.0
        assert float(w @ sel) == 0.25 * kv[j]
    zero = np.zeros((1, 1, 34), dtype=np.uint8)
    assert np.all(formats.dequantize("q8_0", zero) == 0)


# ---------------------------------------------------------------- q8_1

@pytest.mark.parametrize("case", read_q8_1_cases(), ids=lambda c: " ".join(c["x"][:2]))
def test_q8_1_hand_fixture(case):
    x = np.array(expand(case["x"]), dtype=np.float32)[None, :]
    q, d, s = q8_1.quantize_q8_1(x)
    assert q[0].tolist() == [int(v) for v in case["q"]]
    assert float(d[0, 0]) == float(case["d"][0])
    assert float(s[0, 0]) == float(case["s"][0])


def _roundf(fr: Fraction) -> int:
    """C roundf on an exact rational: half away from zero."""
    a = abs(fr)
    n = math.floor(a + Fraction(1, 2))
    return n if fr >= 0 else -n


def _f32(v) -> float:
    return float(np.float32(v))


def test_q8_1_brute_force_exact_rationals():
    """Every step redone with exact rationals and explicit FP32 rounding."""
    g = synth.rng(5)
    x = (g.standard_normal((4, 96)) * g.choice([1e-3, 1, 1e3], (4, 1))).astype(np.float32)
    x[1, 32:64] = 0.0
    q, d, s = q8_1.quantize_q8_1(x)
    for c in range(4):
        for b in range(3):
            blk = x[c, 32 * b:32 * b + 32]
            amax = max(abs(float(v)) for v in blk)
            if amax == 0:
                assert d[c, b] == 0 and s[c, b] == 0 and not q[c, 32 * b:32 * b + 32].any()
                continue
            dd = _f32(Fraction(amax) / 127)                   # one FP32 rounding
            assert float(d[c, b]) == dd
            qs = []
            for v in blk:
                ratio = _f32(Fraction(float(v)) / Fraction(dd))  # FP32 division
                qs.append(_roundf(Fraction(ratio)))
            assert q[c, 32 * b:32 * b + 32].tolist() == qs
            assert float(s[c, b]) == _f32(Fraction(dd) * sum(qs))


def test_q8_1_invariants():
    g = synth.rng(6)
    x = g.standard_normal((8, 2048)).astype(np.float32) * 3
    x[0, :32] = 0.0
    x[1, 5] = 3e4                      # outlier
    q, d, s = q8_1.quantize_q8_1(x)
    xb = x.reshape(8, -1, 32).astype(np.float64)
    qb = q.reshape(8, -1, 32).astype(np.float64)
    db = d.astype(np.float64)[:, :, None]
    # round trip within half a step (plus one FP32 ulp of x/d)
    assert np.all(np.abs(xb - db * qb) <= db * (0.5 + 1e-6) + 1e-30)
    # the amax element maps to +-127
    amax_idx = np.argmax(np.abs(xb), axis=2)
    qa = np.take_along_axis(qb, amax_idx[:, :, None], axis=2)[:, :, 0]
    nz = d > 0
    assert np.all(np.abs(qa[nz]) == 127)
    assert d[0, 0] == 0 and s[0, 0] == 0
    # s is d * sum(q)
    assert np.array_equal(s, (d * qb.sum(axis=2).astype(np.float32)).astype(np.float32))


def test_round_half_away_not_even():
    r = np.array([0.5, 1.5, 2.5, -0.5, -2.5, 0.49999997, 126.5], dtype=np.float32)
    assert q8_1.round_half_away(r).tolist() == [1, 2, 3, -1, -3, 0, 127]


# ---------------------------------------------------------------- GEMV

@pytest.mark.parametrize("fmt", ["q8_0", "iq4_nl"])
def test_gemv_brute_force_tiny(fmt):
    """y from the block formula == sum over K of dequant(w) * dequant(x)."""
    g = synth.rng(7)
    R, K, C = 5, 96, 3
    blocks = synth.weight_blocks(fmt, g, R, K)
    x = synth.activations(g, C, K)
    xq, xd, _ = q8_1.quantize_q8_1(x)
    y, A = gemv.gemv(fmt, blocks, xq, xd)
    W = formats.dequantize(fmt, blocks)
    for c in range(C):
        for r in range(R):
            exact = sum(Fraction(W[r, i]) * Fraction(float(xd[c, i // 32])) * int(xq[c, i])
                        for i in range(K))
            absum = sum(abs(Fraction(W[r, i]) * Fraction(float(xd[c, i // 32])) * int(xq[c, i]))
                        for i in range(K))
            assert abs(y[c, r] - float(exact)) <= 1e-12 * float(absum)
            assert abs(A[c, r] - float(absum)) <= 1e-12 * float(absum)


def read_bound_case():
    vals = {}
    with open(os.path.join(GOLDEN, "gemv_bound_hand.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, val = line.split(":", 1)
                vals[key.strip()] = [float(v) for v in val.split()]
    return vals


def test_gemv_error_scale_and_tolerance_hand_fixture():
    """y, A and the pass bound of a two-block row worked out by hand
    (tests/golden/gemv_bound_hand.txt)."""
    c = read_bound_case()
    wq = np.zeros((1, 64), dtype=np.int64)
    xq = np.zeros((1, 64), dtype=np.int64)
    for b in (0, 1):
        for i, v in enumerate(c[f"qw{b}"]):
            wq[0, 32 * b + i] = int(v)
        for i, v in enumerate(c[f"qx{b}"]):
            xq[0, 32 * b + i] = int(v)
    dw = np.array([c["dw"]], dtype=np.float32)
    dx = np.array([c["dx"]], dtype=np.float32)
    y, A = gemv.gemv_planes(dw, wq, dx, xq)
    assert y[0, 0] == c["y"][0]
    assert A[0, 0] == c["A"][0]
    assert abs(gemv.tolerance(A)[0, 0] - c["bound"][0]) < 1e-15
    # the bound is exactly 1e-5 * A + 1e-6 element by element, monotone in A
    a = np.array([0.0, 1.0, 1e5])
    assert np.array_equal(gemv.tolerance(a), np.array([1e-6, 1e-5 + 1e-6, 1.0 + 1e-6]))


def test_block_dots_brute_force_and_range():
    g = synth.rng(8)
    wq = g.integers(-127, 128, (3, 64))
    xq = g.integers(-127, 128, (2, 64))
    I = gemv.block_dots(wq, xq)
    for c, r, b in itertools.product(range(2), range(3), range(2)):
        assert I[c, r, b] == sum(int(wq[r, 32 * b + i]) * int(xq[c, 32 * b + i]) for i in range(32))
    # extreme: all -127 x -127 -> 32 * 16129 = 516128
    big = gemv.block_dots(np.full((1, 32), -127), np.full((1, 32), -127))
    assert big[0, 0, 0] == 516128


@pytest.mark.parametrize("fmt", ["q8_0", "iq4_nl"])
def test_gemv_one_hot_column_reproduces_weights(fmt):
    """x = e_k: amax = 1, d = fp32(1/127), q = 127 at k -> y = w[:, k] * d * 127."""
    g = synth.rng(9)
    R, K = 6, 64
    blocks = synth.weight_blocks(fmt, g, R, K)
    W = formats.dequantize(fmt, blocks)
    for k in [0, 17, 31, 32, 63]:
        x = np.zeros((1, K), dtype=np.float32)
        x[0, k] = 1.0
        xq, xd, _ = q8_1.quantize_q8_1(x)
        assert xq[0, k] == 127 and float(xd[0, k // 32]) == float(np.float32(1) / np.float32(127))
        y, _ = gemv.gemv(fmt, blocks, xq, xd)
        scale = float(np.float32(1) / np.float32(127)) * 127
        assert np.allclose(y[0], W[:, k] * scale, rtol=1e-15, atol=0)


def test_gemv_columns_independent():
    g = synth.rng(10)
    blocks = synth.q8_0_blocks(g, 7, 128)
    x = synth.activations(g, 11, 128)
    xq, xd, _ = q8_1.quantize_q8_1(x)
    y, _ = gemv.gemv("q8_0", blocks, xq, xd)
    for c in range(11):
        y1, _ = gemv.gemv("q8_0", blocks, xq[c:c + 1], xd[c:c + 1])
        assert np.array_equal(y1[0], y[c])


def test_gemv_zero_block_gives_zero():
    blocks = np.zeros((2, 2, 18), dtype=np.uint8)
    x = synth.activations(synth.rng(3), 1, 64)
    xq, xd, _ = q8_1.quantize_q8_1(x)
    y, A = gemv.gemv("iq4_nl", blocks, xq, xd)
    assert np.all(y == 0) and np.all(A == 0)


# ---------------------------------------------------------------- routing

def test_route_topk_brute_force():
    g = synth.rng(12)
    logits = synth.router_logits(g, 6, 16)
    logits[2, 3] = logits[2, 9] = 5.0        # tie -> lower id first
    ids, w = moe.route_topk(logits, 4)
    for t in range(6):
        pairs = sorted(((-float(logits[t, e]), e) for e in range(16)))[:4]
        assert ids[t].tolist() == [e for _, e in pairs]
        ls = [float(logits[t, e]) for e in ids[t]]
        den = sum(math.exp(v - max(ls)) for v in ls)
        assert np.allclose(w[t], [math.exp(v - max(ls)) / den for v in ls], rtol=1e-14)
        assert abs(w[t].sum() - 1) < 1e-14 and np.all(np.diff(w[t]) <= 0)
    assert ids[2, 0] == 3 and ids[2, 1] == 9


# ---------------------------------------------------------------- SwiGLU / MoE

def test_silu_closed_forms():
    assert moe.silu(np.array([0.0]))[0] == 0.0
    v = np.linspace(-20, 20, 81)
    assert np.allclose(moe.silu(v) - moe.silu(-v), v, atol=1e-12)   # silu(x)-silu(-x) = x
    assert abs(moe.silu(np.array([40.0]))[0] - 40.0) < 1e-12
    assert abs(moe.silu(np.array([-40.0]))[0]) < 1e-15
    assert abs(moe.silu(np.array([1.0]))[0] - 1 / (1 + math.exp(-1))) < 1e-15


def test_swiglu_split_layout():
    gu = np.array([[1.0, 2.0, 3.0, 4.0]])          # inter 2: g = [1,2], u = [3,4]
    h = moe.swiglu(gu, 2)
    assert np.allclose(h, [[moe.silu(np.array([1.0]))[0] * 3, moe.silu(np.array([2.0]))[0] * 4]])


def _tiny_experts(E, hidden, inter, seed=20):
    gu = [synth.expert_blocks("gate_up", e, hidden, inter, "q8_0", seed=seed) for e in range(E)]
    dn = [synth.expert_blocks("down", e, hidden, inter, "iq4_nl", seed=seed) for e in range(E)]
    return gu, dn


def test_moe_single_expert_chain():
    """All k entries of a token on one expert with w = 1/k equals the single
    expert chain gemv -> swiglu -> q8_1 -> gemv written out step by step."""
    hidden, inter, k = 64, 64, 8
    gu, dn = _tiny_experts(4, hidden, inter)
    x = synth.activations(synth.rng(21), 1, hidden)
    ids = np.full((1, k), 2)
    w = np.full((1, k), 1.0 / k)
    r = moe.moe_decode(gu, dn, x, ids, w)
    xq, xd, _ = q8_1.quantize_q8_1(x)
    y, _ = gemv.gemv("q8_0", gu[2], xq, xd)
    g_, u_ = y[0, :inter], y[0, inter:]
    H = (g_ / (1 + np.exp(-g_)) * u_).astype(np.float32)
    hq, hd, _ = q8_1.quantize_q8_1(H[None, :])
    o, _ = gemv.gemv("iq4_nl", dn[2], hq, hd)
    assert np.allclose(r["out"][0], o[0], rtol=1e-13, atol=1e-13)


def test_moe_slot_permutation_invariant():
    hidden, inter, k = 64, 32, 4
    gu, dn = _tiny_experts(6, hidden, inter)
    x = synth.activations(synth.rng(22), 2, hidden)
    ids, w = moe.route_topk(synth.router_logits(synth.rng(23), 2, 6), k)
    r1 = moe.moe_decode(gu, dn, x, ids, w)
    perm = [2, 0, 3, 1]
    r2 = moe.moe_decode(gu, dn, x, ids[:, perm], w[:, perm])
    assert np.allclose(r1["out"], r2["out"], rtol=1e-12, atol=1e-12)


def test_moe_zero_gate_gives_zero_hq_block():
    # x = 0 -> xq = 0 -> gu = 0 -> H = 0 -> Hq zero blocks -> out = 0
    hidden, inter = 64, 32
    gu, dn = _tiny_experts(2, hidden, inter)
    r = moe.moe_decode(gu, dn, np.zeros((1, hidden), np.float32), np.array([[0, 1]]),
                       np.array([[0.5, 0.5]]))
    assert not r["Hq"].any() and not r["Hd"].any() and np.all(r["out"] == 0)


def test_entry_groups_brute_force():
    ids = np.array([[5, 1, 7], [1, 5, 2]])
    assert moe.entry_groups(ids) == [(1, [1, 3]), (2, [5]), (5, [0, 4]), (7, [2])]


# ---------------------------------------------------------------- prefill

def test_fp16_rounding_matches_struct():
    g = synth.rng(30)
    v = g.standard_normal(5000) * g.choice([1e-7, 1e-4, 1, 1e3, 1.5e4], 5000)
    v = v[np.abs(v) < 65504]
    got = prefill.fp16_rn(v).view(np.uint16)
    want = np.array([struct.unpack("<H", struct.pack("<e", float(t)))[0] for t in v], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_dequant_fp16_all_codes_and_scales():
    """fp16_rn(d * kval) for all 16 codes and zero / subnormal / normal / huge
    scales, against exact rationals rounded by Python's own FP16 packer."""
    kv = read_codebook()
    scale_bits = [0x0000, 0x0001, 0x03FF, 0x0400, 0x2E66, 0x3C00, 0x5640, 0x7BFF]
    blocks = np.zeros((len(scale_bits), 1, 18), dtype=np.uint8)
    for i, sb in enumerate(scale_bits):
        blocks[i, 0, 0] = sb & 0xFF
        blocks[i, 0, 1] = sb >> 8
        blocks[i, 0, 2:18] = [(15 - j) << 4 | j for j in range(16)]
    got = prefill.dequant_fp16("iq4_nl", blocks)
    for i, sb in enumerate(scale_bits):
        d = _fp16_exact(sb)
        for j in range(16):
            exact = float(d * kv[j])
            try:
                want = struct.unpack("<e", struct.pack("<e", exact))[0]
            except OverflowError:
                want = math.copysign(math.inf, exact)
            assert float(got[i, j]) == want or (math.isinf(want) and math.isinf(float(got[i, j])))


def test_sort_entries_brute_force():
    g = synth.rng(31)
    ids = g.integers(0, 9, (50, 3))
    order, offs = prefill.sort_entries(ids, 9)
    flat = ids.reshape(-1).tolist()
    want = sorted(range(len(flat)), key=lambda j: (flat[j], j))
    assert order.tolist() == want
    assert offs.tolist() == [0] + list(itertools.accumulate(flat.count(e) for e in range(9)))


def test_prefill_one_hot_rows_reproduce_fp16_weights():
    """With x = e_i and w = 1 on one slot, g/u equal column i of the FP16 weights."""
    hidden, inter = 64, 32
    gu = [synth.expert_blocks("gate_up", e, hidden, inter, "iq4_nl", seed=40) for e in range(2)]
    dn = [synth.expert_blocks("down", e, hidden, inter, "iq4_nl", seed=40) for e in range(2)]
    x = np.zeros((1, hidden), dtype=np.float32)
    x[0, 13] = 1.0
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    r = prefill.moe_prefill(gu, dn, xb, np.array([[1]]), np.array([[1.0]]))
    Wh = prefill.dequant_fp16("iq4_nl", gu[1]).astype(np.float64)
    assert np.array_equal(r["g"][0, 0], Wh[:inter, 13]) and np.array_equal(r["u"][0, 0], Wh[inter:, 13])


def test_prefill_brute_force_tiny():
    hidden, inter, k = 32, 32, 2
    gu = [synth.expert_blocks("gate_up", e, hidden, inter, "iq4_nl", seed=41) for e in range(3)]
    dn = [synth.expert_blocks("down", e, hidden, inter, "iq4_nl", seed=41) for e in range(3)]
    xb = synth.bf16_activations(synth.rng(42), 2, hidden)
    ids = np.array([[0, 2], [2, 1]])
    w = np.array([[0.75, 0.25], [0.5, 0.5]])
    r = prefill.moe_prefill(gu, dn, xb, ids, w)
    kv = read_codebook()

    def fp16w(blocks, row, col):
        blk = bytes(blocks[row, col // 32])
        d = _fp16_exact(blk[0] | (blk[1] << 8))
        byte = blk[2 + (col % 32) % 16]
        q = kv[(byte & 15) if (col % 32) < 16 else (byte >> 4)]
        return struct.unpack("<e", struct.pack("<e", float(d * q)))[0]

    for t in range(2):
        xs = [struct.unpack("<e", struct.pack("<e", struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]))[0]
              for b in xb[t]]
        out = [0.0] * hidden
        for s in range(k):
            e = ids[t, s]
            gg = [sum(fp16w(gu[e], i, c) * xs[c] for c in range(hidden)) for i in range(inter)]
            uu = [sum(fp16w(gu[e], inter + i, c) * xs[c] for c in range(hidden)) for i in range(inter)]
            h = [struct.unpack("<e", struct.pack("<e", a / (1 + math.exp(-a)) * b))[0] for a, b in zip(gg, uu)]
            for o in range(hidden):
                out[o] += w[t, s] * sum(fp16w(dn[e], o, i) * h[i] for i in range(inter))
        assert np.allclose(r["out"][t], out, rtol=1e-12, atol=1e-12)


def _iq4_row_ints(blocks, row, kv):
    """Codebook integers and exact scales of one IQ4_NL row, decoded by hand
    from the block bytes (low nibble of byte j: element j, high: j + 16)."""
    ints, scales = [], []
    for blk in blocks[row]:
        b = bytes(blk)
        scales.append(_fp16_exact(b[0] | (b[1] << 8)))
        lo = [kv[v & 15] for v in b[2:18]]
        hi = [kv[v >> 4] for v in b[2:18]]
        ints.append(lo + hi)
    return ints, scales


def test_prefill_q8_brute_force_tiny():
    """The integer route redone by hand: g, u from the FP16 weights and
    tokens in plain floats, H rounded to FP32 by struct, q8_1 with exact
    rationals, the down product as integer block dots with exact scales."""
    hidden, inter, k = 64, 64, 2
    gu = [synth.expert_blocks("gate_up", e, hidden, inter, "iq4_nl", seed=43) for e in range(3)]
    dn = [synth.expert_blocks("down", e, hidden, inter, "iq4_nl", seed=43) for e in range(3)]
    xb = synth.bf16_activations(synth.rng(44), 2, hidden)
    ids = np.array([[1, 2], [0, 1]])
    w = np.array([[0.625, 0.375], [0.5, 0.5]])
    kv = read_codebook()

    def fp16w(blocks, row, col):
        blk = bytes(blocks[row, col // 32])
        d = _fp16_exact(blk[0] | (blk[1] << 8))
        byte = blk[2 + (col % 32) % 16]
        q = kv[(byte & 15) if (col % 32) < 16 else (byte >> 4)]
        return struct.unpack("<e", struct.pack("<e", float(d * q)))[0]

    H32, H64 = {}, {}
    for t in range(2):
        xs = [struct.unpack("<e", struct.pack("<e", struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]))[0]
              for b in xb[t]]
        for s in range(k):
            e = ids[t, s]
            gg = [sum(fp16w(gu[e], i, c) * xs[c] for c in range(hidden)) for i in range(inter)]
            uu = [sum(fp16w(gu[e], inter + i, c) * xs[c] for c in range(hidden)) for i in range(inter)]
            H64[t, s] = [a / (1 + math.exp(-a)) * b for a, b in zip(gg, uu)]
            H32[t, s] = [_f32(Fraction(v)) for v in H64[t, s]]
    own = prefill.moe_prefill_q8(gu, dn, xb, ids, w)
    for (t, s), h in H64.items():
        assert np.allclose(own["H"][t, s], h, rtol=1e-9, atol=1e-12)
    r = prefill.moe_prefill_q8(gu, dn, xb, ids, w, h_override=lambda t, s: np.array(H32[t, s], np.float32))
    for t in range(2):
        out = [Fraction(0)] * hidden
        for s in range(k):
            h = H32[t, s]
            qs, ds = [], []
            for b in range(inter // 32):
                blk = h[32 * b:32 * b + 32]
                amax = max(abs(v) for v in blk)
                dd = _f32(Fraction(amax) / 127) if amax else 0.0
                q = [_roundf(Fraction(_f32(Fraction(v) / Fraction(dd)))) if amax else 0 for v in blk]
                qs += q
                ds.append(dd)
            assert r["Hq"][t, s].tolist() == qs and r["Hd"][t, s].tolist() == ds
            wints, wsc = _iq4_row_ints(dn[ids[t, s]], 0, kv)  # shape check on row 0
            assert len(wints) == inter // 32
            for o in range(hidden):
                wints, wsc = _iq4_row_ints(dn[ids[t, s]], o, kv)
                acc = Fraction(0)
                for b in range(inter // 32):
                    I = sum(wq * xq for wq, xq in zip(wints[b], qs[32 * b:32 * b + 32]))
                    acc += Fraction(_f32(wsc[b])) * Fraction(ds[b]) * I
                out[o] += Fraction(w[t, s]) * acc
        assert np.allclose(r["out"][t], [float(v) for v in out], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- mutations

def test_planted_nibble_swap_is_caught(monkeypatch):
    """Swapping the IQ4_NL nibble order in the oracle must fail a pin."""
    def swapped(blocks):
        qs = blocks[..., 2:18].astype(np.int64)
        idx = np.empty(qs.shape[:-1] + (32,), dtype=np.int64)
        idx[..., 0:16] = qs >> 4
        idx[..., 16:32] = qs & 0x0F
        return idx
    monkeypatch.setattr(formats, "iq4_nl_indices", swapped)
    case = [c for c in read_dequant_cases() if c["fmt"][0] == "iq4_nl"][0]
    with pytest.raises(AssertionError):
        test_dequant_hand_fixture(case)


def test_planted_round_half_even_is_caught(monkeypatch):
    monkeypatch.setattr(q8_1, "round_half_away", lambda r: np.round(r.astype(np.float64)))
    with pytest.raises(AssertionError):
        test_q8_1_hand_fixture(read_q8_1_cases()[0])


def test_planted_dropped_scale_in_prefill_q8_is_caught(monkeypatch):
    orig = gemv.gemv_planes
    monkeypatch.setattr(gemv, "gemv_planes", lambda dw, wq, dx, xq: orig(dw, wq, np.ones_like(dx), xq))
    with pytest.raises(AssertionError):
        test_prefill_q8_brute_force_tiny()


def test_planted_dropped_scale_is_caught(monkeypatch):
    orig = gemv.gemv_planes

    def no_dx(dw, wq, dx, xq):
        return orig(dw, wq, np.ones_like(dx), xq)
    monkeypatch.setattr(gemv, "gemv_planes", no_dx)
    with pytest.raises(AssertionError):
        test_gemv_brute_force_tiny("q8_0")


def test_planted_transposed_gate_up_is_caught(monkeypatch):
    monkeypatch.setattr(moe, "swiglu", lambda gu, inter: moe.silu(gu[..., inter:]) * gu[..., :inter])
    with pytest.raises(AssertionError):
        test_swiglu_split_layout()


def test_dense_prefill_one_hot_rows_and_brute_force():
    """The dense prefill oracle: a one-hot token row (x = 1 at input i)
    returns column i of the FP16 weights exactly; a tiny case equals a plain
    triple loop over the FP16 roundings of each weight and input."""
    g = synth.rng(41)
    R, K = 4, 64
    blocks = synth.iq4_nl_blocks(g, R, K)
    one = np.uint16(0x3F80)                     # BF16 1.0
    x = np.zeros((3, K), dtype=np.uint16)
    for t, i in enumerate([0, 17, 63]):
        x[t, i] = one
    y, _ = prefill.dense_prefill(blocks, x)
    wh = prefill.dequant_fp16("iq4_nl", blocks).astype(np.float64)
    for t, i in enumerate([0, 17, 63]):
        assert np.array_equal(y[t], wh[:, i])
    xb = synth.bf16_activations(g, 3, K)
    y, A = prefill.dense_prefill(blocks, xb)
    d, q = formats.decode("iq4_nl", blocks)
    for t in range(3):
        for r in range(R):
            acc = 0.0
            for i in range(K):
                wv = float(np.float16(np.float32(d[r, i // 32]) * np.float32(q[r, i])))
                xv = float(np.float16(np.uint32(int(xb[t, i]) << 16).view(np.float32)))
                acc += wv * xv
            assert abs(acc - y[t, r]) <= 1e-12 * max(1.0, A[t, r])
    y2, _ = prefill.dense_prefill(blocks, xb, rows=[2, 0])
    assert np.array_equal(y2, y[:, [2, 0]])


def test_dequant_fp16_q8_0_codes_and_scales():
    """fp16_rn(d * q) for Q8_0: every int8 code of a block set (-128..127
    over 8 blocks) at zero / subnormal / normal / huge scales, against exact
    rationals rounded by Python's own FP16 packer."""
    scale_bits = [0x0000, 0x0001, 0x03FF, 0x2E66, 0x3C00, 0x5640, 0x7BFF]
    codes = np.arange(-128, 128, dtype=np.int16).astype(np.int8).reshape(8, 32)
    for sb in scale_bits:
        blocks = np.zeros((1, 8, 34), dtype=np.uint8)
        blocks[0, :, 0] = sb & 0xFF
        blocks[0, :, 1] = sb >> 8
        blocks[0, :, 2:34] = codes.view(np.uint8)
        got = prefill.dequant_fp16("q8_0", blocks).reshape(-1)
        d = _fp16_exact(sb)
        for i, q in enumerate(codes.reshape(-1)):
            exact = float(d * int(q))
            try:
                want = struct.unpack("<e", struct.pack("<e", exact))[0]
            except OverflowError:
                want = math.copysign(math.inf, exact)
            assert float(got[i]) == want or (math.isinf(want) and math.isinf(float(got[i])))
