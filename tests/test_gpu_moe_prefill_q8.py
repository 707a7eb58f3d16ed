"""The integer route of the grouped MoE prefill layer (moex_moe_prefill_q8) on
the GPU, stage by stage:

(a) the expert sort (order, counts) is bit-exact to the oracle's stable sort;
(b) Hq and its {d, s} are bit-exact to the oracle's q8_1 of the GPU's own FP32
    H (the same quantiser arithmetic on the same inputs);
(c) H agrees with the oracle's silu(g) * u within the GEMV tolerance carried
    through SiLU plus a few FP32 ulps (the first product's FP32 tensor-core
    sums and the fast exponential);
(d) out, computed by the oracle on the GPU's own H, is within
    1e-5 * sum|w*x| + 1e-6 per element (block-integer down product, FP32
    scales, atomic combine).
"""
import numpy as np
import pytest

import synth
from helpers import assert_within, ensure_lib, to_np
from oracle import moe as om
from oracle import prefill as op

pytestmark = pytest.mark.gpu


def build(E, hidden, inter, experts, seed, gu_fmt, dn_fmt):
    import moe_expert_gb300 as mx
    gu = mx.PackedWeight(gu_fmt, E, 2 * inter, hidden).zero_()
    dn = mx.PackedWeight(dn_fmt, E, hidden, inter).zero_()
    gub, dnb = {}, {}
    for e in sorted(set(int(v) for v in experts)):
        gub[e] = synth.expert_blocks("gate_up", e, hidden, inter, gu_fmt, seed=seed)
        dnb[e] = synth.expert_blocks("down", e, hidden, inter, dn_fmt, seed=seed)
        gu.pack_matrix(e, gub[e])
        dn.pack_matrix(e, dnb[e])
    return gu, dn, gub, dnb


def run(T, E, k, hidden, inter, seed, sample=None, gu_fmt="iq4_nl", dn_fmt="iq4_nl", routing=None):
    import torch
    import moe_expert_gb300 as mx
    ensure_lib()
    xb = synth.bf16_activations(synth.rng(seed), T, hidden)
    if routing is None:
        ids, w = om.route_topk(synth.router_logits(synth.rng(seed + 1), T, E), k)
    else:
        ids, w = routing
    w = w.astype(np.float32)
    gu, dn, gub, dnb = build(E, hidden, inter, ids.reshape(-1), seed, gu_fmt, dn_fmt)
    n = T * k
    ws = torch.zeros(mx.moe_prefill_q8_workspace_bytes(T, k, E, hidden, inter), dtype=torch.uint8, device="cuda")
    hdbg = torch.full((n, inter), float("nan"), dtype=torch.float32, device="cuda")
    out = to_np(mx.moe_prefill_q8(gu, dn, torch.from_numpy(xb.view(np.int16)).cuda(),
                                  torch.from_numpy(ids.astype(np.int32)).cuda(), torch.from_numpy(w).cuda(),
                                  ws=ws, h_dbg=hdbg))
    assert mx.device_status() == 0
    off = mx.moe_prefill_q8_workspace_layout(T, k, E, hidden, inter)
    wsh = to_np(ws)
    counts = wsh[off[0]:off[0] + 4 * E].view(np.int32)
    order = wsh[off[1]:off[1] + 4 * n].view(np.int32)
    r_order, r_off = op.sort_entries(ids, E)
    # (a)
    assert np.array_equal(order.astype(np.int64), r_order)
    assert np.array_equal(counts.astype(np.int64), np.diff(r_off))
    pos = np.empty(n, dtype=np.int64)
    pos[order] = np.arange(n)
    Hq = wsh[off[7]:off[7] + n * inter].view(np.int8).reshape(n, inter)
    Hds = wsh[off[8]:off[8] + 8 * n * (inter // 32)].view(np.float32).reshape(n, inter // 32, 2)
    Hg = to_np(hdbg)
    toks = list(range(T)) if sample is None else list(sample)
    gpu_h = lambda t, s: Hg[pos[t * k + s]]  # noqa: E731
    ref = op.moe_prefill_q8(gub, dnb, xb, ids, w.astype(np.float64), tokens=toks, h_override=gpu_h, fmt=gu_fmt,
                            down_fmt=dn_fmt)
    own = op.moe_prefill_q8(gub, dnb, xb, ids, w.astype(np.float64), tokens=toks, fmt=gu_fmt, down_fmt=dn_fmt)
    for i, t in enumerate(toks):
        for s in range(k):
            row = pos[t * k + s]
            # (b)
            assert np.array_equal(Hq[row], ref["Hq"][i, s]), (t, s)
            assert np.array_equal(Hds[row, :, 0], ref["Hd"][i, s]), (t, s)
    # (b) the block sums s = d * sum(q), one FP32 product
    rows = pos[np.array([t * k + s for t in toks for s in range(k)])]
    qs = Hq[rows].reshape(len(rows), inter // 32, 32).astype(np.int64).sum(axis=2).astype(np.float32)
    assert np.array_equal(Hds[rows, :, 1], (Hds[rows, :, 0] * qs).astype(np.float32))
    # (c)
    g, u = own["g"], own["u"]
    gA, uA = own["gu_A"][..., :inter], own["gu_A"][..., inter:]
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    Hgpu = np.stack([np.stack([gpu_h(t, s) for s in range(k)]) for t in toks]).astype(np.float64)
    bound = 1e-5 * (np.abs(dsilu * u) * gA + np.abs(g * sig) * uA) + 8 * 2.0 ** -24 * np.abs(own["H"]) + 1e-30
    ratio = np.abs(Hgpu - own["H"]) / bound
    assert np.all(ratio <= 1.0), float(ratio.max())
    # (d)
    return assert_within(out[toks], ref["out"], ref["out_A"], "integer-route out on the GPU's H")


@pytest.mark.parametrize("T,E,k,hidden,inter", [
    (64, 8, 2, 256, 128),      # CTA pairs in the first product
    (600, 4, 2, 256, 64),      # single CTAs (odd feature-tile count); 300 rows an expert
    (333, 16, 4, 512, 256),
])
def test_prefill_q8_small(T, E, k, hidden, inter):
    worst = run(T, E, k, hidden, inter, seed=T + E + 1)
    print(f"worst out error / tolerance {worst:.3f}")


def test_prefill_q8_tile_boundaries():
    """Experts with 0, 1, 63, 64, 65, 128, 130 and 193 rows (k = 1): the down
    product's 64-row token tiles (empty, one row, full, one over, two full,
    ragged) and the first product's 192-row tiles."""
    counts = [0, 1, 63, 64, 65, 128, 130, 193]
    E, T = len(counts), sum(counts)
    g = np.random.default_rng(23)
    ids = np.repeat(np.arange(E), counts)
    g.shuffle(ids)
    w = g.uniform(0.2, 1.0, size=T).astype(np.float32)
    worst = run(T, E, 1, 256, 128, seed=31, routing=(ids.reshape(T, 1), w.reshape(T, 1)))
    print(f"worst out error / tolerance {worst:.3f}")


def test_prefill_q8_q8_0_weights():
    """Q8_0 gate/up and Q8_0 down."""
    worst = run(300, 8, 2, 512, 128, seed=97, gu_fmt="q8_0", dn_fmt="q8_0")
    print(f"worst out error / tolerance {worst:.3f}")


def test_prefill_q8_workload_full_size_sampled():
    """8192 tokens, 128 IQ4_NL experts top-8, hidden 2560, inter 1536: the whole
    sort, and every expert's first and last sorted row plus 64 drawn tokens
    recomputed by the oracle."""
    T, E, k, seed = 8192, 128, 8, 0
    ids, _ = om.route_topk(synth.router_logits(synth.rng(seed + 1), T, E), k)
    order, off = op.sort_entries(ids, E)
    edge = [order[off[e]] // k for e in range(E) if off[e + 1] > off[e]]
    edge += [order[off[e + 1] - 1] // k for e in range(E) if off[e + 1] > off[e]]
    extra = np.random.default_rng(12).choice(T, 64, replace=False)
    sample = sorted(set(int(t) for t in edge) | set(int(t) for t in extra))
    worst = run(T, E, k, 2560, 1536, seed=seed, sample=sample)
    print(f"{len(sample)} tokens: worst out error / tolerance {worst:.3f}")
