"""Benchmark of the block-quantized decode GEMV path on GB300.

Headline workload: Q8_0 weights 8192 x 2560 against q8_1 activations; one
step = quantize_q8_1 of the step's 15 FP32 columns (one launch), then the
multi-column GEMV for ncols 1, 2, 4 and 8, each on the next of enough rotated
weight copies that the weights are cold (3x L2).  value = weight GB/s over the timed steps (bytes of
the four GEMVs / time); the per-column-count microseconds per call, the
IQ4_NL 12288 x 2560 GEMV and the grouped MoE decode layer are reported in
"detail".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the only reference of this method) on
a bounded sample of the same workload.  N > 1 (torchrun) runs independent
replicas, one per GPU, with a barrier and the max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "quantized GEMV µs/call + weight GB/s (% of GB300 HBM peak), 1–8 cols; MoE layer µs"
ROWS, K = 8192, 2560
NCOLS = (1, 2, 4, 8)
W_BYTES = ROWS * (K // 32) * 34           # algorithmic Q8_0 bytes per GEMV call


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], "measured"
    return 6800.0, "fallback"


def peak_fp16():
    """Dense FP16 tensor peak in TFLOP/s: the measured BF16 cuBLAS burst figure
    (FP16 and BF16 run at the same tcgen05 rate)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return json.load(open(p)).get("bf16_tflops", 1900.0)
    return 1900.0


# ---------------------------------------------------------------- distributed

def dist_setup(n_gpus):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, ws):
    """The largest v over the ranks (the job's time is its slowest rank's)."""
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.proc, self.out = gpu, None, None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            self.out = ""

    def summary(self):
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- our arm

def cold_copies(nbytes, l2_bytes):
    return max(6, math.ceil(3 * l2_bytes / nbytes))


class GemvCase:
    """Rotated cold copies of one weight matrix plus activations per ncols."""

    def __init__(self, fmt, rows, k, ncols_list, l2_bytes):
        import torch
        import moe_expert_gb300 as mx
        self.fmt, self.rows, self.K = fmt, rows, k
        blocks, _ = synth.dense_case(fmt, rows, k, 1)
        self.bytes = rows * (k // 32) * (34 if fmt == "q8_0" else 18)
        self.ncopies = cold_copies(self.bytes, l2_bytes)
        w0 = mx.PackedWeight.from_gguf(fmt, blocks)
        self.W = [w0]
        for _ in range(self.ncopies - 1):
            w = mx.PackedWeight(fmt, 1, rows, k)
            w.qs.copy_(w0.qs)
            w.scales.copy_(w0.scales)
            self.W.append(w)
        # the activations of every column count of a step, stacked so one
        # quantize_q8_1 call covers the step; x[c], xq[c], xds[c] are views
        ntot = sum(ncols_list)
        self.x_all = torch.empty((ntot, k), dtype=torch.float32, device="cuda")
        self.y_all = torch.empty((ntot, rows), dtype=torch.float32, device="cuda")
        self.xq_all = torch.empty((ntot, k), dtype=torch.int8, device="cuda")
        self.xds_all = torch.empty((ntot, k // 32, 2), dtype=torch.float32, device="cuda")
        self.x, self.xq, self.xds, self.y = {}, {}, {}, {}
        o = 0
        for c in ncols_list:
            self.x_all[o:o + c].copy_(torch.from_numpy(synth.activations(synth.rng(100 + c), c, k)))
            self.x[c], self.xq[c], self.xds[c] = self.x_all[o:o + c], self.xq_all[o:o + c], self.xds_all[o:o + c]
            self.y[c] = self.y_all[o:o + c]
            o += c

    def step(self, i, ncols_list, quantize=True):
        """One step: q8_1 of all the step's columns (one launch), then the
        GEMV of each column count on the next cold weight copy."""
        import moe_expert_gb300 as mx
        if quantize:
            mx.quantize_q8_1(self.x_all, self.xq_all, self.xds_all)
        for j, c in enumerate(ncols_list):
            w = self.W[(i * len(ncols_list) + j) % self.ncopies]
            mx.qgemv(w, self.xq[c], self.xds[c], self.y[c])


def graphs_for(fn, n):
    """n CUDA graphs, graph i capturing fn(i); each is replayed once after
    capture (untimed), so no first-launch upload lands in a timed region."""
    import torch
    gs = []
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(min(n, 3)):
            fn(i)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for i in range(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(i)
        gs.append(g)
    for g in gs:
        g.replay()
    torch.cuda.synchronize()
    return gs


def time_graphs(gs, steps, warmup):
    """Replays graph (i mod len) for warmup + steps; returns seconds of the timed steps."""
    import torch
    for i in range(warmup):
        gs[i % len(gs)].replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        gs[(warmup + i) % len(gs)].replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e-3


def rotation_graph_seconds(case, c, reps):
    """Seconds per GEMV call: one graph holds one call on every cold copy (so
    graph launch overhead is amortised over case.ncopies kernels); replayed
    until at least `reps` calls were timed."""
    import moe_expert_gb300 as mx

    def body(_):
        for i in range(case.ncopies):
            mx.qgemv(case.W[i], case.xq[c], case.xds[c], case.y[c])
    gs = graphs_for(body, 1)
    n = max(1, math.ceil(reps / case.ncopies))
    t = time_graphs(gs, n, 3)
    return t / (n * case.ncopies)


def gemv_detail(case, ncols_list, reps, peak):
    """Per-ncols microseconds per GEMV call over the rotated cold copies."""
    out = {}
    for c in ncols_list:
        per = rotation_graph_seconds(case, c, reps)
        us = per * 1e6
        gbs = case.bytes / per / 1e9
        out[str(c)] = {"us_per_call": round(us, 3), "weight_GBps": round(gbs, 1), "frac_hbm": round(gbs / peak, 3)}
    return out


def decode_layer_detail(reps, copies=3):
    """Grouped MoE decode layer (route + 2 kernels) on the 20-expert routing,
    rotating `copies` full 128-expert layers so the weights are cold."""
    import torch
    import moe_expert_gb300 as mx
    ref = json.load(open(os.path.join(ROOT, "tests", "golden", "decode_routing.json")))
    T, E, k = ref["tokens"], ref["experts"], ref["top_k"]
    hidden, inter = 2560, 1536
    logits = torch.from_numpy(synth.decode_logits(T, E, ref["sub_seed"])).cuda()
    x = torch.from_numpy(synth.decode_tokens(T, hidden)).cuda()
    routed = sorted(set(int(v) for v in np.array(ref["ids"]).reshape(-1)))
    layers = []
    for c in range(copies):
        gu = mx.PackedWeight("q8_0", E, 2 * inter, hidden).zero_()
        dn = mx.PackedWeight("iq4_nl", E, hidden, inter).zero_()
        for e in routed:
            gu.pack_matrix(e, synth.expert_blocks("gate_up", e, hidden, inter, "q8_0"))
            dn.pack_matrix(e, synth.expert_blocks("down", e, hidden, inter, "iq4_nl"))
        layers.append((gu, dn))
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    out = torch.empty((T, hidden), dtype=torch.float32, device="cuda")
    ws = torch.empty(mx.moe_decode_workspace_bytes(T, k, hidden, inter), dtype=torch.uint8, device="cuda")

    def layer(i, route=True):
        gu, dn = layers[i % copies]
        if route:
            mx.route_topk(logits, k, ids, w)
        mx.moe_decode(gu, dn, x, ids, w, out, ws)

    gs = graphs_for(lambda i: layer(i, True), copies)
    t = time_graphs(gs, reps, 10)
    gs2 = graphs_for(lambda i: layer(i, False), copies)
    t2 = time_graphs(gs2, reps, 10)
    wbytes = len(routed) * (2 * inter * (hidden // 32) * 34 + hidden * (inter // 32) * 18)
    return {"tokens": T, "entries": T * k, "experts_routed": len(routed),
            "layer_us": round(t / reps * 1e6, 2), "decode_only_us": round(t2 / reps * 1e6, 2),
            "weight_bytes": wbytes, "weight_GBps": round(wbytes / (t2 / reps) / 1e9, 1)}


def prefill_layer_detail(reps=5, peak_tflops=None, T=8192, E=128, route="fp16"):
    """Grouped MoE prefill layer: T tokens x top-8 of E IQ4_NL experts,
    hidden 2560, inter 1536 (route + sort + gather + two tcgen05 GEMMs).
    The workload is 8192 tokens over 128 experts; 4096 over 64 keeps the
    same rows per expert at half the memory (the profiler's case)."""
    import torch
    import moe_expert_gb300 as mx
    k, hidden, inter = 8, 2560, 1536
    gu = mx.PackedWeight("iq4_nl", E, 2 * inter, hidden)
    dn = mx.PackedWeight("iq4_nl", E, hidden, inter)
    for e in range(E):
        gu.pack_matrix(e, synth.expert_blocks("gate_up", e, hidden, inter, "iq4_nl"))
        dn.pack_matrix(e, synth.expert_blocks("down", e, hidden, inter, "iq4_nl"))
    x = torch.from_numpy(synth.prefill_tokens(T, hidden).view(np.int16)).cuda()
    logits = torch.from_numpy(synth.prefill_logits(T, E)).cuda()
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    out = torch.empty((T, hidden), dtype=torch.float32, device="cuda")
    if route == "int8":
        ws = torch.empty(mx.moe_prefill_q8_workspace_bytes(T, k, E, hidden, inter), dtype=torch.uint8, device="cuda")
    else:
        ws = torch.empty(mx.moe_prefill_workspace_bytes(T, k, E, hidden, inter), dtype=torch.uint8, device="cuda")

    def layer():
        mx.route_topk(logits, k, ids, w)
        if route == "int8":
            mx.moe_prefill_q8(gu, dn, x, ids, w, out, ws)
        else:
            mx.moe_prefill(gu, dn, x, ids, w, out, ws)
    for _ in range(2):
        layer()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        layer()
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / reps
    flops = 2.0 * T * k * (2 * inter * hidden + hidden * inter)
    d = {"route": route, "tokens": T, "experts": E, "top_k": k, "layer_ms": round(t * 1e3, 3),
         "algorithmic_tflop": round(flops / 1e12, 4), "layer_tflops": round(flops / t / 1e12, 1)}
    if peak_tflops:
        d["frac_of_fp16_dense_peak"] = round(flops / t / 1e12 / peak_tflops, 3)
    return d


GEMV_SOURCES = ("moe_expert_gb300/csrc/qgemv.cu", "moe_expert_gb300/csrc/gemv_core.cuh",
                "moe_expert_gb300/csrc/common.cuh")


def sources_digest(paths):
    import hashlib
    h = hashlib.sha256()
    for p in paths:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(name, sources):
    """DRAM bytes per launch of the dominant kernel from its ncu summary in
    profiles/ (lines 'dram_bytes_per_launch: N' and 'sources_sha256_16: H');
    None when the kernel sources changed since that capture."""
    p = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p):
        if ":" in line:
            key, _, v = line.partition(":")
            vals[key.strip().lstrip("-* ")] = v.strip().strip("`")
    if vals.get("sources_sha256_16") != sources_digest(sources):
        return None
    try:
        return int(float(vals["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


def dense_prefill_detail(reps=10, peak_tflops=None, T=8192, R=12288, K=2560):
    """Dense prefill product of an IQ4_NL R x K matrix over T BF16 tokens on
    the tensor cores (tile list + BF16 -> FP16 rows + the GEMM)."""
    import torch
    import moe_expert_gb300 as mx
    blocks, _ = synth.dense_case("iq4_nl", R, K, 1)
    W = mx.PackedWeight.from_gguf("iq4_nl", blocks)
    x = torch.from_numpy(synth.prefill_tokens(T, K).view(np.int16)).cuda()
    y = torch.empty((T, R), dtype=torch.float32, device="cuda")
    wsb = torch.empty(mx.lib().moex_dense_prefill_workspace_bytes(T, R, K), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        mx.dense_prefill(W, x, y, wsb)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        mx.dense_prefill(W, x, y, wsb)
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / reps
    flops = 2.0 * T * R * K
    d = {"tokens": T, "rows": R, "K": K, "ms": round(t * 1e3, 3), "tflops": round(flops / t / 1e12, 1)}
    if peak_tflops:
        d["frac_of_fp16_dense_peak"] = round(flops / t / 1e12 / peak_tflops, 3)
    return d


def run_ours(args, ws, rank, local):
    import torch
    import moe_expert_gb300 as mx
    mx.lib()
    torch.cuda.set_device(local)
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 126 * 2**20) or 126 * 2**20
    peak, peak_src = peaks()
    case = GemvCase("q8_0", ROWS, K, NCOLS, l2)
    # step i runs on rotation position i mod G of the cold weight copies.  The
    # timed steps start at position p0 = W mod G and are replayed as graphs of
    # `chunk` consecutive steps (whole rotations, so every chunk starts at p0),
    # the rest (fewer than a chunk) as one-step graphs: one graph launch paces
    # at most one chunk, for any step count.
    G = case.ncopies
    p0 = args.warmup % G
    chunk = G * max(1, min(args.steps, 512) // G)
    gs = graphs_for(lambda i: case.step(i, NCOLS), G)
    big = graphs_for(lambda _: [case.step(p0 + j, NCOLS) for j in range(chunk)], 1)[0]

    def run_timed(count):
        n_big, rem = divmod(count, chunk)
        for _ in range(n_big):
            big.replay()
        for j in range(rem):
            gs[(p0 + j) % G].replay()
    # warm-up + timed steps (device time, CUDA events), clocks sampled meanwhile
    for i in range(args.warmup):
        gs[i % G].replay()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run_timed(args.steps)
        e1.record()
        torch.cuda.synchronize()
    barrier(ws)
    t = max_over_ranks(e0.elapsed_time(e1) * 1e-3, ws)
    step_bytes = W_BYTES * len(NCOLS)
    value = ws * step_bytes * args.steps / t / 1e9
    ms_per_step = t / args.steps * 1e3

    # dominant kernel: the GEMV alone, average launch duration over the cold copies
    kern = {}
    kt = 0.0
    for c in NCOLS:
        kern[c] = rotation_graph_seconds(case, c, max(1000, args.steps // 4))
        kt += kern[c]
    avg_launch = kt / len(NCOLS)
    achieved = W_BYTES / avg_launch / 1e9
    traffic = profiled_traffic("qgemv_q8_0_8192x2560.md", GEMV_SOURCES)

    # end to end through the public API: pinned host X in, host Y out, eager calls
    xs_h = case.x_all.cpu().pin_memory()
    ys_h = torch.empty(case.y_all.shape, dtype=torch.float32).pin_memory()  # every column count's Y, one read
    e2e_steps = max(50, min(args.steps, 2000))

    def e2e_step(i):
        case.x_all.copy_(xs_h, non_blocking=True)
        mx.quantize_q8_1(case.x_all, case.xq_all, case.xds_all)
        for j, c in enumerate(NCOLS):
            w = case.W[(i * len(NCOLS) + j) % case.ncopies]
            mx.qgemv(w, case.xq[c], case.xds[c], case.y[c])
        ys_h.copy_(case.y_all, non_blocking=True)
    for i in range(min(args.warmup, 20)):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(ws)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    te = max_over_ranks(time.perf_counter() - t0, ws)
    e2e_value = ws * step_bytes * e2e_steps / te / 1e9
    h2d = sum(c * K * 4 for c in NCOLS)
    d2h = sum(c * ROWS * 4 for c in NCOLS)

    detail = {}
    if rank == 0 and not args.no_detail:
        detail["q8_0_8192x2560"] = gemv_detail(case, NCOLS, 2000, peak)
        del case, gs, big
        torch.cuda.empty_cache()
        iq = GemvCase("iq4_nl", 12288, K, (1, 2, 3, 4, 8), l2)
        for c in (1, 2, 3, 4, 8):
            mx.quantize_q8_1(iq.x[c], iq.xq[c], iq.xds[c])
        detail["iq4_nl_12288x2560"] = gemv_detail(iq, (1, 2, 3, 4, 8), 2000, peak)
        del iq
        torch.cuda.empty_cache()
        head = GemvCase("q8_0", 128256, K, (1, 8), l2)
        for c in (1, 8):
            mx.quantize_q8_1(head.x[c], head.xq[c], head.xds[c])
        detail["q8_0_head_128256x2560"] = gemv_detail(head, (1, 8), 200, peak)
        del head
        torch.cuda.empty_cache()
        small = GemvCase("q8_0", 512, 2048, (1,), l2)
        mx.quantize_q8_1(small.x[1], small.xq[1], small.xds[1])
        detail["q8_0_512x2048"] = gemv_detail(small, (1,), 2000, peak)
        del small
        torch.cuda.empty_cache()
        detail["moe_decode_20_experts"] = decode_layer_detail(500)
        torch.cuda.empty_cache()
        detail["moe_prefill_8192_tokens"] = prefill_layer_detail(5, peak_fp16())
        torch.cuda.empty_cache()
        detail["moe_prefill_int8_route_8192_tokens"] = prefill_layer_detail(3, None, route="int8")
        torch.cuda.empty_cache()
        detail["dense_prefill_iq4_nl_12288x2560_8192_tokens"] = dense_prefill_detail(10, peak_fp16())

    cpu = cpu_baseline(budget_s=args.cpu_budget) if (rank == 0 and not args.no_cpu) else None
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": workload_config(l2, ws),
        "gpu_launches": args.steps * (1 + len(NCOLS)),
        "clocks": clk.summary(),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "qgemv_kernel (Q8_0, 8192x2560), mean over ncols 1/2/4/8",
                     "avg_launch_us": round(avg_launch * 1e6, 3), "peak_source": peak_src},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "how": "public Python API, eager launches, pinned host X in and host Y out every step"},
        "cpu_baseline": cpu,
        "detail": detail,
    }
    print(json.dumps(line))


def case_copies(l2):
    return cold_copies(W_BYTES, l2)


def workload_config(l2, ws):
    """The config of both arms' JSON lines (the reference arm reports the
    same workload it samples)."""
    return {"workload": "Q8_0 decode GEMV 8192x2560 x q8_1 activations, ncols 1/2/4/8 per step "
                        "(one quantize_q8_1 of the step's 15 columns, then a qgemv per column count), "
                        "cold weights",
            "rows": ROWS, "K": K, "ncols": list(NCOLS), "weight_copies": case_copies(l2),
            "l2": "inputs larger than L2: rotated weight copies totalling 3x L2",
            "parallelism": f"replicas x{ws}"}


def device_l2_bytes():
    """L2 size of GPU 0 when torch sees one, else the GB300 figure."""
    try:
        import torch
        if torch.cuda.is_available():
            v = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 0)
            if v:
                return v
    except Exception:
        pass
    return 126 * 2**20


# ---------------------------------------------------------------- CPU oracle

def oracle_step(rows_sample: int, row0: int = 0):
    """The oracle on a row slab of the same workload: q8_1 of the columns and
    the GEMV of rows row0 .. row0+rows_sample-1, for ncols 1, 2, 4, 8."""
    from oracle import gemv as og
    from oracle import q8_1 as oq
    blocks, _ = synth.dense_case("q8_0", ROWS, K, 1)
    blocks = blocks[row0:row0 + rows_sample]
    xs = {c: synth.activations(synth.rng(100 + c), c, K) for c in NCOLS}

    def step():
        for c in NCOLS:
            q, d, _ = oq.quantize_q8_1(xs[c])
            og.gemv("q8_0", blocks, q, d)
    return step, rows_sample * (K // 32) * 34 * len(NCOLS)


# One oracle slab per pool worker (processes started with spawn, so no CUDA
# state is inherited).  The worker builds its slab once, then runs it per task.
_SLAB = None


def _slab_init(rows, row0):
    global _SLAB
    _SLAB = oracle_step(rows, row0)[0]


def _slab_run(_):
    _SLAB()
    return 0


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


class OraclePool:
    """The oracle over all host cores: one spawn process per core, each owning
    a contiguous slab of the rows; a step runs every slab once."""

    def __init__(self, rows: int, ncores: int):
        import multiprocessing as mp
        self.rows, self.ncores = rows, ncores
        ctx = mp.get_context("spawn")
        bounds = [rows * i // ncores for i in range(ncores + 1)]
        self.pools = [ctx.Pool(1, initializer=_slab_init, initargs=(bounds[i + 1] - bounds[i], bounds[i]))
                      for i in range(ncores) if bounds[i + 1] > bounds[i]]
        self.nbytes = rows * (K // 32) * 34 * len(NCOLS)

    def step(self):
        rs = [p.apply_async(_slab_run, (0,)) for p in self.pools]
        for r in rs:
            r.get()

    def close(self):
        for p in self.pools:
            p.close()
            p.join()


def cpu_baseline(budget_s=15.0):
    """The oracle as it stands on the host: one core on a 512-row sample, then
    all cores (a spawn pool, one row slab per core) on the whole workload."""
    step1, nb1 = oracle_step(512)
    step1()
    t0 = time.perf_counter()
    n1 = 0
    while time.perf_counter() - t0 < budget_s / 4:
        step1()
        n1 += 1
    one_core = nb1 * n1 / (time.perf_counter() - t0) / 1e9
    ncores = os.cpu_count() or 1
    pool = OraclePool(ROWS, ncores)
    pool.step()  # slabs built, warm
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < budget_s * 3 / 4:
        pool.step()
        n += 1
    wall = time.perf_counter() - t0
    pool.close()
    return {"value": round(pool.nbytes * n / wall / 1e9, 4), "unit": "GB/s", "cores": len(pool.pools),
            "kind": "oracle", "cpu_model": cpu_model(), "one_core_value": round(one_core, 4),
            "sample": f"{n} oracle step(s) of the whole workload ({ROWS} rows, q8_1 + block-integer GEMV, "
                      f"ncols 1/2/4/8) over {len(pool.pools)} processes (one row slab each), {wall:.1f} s wall; "
                      f"one core: {n1} step(s) on 512 rows",
            "wall_s": round(wall, 2)}


def run_reference(args, ws, rank):
    if rank != 0:
        return
    ncores = os.cpu_count() or 1
    # size the per-step sample (whole slabs over all cores) so warm-up + timed
    # steps end within about two minutes
    probe_rows = 64
    step, _ = oracle_step(probe_rows)
    step()
    t0 = time.perf_counter()
    step()
    per_row_core = (time.perf_counter() - t0) / probe_rows
    budget = 120.0
    rows = int(budget * ncores / max(1, args.steps + args.warmup) / max(per_row_core, 1e-9))
    rows = max(ncores, min(ROWS, rows))
    pool = OraclePool(rows, ncores)
    for _ in range(args.warmup):
        pool.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        pool.step()
    wall = time.perf_counter() - t0
    pool.close()
    value = pool.nbytes * args.steps / wall / 1e9
    sample = (f"each step: the oracle's q8_1 + block-integer GEMV on {rows} of {ROWS} rows, ncols 1/2/4/8, "
              f"over {len(pool.pools)} processes (one row slab each)")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64+f64",
            "data": "synthetic", "config": workload_config(device_l2_bytes(), ws),
            "gpu_launches": 0,
            "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": len(pool.pools),
                             "kind": "oracle", "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_only(args):
    """One kernel in an eager loop on the full-size workload (for profilers)."""
    import torch
    import moe_expert_gb300 as mx
    mx.lib()
    props = torch.cuda.get_device_properties(0)
    l2 = getattr(props, "L2_cache_size", 126 * 2**20) or 126 * 2**20
    c = args.ncols
    if args.only in ("gemv_q8_0", "gemv_iq4_nl"):
        fmt, rows = ("q8_0", ROWS) if args.only == "gemv_q8_0" else ("iq4_nl", 12288)
        case = GemvCase(fmt, rows, K, (c,), l2)
        mx.quantize_q8_1(case.x[c], case.xq[c], case.xds[c])
        fn = lambda i: mx.qgemv(case.W[i % case.ncopies], case.xq[c], case.xds[c], case.y[c])  # noqa: E731
    elif args.only == "prefill":
        d = prefill_layer_detail(max(1, args.steps), peak_fp16(), args.pf_tokens, args.pf_experts)
        print(json.dumps({"only": "prefill", **d}))
        return
    elif args.only == "prefill_q8":
        d = prefill_layer_detail(max(1, args.steps), None, args.pf_tokens, args.pf_experts, route="int8")
        print(json.dumps({"only": "prefill_q8", **d}))
        return
    elif args.only == "dense_prefill":
        print(json.dumps({"only": "dense_prefill", **dense_prefill_detail(max(1, args.steps), peak_fp16())}))
        return
    elif args.only == "decode":
        d = decode_layer_detail(max(1, args.steps))
        print(json.dumps({"only": "decode", **d}))
        return
    else:
        raise SystemExit(f"unknown --only {args.only}")
    for i in range(args.warmup):
        fn(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        fn(args.warmup + i)
    torch.cuda.synchronize()
    print(json.dumps({"only": args.only, "ncols": c, "steps": args.steps,
                      "us_per_call_eager": round((time.perf_counter() - t0) / args.steps * 1e6, 2)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--only", default=None, help="profile helper: gemv_q8_0 | gemv_iq4_nl | decode | prefill | prefill_q8 | dense_prefill")
    ap.add_argument("--ncols", type=int, default=1)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-detail", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--pf-tokens", type=int, default=8192, help="--only prefill: tokens")
    ap.add_argument("--pf-experts", type=int, default=128, help="--only prefill: experts")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.only:
        run_only(args)
        return
    if args.impl == "reference":
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, ws, rank)
        return
    ws, rank, local = dist_setup(args.gpus)
    run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
