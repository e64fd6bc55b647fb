"""Benchmark of the weight-only-quantized linear layer on GB300.

Workload: a 7B-shaped decoder layer sweep -- per layer the projections
q, k, v, o (N=4096, K=4096), gate, up (N=11008, K=4096) and down (N=4096,
K=11008), 32 distinct layers, each in two formats: 4-bit GPTQ (group 128,
symmetric, bf16 activations and output) and ternary W2A8 (PQ2 blocks, int8
activations quantised per row, bf16 output).  Weights: 3.34 GB (4-bit) plus
1.72 GB (ternary), far larger than L2, so no timed iteration is served from
L2.  Synthetic, seeded weights and activations.

One step = the decode pass at M = 1 over all 32 layers and both formats,
captured in one CUDA graph that follows a decoder layer's data flow in
stream order: q|k|v (the three projections that read one input, prepared as
one stacked 12288x4096 layer), o, gate|up (stacked, 22016x4096), down -- 256
pq_linear calls dispatched to the decode GEMVs.  The same pass over the
seven separate projections per layer (448 calls, q|k|v and gate|up on
fork/join streams) is reported beside it.  The headline value is
packed-weight GB/s: prepared code + scale bytes of every layer read per step
/ step time.  The same JSON line carries alternating-pair medians against the
copy-only read probe over the same bytes and launch chain, the prefill pass
at M = 2048 (tensor-core GEMM) in TFLOP/s, the dominant kernels' rooflines,
end-to-end numbers through the C ABI with host buffers (graph replay, and
256 ctypes calls per step), the fused activation producer of the ternary
layers, and the CPU oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --table      # one JSON line per configuration, oracle beside it
  python bench.py --producer   # only the fused producer figures
  python bench.py --probe      # only the copy-only read probe
  python bench.py --table --rows 7 --reps 1   # one configuration (profiler captures)
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "packed-weight GB/s (% of HBM peak) at M=1; TFLOP/s (% bf16 peak) at M=2048"
UNIT = "GB/s"
WORKLOAD = ("7B-shaped decoder layer sweep: q/k/v/o 4096x4096, gate/up 11008x4096, down 4096x11008 "
            "(q|k|v and gate|up stacked into one layer each); 32 layers; W4A16 g128 + ternary W2A8")
SHAPES = [("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
          ("gate", 11008, 4096), ("up", 11008, 4096), ("down", 4096, 11008)]   # (name, N, K)
# the projections that read one input, prepared as one concatenated layer
MERGED = [("qkv", 12288, 4096), ("gu", 22016, 4096)]
LAYERS = 32
PREFILL_M = 2048
PAIRS = 9                      # alternating (decode step, probe step) pairs


def w4_bytes(N, K):
    return N * K // 2 + N * (K // 128) * 2          # codes + fp16 scales


def w2_bytes(N, K):
    return N * K // 4 + N * (K // 128) * 2          # 34 bytes per 128 weights


def flops(M, N, K):
    return 2.0 * M * N * K


def peaks():
    p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            m = json.load(fh)
        p.update({k: float(m[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained") if k in m})
        p["source"] = "measured"
    except (OSError, ValueError, KeyError):
        pass
    return p


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons, taken while
    the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ our arm

def build_layers(torch, pq, pq_inputs, dev, M_max, rank):
    """32 layers x 7 projections in both formats, prepared on the device,
    plus each layer's q|k|v and gate|up projections prepared a second time
    as one concatenated layer (12288x4096 and 22016x4096: the same weights,
    rows stacked, so one call computes the three or two outputs side by
    side).  All handles share one workspace (calls run in stream order).

    Returns (w4, w2, w4m, w2m, keep, workspace): the per-projection lists of
    (name, N, K, handle), the merged lists (qkv, o, gu, down per layer; o and
    down are the same handles), the handle -> prepared-planes map and the
    workspace."""
    shapes = SHAPES
    ws_bytes = 0
    for _, N, K in shapes + MERGED:
        for d in (pq.make_desc(pq.PQ_FMT_W4_GPTQ, N, K, max_m=M_max),
                  pq.make_desc(pq.PQ_FMT_W2_PQ2, N, K, act_group=K, max_m=M_max)):
            ws_bytes = max(ws_bytes, pq.pq_workspace_bytes(d))
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    w4, w2, w4m, w2m = [], [], [], []
    keep = {}                                    # handle -> its prepared planes (device tensor)

    def prep_w4(N, K, qweight, scales):
        d = pq.make_desc(pq.PQ_FMT_W4_GPTQ, N, K, act_dtype=pq.PQ_BF16, max_m=M_max)
        prep = torch.empty(pq.pq_prepared_bytes(d), dtype=torch.uint8, device=dev)
        h = pq.pq_prepare_w4(d, qweight, scales, None, None, prep, prep.numel(), workspace, ws_bytes, stream)
        keep[h] = prep
        return h

    def prep_w2(N, K, raw):
        d = pq.make_desc(pq.PQ_FMT_W2_PQ2, N, K, act_dtype=pq.PQ_BF16, act_group=K, max_m=M_max)
        prep = torch.empty(pq.pq_prepared_bytes(d), dtype=torch.uint8, device=dev)
        h = pq.pq_prepare_w2(d, raw, raw.stride(0), prep, prep.numel(), workspace, ws_bytes, stream)
        keep[h] = prep
        return h

    for layer in range(LAYERS):
        f4, f2 = {}, {}
        for j, (name, N, K) in enumerate(shapes):
            seed = 1000 * rank + 10 * layer + j
            f4[name] = pq_inputs.device_w4_frame(seed, K, N, 0.002, 0.01, dev)
            f2[name] = pq_inputs.device_pq2_rows(seed + 500000, N, K, dev)
            w4.append((name, N, K, prep_w4(N, K, *f4[name])))
            w2.append((name, N, K, prep_w2(N, K, f2[name])))
        by4 = {n: e for n, *e in w4[-len(shapes):]}
        by2 = {n: e for n, *e in w2[-len(shapes):]}
        for mname, parts in (("qkv", ("q", "k", "v")), ("o", ("o",)), ("gu", ("gate", "up")), ("down", ("down",))):
            if len(parts) == 1:
                w4m.append((mname, *by4[parts[0]]))
                w2m.append((mname, *by2[parts[0]]))
                continue
            K = by4[parts[0]][1]
            N = sum(by4[p][0] for p in parts)
            qw = torch.cat([f4[p][0] for p in parts], dim=1).contiguous()
            sc = torch.cat([f4[p][1] for p in parts], dim=1).contiguous()
            w4m.append((mname, N, K, prep_w4(N, K, qw, sc)))
            raw = torch.cat([f2[p] for p in parts], dim=0).contiguous()
            w2m.append((mname, N, K, prep_w2(N, K, raw)))
            del qw, sc, raw
        del f4, f2
    torch.cuda.synchronize()
    return w4, w2, w4m, w2m, keep, workspace


def max_over_ranks(values, device):
    """Element-wise maximum of per-rank timings over the process group (the
    slowest replica sets the whole job's time)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()                                    # warm the launch path (attributes, maps)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def time_graph(torch, g, reps, stream, warm=True):
    """Average ms per replay with CUDA events on the replay stream (one
    untimed replay first unless warm is False)."""
    with torch.cuda.stream(stream):
        if warm:
            g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def read_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if present."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as fh:
            for line in fh:
                f = line.split()
                if len(f) >= 2 and f[0] == kernel:
                    return float(f[1])
    except OSError:
        pass
    return None


def run_ours(args, rank, world):
    import numpy as np
    import torch

    import bit_weight_quantized_pq_gb300 as pq
    import pq_inputs

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    pq.build()
    pq.lib()
    peak = peaks()
    M1, MP = 1, PREFILL_M
    w4, w2, w4m, w2m, keep, workspace = build_layers(torch, pq, pq_inputs, dev, MP, rank)
    stream = torch.cuda.Stream(dev)

    g = torch.Generator(device=dev)
    g.manual_seed(7 + rank)
    ks = sorted({k for _, _, k in SHAPES})
    ns = sorted({n for _, n, _ in SHAPES})
    x1 = {k: torch.randn((M1, k), generator=g, device=dev).to(torch.bfloat16) for k in ks}
    y1 = {n: torch.empty((M1, n), dtype=torch.bfloat16, device=dev) for n in ns}
    xp = {}
    for k in ks:
        a = torch.randn((MP, k), generator=g, device=dev)
        mask = torch.rand((MP, k), generator=g, device=dev) < 0.001       # 0.1% outliers x20
        xp[k] = torch.where(mask, a * 20.0, a).to(torch.bfloat16)
    yp = {n: torch.empty((MP, n), dtype=torch.bfloat16, device=dev) for n in ns}

    # Decode data flow of one layer: q, k and v read the same input and are
    # independent, as are gate and up; o needs q/k/v, down needs gate/up.
    # The step runs each layer as four calls in stream order on the merged
    # planes (qkv -> o -> gu -> down); the same pass over the seven separate
    # projections, with q|k|v and gate|up on fork/join streams, is measured
    # beside it (decode_per_projection).
    side = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    yproj = {name: torch.empty((M1, N), dtype=torch.bfloat16, device=dev) for name, N, _ in SHAPES + MERGED}
    groups = [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]]

    def decode_model(calls, issue):
        """The per-projection pass over `calls` (name, N, K, handle), one layer
        after another, each projection issued by issue(name, N, K, handle,
        stream), independent projections on fork/join streams."""
        by_layer = [calls[i:i + len(SHAPES)] for i in range(0, len(calls), len(SHAPES))]
        for layer in by_layer:
            proj = {name: (N, K, h) for name, N, K, h in layer}
            for grp in groups:
                if len(grp) == 1:
                    issue(grp[0], *proj[grp[0]], stream)
                    continue
                fork = torch.cuda.Event()
                fork.record(stream)
                joins = []
                for i, name in enumerate(grp):
                    s = stream if i == 0 else side[i - 1]
                    if i:
                        s.wait_event(fork)
                    issue(name, *proj[name], s)
                    if i:
                        ev = torch.cuda.Event()
                        ev.record(s)
                        joins.append(ev)
                for ev in joins:
                    stream.wait_event(ev)

    def chain(calls, issue):
        """The merged pass: every call in stream order on one stream."""
        for name, N, K, h in calls:
            issue(name, N, K, h, stream)

    def linear(name, N, K, h, s):
        pq.pq_linear(x1[K], h, yproj[name], M1, s)

    # the copy-only probe over the same bytes in the same launch chain: each
    # call replaced by one read of its layer's prepared planes, either waiting
    # for its predecessor first (as a layer waits for its input) or not (the
    # HBM limit of back-to-back launches)
    sink = torch.zeros(64, dtype=torch.int32, device=dev)
    nbytes_of = {h: w4_bytes(N, K) for _, N, K, h in w4 + w4m}
    nbytes_of.update({h: w2_bytes(N, K) for _, N, K, h in w2 + w2m})

    def probe(dep, cps):
        def issue(name, N, K, h, s):
            pq.pq_probe_read(keep[h], nbytes_of[h], sink, cps, dep, s)
        return issue

    def decode_w4():
        chain(w4m, linear)

    def decode_w2():
        chain(w2m, linear)

    def decode_step():
        decode_w4()
        decode_w2()

    def per_projection_step():
        decode_model(w4, linear)
        decode_model(w2, linear)

    def prefill_w4():
        for _, N, K, h in w4:
            pq.pq_linear(xp[K], h, yp[N], MP, stream)

    def prefill_w2():
        for _, N, K, h in w2:
            pq.pq_linear(xp[K], h, yp[N], MP, stream)

    step_bytes = sum(w4_bytes(N, K) for _, N, K, _ in w4m) + sum(w2_bytes(N, K) for _, N, K, _ in w2m)
    assert step_bytes == sum(w4_bytes(N, K) for _, N, K, _ in w4) + sum(w2_bytes(N, K) for _, N, K, _ in w2)
    g_step = capture(torch, decode_step, stream)
    g_probe_wait = capture(torch, lambda: chain(w4m + w2m, probe(1, 8)), stream)
    g_probe_free = capture(torch, lambda: chain(w4m + w2m, probe(0, 2)), stream)

    # ---- timed region: W warm-up steps, then exactly K steps
    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            g_step.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            g_step.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ms_step = e0.elapsed_time(e1) / args.steps
    # alternating (decode step, probe steps) replays, each timed alone;
    # medians over the pairs
    pair = {"step": [], "probe_wait": [], "probe_free": []}
    for _ in range(max(7, PAIRS)):
        pair["step"].append(time_graph(torch, g_step, 1, stream, warm=False))
        pair["probe_wait"].append(time_graph(torch, g_probe_wait, 1, stream, warm=False))
        pair["probe_free"].append(time_graph(torch, g_probe_free, 1, stream, warm=False))
    # per-projection pass, prefill pass, the dominant kernels' rooflines and
    # the read probe, inside the sampled window
    g_pp = capture(torch, per_projection_step, stream)
    ms_pp = time_graph(torch, g_pp, max(3, args.steps), stream)
    g_w4 = capture(torch, decode_w4, stream)
    g_w2 = capture(torch, decode_w2, stream)
    ms_w4 = time_graph(torch, g_w4, max(3, args.steps), stream)
    ms_w2 = time_graph(torch, g_w2, max(3, args.steps), stream)
    g_pw4 = capture(torch, prefill_w4, stream)
    g_pw2 = capture(torch, prefill_w2, stream)
    ms_p4 = time_graph(torch, g_pw4, 3, stream)
    ms_p2 = time_graph(torch, g_pw2, 3, stream)
    probe_rates = read_probe_rates(torch, pq, dev, stream)
    producer = measure_producer(torch, pq, dev, [h for *_, h in w2[:3]], stream, MP)
    producer["frac_of_hbm_peak_M2048"] = round(producer[f"GBs_M{MP}"] / peak["hbm_gbs"], 4)
    clk = clocks.stop()

    if world > 1:
        ms_step, ms_p4, ms_p2 = max_over_ranks([ms_step, ms_p4, ms_p2], dev)

    value = step_bytes * world / (ms_step * 1e-3) / 1e9
    n4, n2 = len(w4m), len(w2m)
    bytes_w4 = sum(w4_bytes(N, K) for _, N, K, _ in w4m) / n4
    bytes_w2 = sum(w2_bytes(N, K) for _, N, K, _ in w2m) / n2
    us_w4 = ms_w4 * 1e3 / n4
    us_w2 = ms_w2 * 1e3 / n2
    gbs_w4 = bytes_w4 / (us_w4 * 1e-6) / 1e9
    gbs_w2 = bytes_w2 / (us_w2 * 1e-6) / 1e9
    pf = [(N, K) for _, N, K, _ in w4]
    tf_p4 = sum(flops(MP, N, K) for N, K in pf) / (ms_p4 * 1e-3) / 1e12
    tf_p2 = sum(flops(MP, N, K) for N, K in pf) / (ms_p2 * 1e-3) / 1e12
    # the prefill runs as a burst at the clock the sampler saw: the burst
    # bf16 peak applies when the SM clock stayed at its maximum, the
    # sustained (power-capped) one otherwise
    at_max = bool(clk.get("sm_mhz") and clk.get("sm_max_mhz") and clk["sm_mhz"] >= 0.97 * clk["sm_max_mhz"])
    gemm_peak = peak["bf16_tflops"] if at_max else peak["bf16_tflops_sustained"]
    gemm_peak_kind = ("bf16_tflops (burst; SM clock at max while timed)" if at_max
                      else "bf16_tflops_sustained (SM clock below max while timed)") + f" ({peak['source']})"

    # ---- end to end through the C ABI with host buffers: every step copies
    # the step's activations from pinned host memory and reads the outputs back
    hx = {k: x1[k].cpu().pin_memory() for k in ks}
    hy = {name: torch.empty_like(yproj[name], device="cpu").pin_memory() for name in ("qkv", "o", "gu", "down")}
    h2d = sum(hx[k].numel() * 2 for k in ks)
    d2h = sum(hy[name].numel() * 2 for name in hy)

    def e2e_step(replay):
        with torch.cuda.stream(stream):
            for k in ks:
                x1[k].copy_(hx[k], non_blocking=True)
            if replay:
                g_step.replay()
            else:
                decode_step()
            for name in hy:
                hy[name].copy_(yproj[name], non_blocking=True)

    def e2e_time(replay):
        e2e_step(replay)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step(replay)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) * 1e3 / args.steps

    e2e_ms = e2e_time(True)
    e2e_value = step_bytes * world / (e2e_ms * 1e-3) / 1e9
    # the same without the graph: 448 pq_linear calls through ctypes per step
    # (argument checks, dispatch and launches on the host every call)
    eager_ms = e2e_time(False)
    eager_value = step_bytes * world / (eager_ms * 1e-3) / 1e9

    # ---- sampled outputs of the timed layers, checked in the CPU-baseline leg
    spot = spot_outputs(torch, pq, x1, w4, w2, stream)

    med = {k: statistics.median(v) for k, v in pair.items()}
    sustained = peak["bf16_tflops_sustained"]
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 activations; u4 / ternary codes; fp32 accumulate",
        "data": f"synthetic (seeded; {LAYERS} distinct layers, {step_bytes / 1e9:.2f} GB of packed weights)",
        "config": {"workload": WORKLOAD, "decode_M": M1, "prefill_M": MP, "layers": LAYERS,
                   "formats": ["W4A16 g128 sym", "W2A8 ternary PQ2, per-row int8 activations"],
                   "decode_dataflow": "per layer qkv (q|k|v stacked, 12288x4096) -> o -> gu (gate|up stacked, "
                                      "22016x4096) -> down, in stream order: 4 calls per layer and format",
                   "l2": f"weights per step {step_bytes / 1e9:.2f} GB > 129 MB L2 (inputs larger than L2, no flush needed)",
                   "parallelism": f"replicas x{world}"},
        "frac_of_hbm_peak": round(value / world / peak["hbm_gbs"], 4),
        "decode": {"w4a16_gemv_GBs": round(gbs_w4, 1), "w4a16_us_per_call": round(us_w4, 3),
                   "w2a8_gemv_GBs": round(gbs_w2, 1), "w2a8_us_per_call": round(us_w2, 3),
                   "calls_per_step": n4 + n2},
        "decode_per_projection": {
            "ms_per_step": round(ms_pp, 4), "GBs": round(step_bytes / (ms_pp * 1e-3) / 1e9, 1),
            "calls_per_step": len(w4) + len(w2),
            "dataflow": "per layer q|k|v -> o -> gate|up -> down, seven separate layers, independent projections "
                        "on fork/join streams"},
        "decode_paired": {
            "pairs": len(pair["step"]), "step_ms_median": round(med["step"], 4),
            "step_GBs_median": round(step_bytes / (med["step"] * 1e-3) / 1e9, 1),
            "probe_wait_ms_median": round(med["probe_wait"], 4),
            "probe_wait_GBs_median": round(step_bytes / (med["probe_wait"] * 1e-3) / 1e9, 1),
            "probe_free_ms_median": round(med["probe_free"], 4),
            "probe_free_GBs_median": round(step_bytes / (med["probe_free"] * 1e-3) / 1e9, 1),
            "step_over_probe_wait": round(med["step"] / med["probe_wait"], 3),
            "probe": "pq_probe_read over each call's prepared planes (same bytes, same launch chain): 'wait' launches "
                     "each wait for their predecessor before reading (8 CTAs/SM), 'free' ones do not (2 CTAs/SM)"},
        "prefill": {"metric": "TFLOP/s at M=2048", "w4a16_tflops": round(tf_p4, 1),
                    "w4a16_frac_of_bf16_peak": round(tf_p4 / gemm_peak, 4),
                    "w2a8_tflops": round(tf_p2, 1), "w2a8_frac_of_bf16_peak": round(tf_p2 / gemm_peak, 4),
                    "peak": gemm_peak, "peak_kind": gemm_peak_kind,
                    "w4a16_frac_of_bf16_peak_sustained": round(tf_p4 / sustained, 4)},
        "roofline": {"bound": "hbm", "kernel": "gemv_w4_m1_kernel (W4A16 decode GEMV, M=1)",
                     "achieved": round(gbs_w4, 1), "peak": peak["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gbs_w4 / peak["hbm_gbs"], 4), "traffic": read_traffic("gemv_w4_m1_kernel"),
                     "bytes_per_launch": round(bytes_w4), "peak_kind": f"hbm_gbs ({peak['source']})"},
        "roofline_w2": {"bound": "hbm", "kernel": "w2_gemv_kernel (ternary W2A8 decode GEMV, M=1, quantiser fused)",
                        "achieved": round(gbs_w2, 1), "peak": peak["hbm_gbs"], "unit": "GB/s",
                        "frac": round(gbs_w2 / peak["hbm_gbs"], 4), "traffic": read_traffic("w2_gemv_kernel"),
                        "bytes_per_launch": round(bytes_w2), "peak_kind": f"hbm_gbs ({peak['source']})"},
        "roofline_gemm": {"bound": "tensor", "kernel": "gemm_wt_kernel (W4A16 weight-stationary tcgen05 GEMM, M=2048)",
                          "achieved": round(tf_p4, 1),
                          "peak": gemm_peak, "unit": "TFLOP/s", "frac": round(tf_p4 / gemm_peak, 4),
                          "peak_kind": gemm_peak_kind, "traffic": read_traffic("gemm_wt_kernel")},
        "read_probe": probe_rates,
        "producer": producer,
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4), "path": "pq_linear via ctypes captured in a CUDA graph, pinned host buffers"},
        "e2e_eager": {"value": round(eager_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "ms_per_step": round(eager_ms, 4),
                      "path": f"{len(w4m) + len(w2m)} pq_linear ctypes calls per step, no graph, pinned host buffers"},
        "gpu_launches": args.steps * (len(w4m) + len(w2m)),
        "clocks": clk,
    }
    if rank == 0:
        # CPU-baseline leg: the oracle timed on the host cores, and the
        # oracle's values for the sampled outputs of the timed layers
        result["cpu_baseline"] = cpu_baseline()
        result["parity_spot_check"] = spot_check(spot, rank, dev)
    for h in [h for *_, h in w4 + w2]:
        pq.pq_destroy(h)
    return result


def read_probe_rates(torch, pq, dev, stream):
    """Copy-only read rate (pq_probe_read, 16-byte loads) for the decode
    layers' plane sizes: the 4096x4096 4-bit layer (8.65 MB), the 11008x4096
    one (23.2 MB) and the 27648x5120 one with zero points and act order
    (73.6 MB).  Each size is read from distinct buffers totalling at least
    4x L2, launched back to back in one graph (independent launches, and
    launches that each wait for their predecessor to finish)."""
    sink = torch.zeros(64, dtype=torch.int32, device=dev)
    big = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    big.random_(0, 256)
    out = {"kernel": "read_probe_kernel", "loads": "16-byte ld.global.nc.L1::no_allocate, every byte once"}
    for label, nb in (("8.65MB", 8650752), ("23.2MB", 23248896), ("73.6MB", 73574400)):
        nb = nb // 256 * 256
        copies = max(2, min((1 << 30) // nb, -(-4 * 129 * 10 ** 6 // nb)))
        for dep in (0, 1):
            def reads(dep=dep):
                for i in range(copies):
                    pq.pq_probe_read(big[i * nb:], nb, sink, 0, dep, stream)
            ms = time_graph(torch, capture(torch, reads, stream), 5, stream)
            us = ms * 1e3 / copies
            key = f"{label}_{'dependent' if dep else 'overlapped'}"
            out[key] = {"us_per_launch": round(us, 3), "GBs": round(nb / (us * 1e-6) / 1e9, 1)}
    del big
    torch.cuda.empty_cache()
    return out


def measure_producer(torch, pq, dev, qkv, stream, MP):
    """The fused activation producer of ternary layers (residual add, RMSNorm,
    random-sign Hadamard of 1024, int8 quantiser; K = 4096, bf16) at M = 1 and
    M = MP, and one layer's q, k, v projections (ternary 4096 x 4096, per-row
    activation scale) at M = 1 three ways: three pq_linear calls; one
    pq_quantize_act and three pq_linear_act calls; one pq_norm_quantize (which
    also does the norm) and three pq_linear_act calls."""
    K = 4096
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    gamma = (torch.randn(K, generator=g, device=dev) * 0.1).to(torch.bfloat16)
    signs = torch.where(torch.rand(K, generator=g, device=dev) < 0.5, -1, 1).to(torch.int8)
    nrm = pq.pq_norm(gamma.data_ptr(), signs.data_ptr(), 1e-6, 1, 1024)
    desc = pq.make_desc(pq.PQ_FMT_W2_PQ2, 4096, K, act_group=K, max_m=MP)
    h0 = qkv[0]
    out = {"kernel": "w2_norm_quant_kernel",
           "op": "residual add + RMSNorm (1 + gamma) + random-sign Hadamard(1024) + per-row int8 quantise, K=4096, bf16"}
    bufs = {}
    for M, reps in ((1, 50), (MP, 10)):
        h = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
        r = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
        r_out = torch.empty_like(h)
        ab = pq.pq_act_bytes(desc, M)
        act = torch.empty(ab, dtype=torch.uint8, device=dev)
        bufs[M] = (h, r, r_out, act, ab)

        def prod(h=h, r=r, r_out=r_out, act=act, ab=ab, M=M, reps=reps):
            for _ in range(reps):
                pq.pq_norm_quantize(h, r, nrm, h0, r_out, None, act, ab, M, stream)

        us = time_graph(torch, capture(torch, prod, stream), 3, stream) * 1e3 / reps
        # reads h, r (twice: the second pass is served from L2), gamma; writes
        # r_out, the codes (int8 for M <= 16, bf16 above), scales and block sums
        byts = 3 * M * K * 2 + 2 * K + (M * K if M <= 16 else 2 * M * K) + 4 * M + 4 * M * (K // 128)
        out[f"us_M{M}"] = round(us, 3)
        out[f"GBs_M{M}"] = round(byts / (us * 1e-6) / 1e9, 1)
        out[f"bytes_M{M}"] = byts
    h, r, r_out, act, ab = bufs[1]
    x = torch.randn((1, K), generator=g, device=dev).to(torch.bfloat16)
    ys = [torch.empty((1, 4096), dtype=torch.bfloat16, device=dev) for _ in qkv]
    reps = 20

    def plain():
        for _ in range(reps):
            for hh, yy in zip(qkv, ys):
                pq.pq_linear(x, hh, yy, 1, stream)

    def shared():
        for _ in range(reps):
            pq.pq_quantize_act(x, h0, act, ab, 1, stream)
            for hh, yy in zip(qkv, ys):
                pq.pq_linear_act(act, ab, hh, yy, 1, stream)

    def fused():
        for _ in range(reps):
            pq.pq_norm_quantize(h, r, nrm, h0, r_out, None, act, ab, 1, stream)
            for hh, yy in zip(qkv, ys):
                pq.pq_linear_act(act, ab, hh, yy, 1, stream)

    out["w2_qkv_M1_us"] = {name: round(time_graph(torch, capture(torch, fn, stream), 3, stream) * 1e3 / reps, 3)
                           for name, fn in (("pq_linear_x3", plain), ("quantize_act_then_linear_act_x3", shared),
                                            ("norm_quantize_then_linear_act_x3", fused))}
    return out


def run_producer(args):
    """Only the fused producer figures (one JSON line): three ternary
    4096 x 4096 layers, quick enough for a profiler capture."""
    import torch

    import bit_weight_quantized_pq_gb300 as pq
    import pq_inputs

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    pq.build()
    peak = peaks()
    stream = torch.cuda.Stream(dev)
    layers = [pq.QuantizedLinear.from_pq2(pq_inputs.device_pq2_rows(21 + i, 4096, 4096, dev), 4096,
                                          act_group=4096, max_m=PREFILL_M) for i in range(3)]
    res = measure_producer(torch, pq, dev, [ly.handle for ly in layers], stream, PREFILL_M)
    res["frac_of_hbm_peak_M2048"] = round(res[f"GBs_M{PREFILL_M}"] / peak["hbm_gbs"], 4)
    for ly in layers:
        ly.close()
    print(json.dumps({"producer": res}), flush=True)


def spot_outputs(torch, pq, x1, w4, w2, stream):
    """Re-run the last layer's down projection in both formats and keep the
    activations and a sample of the outputs on the host; the comparison with
    the oracle happens in the CPU-baseline leg (``spot_check``)."""
    import numpy as np
    out = {"layer": LAYERS - 1, "proj": len(SHAPES) - 1}
    for fmt, lst in (("w4", w4), ("w2", w2)):
        name, N, K, h = lst[-1]
        x = x1[K]
        y = torch.empty((1, N), dtype=torch.bfloat16, device=x.device)
        pq.pq_linear(x, h, y, 1, stream)
        torch.cuda.synchronize()
        cols = np.arange(0, N, 17)
        out[fmt] = {"N": N, "K": K, "cols": cols,
                    "x": x.view(torch.int16).cpu().numpy().view(np.uint16),
                    "y": y.view(torch.int16).cpu().numpy().view(np.uint16)[:, cols]}
    return out


def spot_check(spot, rank, dev):
    """Oracle values for the sampled outputs of ``spot_outputs``.  The
    weights are regenerated from their seeds (the same device generators the
    benchmark prepared them from) and copied to the host, so the check
    depends on the GPU path only through the outputs it compares."""
    import numpy as np
    import torch

    import pq_inputs
    from oracle import pq_oracle as O
    from tests.helpers import o8_error
    out = {}
    seed = 1000 * rank + 10 * spot["layer"] + spot["proj"]
    for fmt in ("w4", "w2"):
        d = spot[fmt]
        N, K, cols = d["N"], d["K"], d["cols"]
        if fmt == "w4":
            qweight, scales = pq_inputs.device_w4_frame(seed, K, N, 0.002, 0.01, dev)
            qw = qweight.cpu().numpy().view(np.uint32)
            sc = scales.view(torch.int16).cpu().numpy().view(np.uint16)
            ref = O.w4a16_linear_columns(d["x"], "bf16", qw, sc, None, None, cols)
        else:
            raw = pq_inputs.device_pq2_rows(seed + 500000, N, K, dev).cpu().numpy()
            ref = O.w2a8_linear_columns(d["x"], "bf16", raw, K, cols)
        out[fmt] = round(o8_error(d["y"], ref, "bf16"), 6)
    out["tolerance"] = 2e-3
    out["sample"] = (f"every 17th output of layer {spot['layer']}'s down projection (4096x11008) at M=1, "
                     "both formats")
    return out


# ------------------------------------------------------------------ CPU oracle

def _oracle_sample(seconds_target=10.0):
    """Oracle throughput on one 4-bit and one ternary 4096x4096 projection at
    M = 1, repeated for about `seconds_target` seconds."""
    import numpy as np
    import pq_inputs
    from oracle import pq_oracle as O
    N = K = 4096
    fr = pq_inputs.w4_frame(0, K, N, 0.002, 0.01)
    raw = pq_inputs.pq2_rows(1, N, K)
    x = pq_inputs.activations(2, 1, K, "bf16")
    nbytes = w4_bytes(N, K) + w2_bytes(N, K)
    reps, t = 0, 0.0
    t0 = time.perf_counter()
    while t < seconds_target or reps == 0:
        O.w4a16_linear(x, "bf16", fr["qweight"], fr["scales"])
        O.w2a8_linear(x, "bf16", raw, K)
        reps += 1
        t = time.perf_counter() - t0
    return {"value": round(nbytes * reps / t / 1e9, 4), "unit": UNIT, "reps": reps, "seconds": round(t, 2)}


def cpu_baseline(seconds_target=10.0):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json,sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench._oracle_sample(%r)))" % (ROOT, seconds_target))
    try:
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=600)
        d = json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # noqa: BLE001
        return {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": f"failed: {e}"}
    return {"value": d["value"], "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"W4A16 + ternary W2A8 4096x4096 projections at M=1, numpy fp64 oracle, one thread, "
                      f"{d['reps']} repetitions in {d['seconds']} s"}


# ------------------------------------------------------------------ per-config table

def table_cases():
    """One row per configuration of the workload set: the W4A16 GEMV at
    M = 1 (4096x4096, fp16), the ternary GEMV at M = 1 (three shapes),
    W4A16 with zero points and act order at K = 5120 (M = 1, 4, 16), the
    W4A16 prefill GEMM at M = 512, 2048, 3314 in both orientations, the
    ternary GEMV at M = 16 (two shapes), and MLX affine 4-bit at M = 1, 16
    and 2048 on 4096x4096 and 11008x4096."""
    cases = [dict(cfg="W4A16 GEMV 4096x4096 fp16", fmt="w4", M=1, N=4096, K=4096, act="f16")]
    for N, K in ((4096, 4096), (11008, 4096), (4096, 11008)):
        cases.append(dict(cfg="ternary W2A8 GEMV", fmt="w2", M=1, N=N, K=K, act="bf16"))
    for N in (5120, 27648):
        for M in (1, 4, 16):
            cases.append(dict(cfg="W4A16 asym + act order", fmt="w4", M=M, N=N, K=5120, act="bf16",
                              zp=True, ao="scatter"))
    for K, N in ((4096, 14336), (14336, 4096)):
        for M in (512, 2048, 3314):
            cases.append(dict(cfg="W4A16 prefill GEMM", fmt="w4", M=M, N=N, K=K, act="bf16", outliers=True))
    # ternary decode at 16 tokens (the cluster split-K decode)
    for N, K in ((4096, 4096), (11008, 4096)):
        cases.append(dict(cfg="ternary W2A8 GEMV", fmt="w2", M=16, N=N, K=K, act="bf16"))
    # MLX affine 4-bit (scale and bias per 64 inputs): decode, split-K decode, GEMM
    for N, K in ((4096, 4096), (11008, 4096)):
        for M in (1, 16, 2048):
            cases.append(dict(cfg="MLX affine 4-bit", fmt="aff", M=M, N=N, K=K, act="bf16", outliers=M > 16))
    return cases


def plane_bytes(c):
    """Prepared weight-plane bytes one call reads: codes + fp16 scales
    (+ the u8 zero plane, + the int32 act-order permutation)."""
    N, K = c["N"], c["K"]
    if c["fmt"] == "w2":
        return w2_bytes(N, K)
    if c["fmt"] == "aff":                       # codes + a 16-bit scale and bias per 64 inputs
        return N * K // 2 + N * (K // 64) * 4
    b = w4_bytes(N, K)
    if c.get("zp"):
        b += N * (K // 128)
    if c.get("ao"):
        b += K * 4
    return b


def _case_inputs(c):
    """Host inputs of a table row (seeded; the oracle leg regenerates them)."""
    import pq_inputs
    N, K = c["N"], c["K"]
    x = pq_inputs.activations(11, c["M"], K, c["act"], 0.001 if c.get("outliers") else 0.0)
    if c["fmt"] == "w2":
        return x, pq_inputs.pq2_rows(12, N, K)
    if c["fmt"] == "aff":
        return x, pq_inputs.affine4_layer(14, N, K, c["act"])
    floor = 0.001 if c.get("zp") else 0.002
    return x, pq_inputs.w4_frame(13, K, N, floor, 0.01, bool(c.get("zp")), c.get("ao"))


def _oracle_table(cases):
    """Oracle seconds per full call of each row, from a sample of about 256
    output columns (extrapolated linearly in N)."""
    import numpy as np
    from oracle import pq_oracle as O
    out = []
    for c in cases:
        x, w = _case_inputs(c)
        N = c["N"]
        cols = np.arange(0, N, max(1, N // 256))
        t0 = time.perf_counter()
        if c["fmt"] == "w2":
            O.w2a8_linear_columns(x, c["act"], w, c["K"], cols)
        elif c["fmt"] == "aff":                 # the oracle on the sampled output rows of the layer
            O.affine4_linear(x, c["act"], w["wq"][cols], w["scales"][cols], w["biases"][cols], c["act"])
        else:
            O.w4a16_linear_columns(x, c["act"], w["qweight"], w["scales"], w["zeros"], w["g_idx"], cols)
        t = time.perf_counter() - t0
        out.append({"oracle_s": t * N / len(cols), "oracle_cols": int(len(cols))})
    return out


def run_table(args):
    """Per-configuration GPU numbers (CUDA-graph replays of distinct weight
    copies totalling at least 4x L2 for the GEMVs) next to the oracle timed
    on one host core.  Prints one JSON line per row."""
    import math

    import torch

    import bit_weight_quantized_pq_gb300 as pq
    from tests.helpers import to_dev
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    pq.build()
    pq.lib()
    peak = peaks()
    rows_sel = [int(r) for r in args.rows.split(",")] if args.rows else None
    cases = [c for i, c in enumerate(table_cases()) if rows_sel is None or i in rows_sel]
    oracle = None
    if rows_sel is None:
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
        code = ("import json,sys; sys.path.insert(0, %r); import bench; "
                "print(json.dumps(bench._oracle_table(bench.table_cases())))" % ROOT)
        oracle = subprocess.Popen([sys.executable, "-c", code], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                  text=True, env=env)
    stream = torch.cuda.Stream(dev)
    rows = []
    for c in cases:
        x_h, w = _case_inputs(c)
        tdt = torch.float16 if c["act"] == "f16" else torch.bfloat16
        x = to_dev(x_h, dev, tdt)
        M, N, K = c["M"], c["N"], c["K"]
        nb = plane_bytes(c)
        decode = M <= 16
        copies = max(2, math.ceil(4 * 129e6 / nb)) if decode else 2
        with torch.cuda.stream(stream):
            if c["fmt"] == "w2":
                raw = to_dev(w, dev)
                layers = [pq.QuantizedLinear.from_pq2(raw, K, act_dtype=c["act"], act_group=K, max_m=max(M, 16),
                                                      stream=stream) for _ in range(copies)]
            elif c["fmt"] == "aff":
                wq, sc, bi = to_dev(w["wq"], dev), to_dev(w["scales"], dev), to_dev(w["biases"], dev)
                layers = [pq.QuantizedLinear.from_affine4(wq, sc, bi, act_dtype=c["act"], max_m=max(M, 16),
                                                          stream=stream) for _ in range(copies)]
            else:
                qw, sc = to_dev(w["qweight"], dev), to_dev(w["scales"], dev)
                z = None if w["zeros"] is None else to_dev(w["zeros"], dev)
                layers = [pq.QuantizedLinear.from_w4(qw, sc, z, w["g_idx"], act_dtype=c["act"], max_m=max(M, 16),
                                                     stream=stream) for _ in range(copies)]
        y = torch.empty((M, N), dtype=tdt, device=dev)

        def calls():
            for L in layers:
                L(x, out=y, stream=stream)
        g = capture(torch, calls, stream)
        reps = max(3, int(2e-2 / max(1e-6, copies * (nb / 3e12 if decode else 2.0 * M * N * K / 8e14))))
        if args.reps:
            reps = args.reps
        us = time_graph(torch, g, min(reps, 200), stream) * 1e3 / copies
        row = dict(c, us_per_call=round(us, 2), copies=copies)
        if decode:
            row["packed_GBs"] = round(nb / (us * 1e-6) / 1e9, 1)
            row["frac_of_hbm_peak"] = round(row["packed_GBs"] / peak["hbm_gbs"], 4)
        else:
            tf = 2.0 * M * N * K / (us * 1e-6) / 1e12
            row["tflops"] = round(tf, 1)
            row["frac_of_bf16_peak_sustained"] = round(tf / peak["bf16_tflops_sustained"], 4)
        rows.append(row)
        for L in layers:
            L.close()
        del layers, g
        torch.cuda.empty_cache()
    if rows_sel is not None:                 # selected rows only (profiler captures)
        for row in rows:
            print(json.dumps(row), flush=True)
        return
    # the 7B-shaped layer sweep (32 layers, both formats) at M = 1, 16, 256, 2048:
    # every projection called in order on one stream, one graph per pass
    import pq_inputs
    w4, w2, _, _, keep, workspace = build_layers(torch, pq, pq_inputs, dev, PREFILL_M, 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(21)
    for M in (1, 16, 256, PREFILL_M):
        xs = {k: torch.randn((M, k), generator=gen, device=dev).to(torch.bfloat16) for _, _, k in SHAPES}
        ys = {n: torch.empty((M, n), dtype=torch.bfloat16, device=dev) for _, n, _ in SHAPES}
        for fmt, lst in (("w4", w4), ("w2", w2)):
            def sweep():
                for _, N, K, h in lst:
                    pq.pq_linear(xs[K], h, ys[N], M, stream)
            g = capture(torch, sweep, stream)
            ms = time_graph(torch, g, 10 if M <= 16 else 3, stream)
            row = {"cfg": "7B-shaped layer sweep, 32 layers", "fmt": fmt, "M": M, "calls": len(lst),
                   "us_per_call": round(ms * 1e3 / len(lst), 2)}
            if M <= 16:
                nb = sum((w4_bytes if fmt == "w4" else w2_bytes)(N, K) for _, N, K, _ in lst)
                row["packed_GBs"] = round(nb / (ms * 1e-3) / 1e9, 1)
                row["frac_of_hbm_peak"] = round(row["packed_GBs"] / peak["hbm_gbs"], 4)
            else:
                tf = sum(flops(M, N, K) for _, N, K, _ in lst) / (ms * 1e-3) / 1e12
                row["tflops"] = round(tf, 1)
                row["frac_of_bf16_peak_sustained"] = round(tf / peak["bf16_tflops_sustained"], 4)
            print(json.dumps(row), flush=True)
            del g
    for h in [h for *_, h in w4 + w2]:
        pq.pq_destroy(h)
    del keep, workspace
    try:
        ora = json.loads(oracle.communicate(timeout=900)[0].strip().splitlines()[-1])
    except Exception:  # noqa: BLE001
        oracle.kill()
        ora = [{} for _ in rows]
    for row, o in zip(rows, ora):
        if o:
            row["oracle_ms_per_call"] = round(o["oracle_s"] * 1e3, 1)
            row["oracle"] = f"numpy fp64, one host core, {o['oracle_cols']} sampled output columns, extrapolated"
        row["peak_source"] = peak["source"]
        print(json.dumps(row), flush=True)


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle as it stands, timed on the host cores on
    a bounded sample of the workload (one projection of each shape class)."""
    if rank != 0:
        return None
    for _ in range(args.warmup):
        _oracle_sample(0.0)
    samples = [_oracle_sample(2.0) for _ in range(args.steps)]
    v = statistics.median(s["value"] for s in samples)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": {"workload": WORKLOAD, "decode_M": 1},
            "cpu_baseline": {"kind": "oracle", "cores": 1, "value": v, "unit": UNIT,
                             "sample": "W4A16 + ternary W2A8 4096x4096 at M=1 per step, numpy fp64, one thread"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    # fewer layers only for small profiler captures (7 + 7 layers of one
    # decoder block still exceed L2); the benchmark line uses all 32
    ap.add_argument("--layers", type=int, default=LAYERS)
    # per-configuration table (one JSON line per row) instead of the benchmark line
    ap.add_argument("--table", action="store_true")
    # only the fused activation producer's figures
    ap.add_argument("--producer", action="store_true")
    # --table: only these rows of table_cases() (comma-separated indices; no
    # layer sweep, no oracle leg) -- small runs for profiler captures
    ap.add_argument("--rows", default="")
    # graphs of each table row replay this many times (profiler captures: 1)
    ap.add_argument("--reps", type=int, default=0)
    # only the copy-only read probe's figures
    ap.add_argument("--probe", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    globals()["LAYERS"] = max(1, args.layers)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "ours":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.table:
        run_table(args)
        return
    if args.producer:
        run_producer(args)
        return
    if args.probe:
        import torch

        import bit_weight_quantized_pq_gb300 as pq
        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
        pq.build()
        print(json.dumps({"read_probe": read_probe_rates(torch, pq, dev, torch.cuda.Stream(dev))}), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
