#!/usr/bin/env python3
"""Benchmark of libw4 on one B300 (or N independent replicas under torchrun).

Headline: w4_linear HBM throughput in the M=1 decode regime on the Llama-3-8B
decode linears (int4, g=32, 0.1 % x10 outlier weights), one step = one pass
of M=1 through the 7 linears (q, k, v, o, gate, up, down) of all 32 blocks,
224 skinny-kernel launches replayed from one CUDA graph.  The 4.4 GB of packed
weights per step are larger than L2, so every step streams them from HBM.
value = algorithmic bytes (N*K/2 + 4*N*K/g + 2*M*K + 2*M*N per linear) / time.

The same JSON line carries the other rows of the hot path: the tcgen05
prefill GEMMs (TFLOP/s), batched decode (M = 2..32, g=64), the full 32-block
g=128 stack at M=1 and M=16, w4_quantize and w4_dequantize throughput, the
roofline of the dominant kernel, the end-to-end number through the public API
with host buffers, the CPU oracle timed on a bounded sample, and the SM clocks
sampled during the measurements.

--impl reference times the CPU oracle (the slow, plain definition of the
method) on the same workload and metric, a bounded sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "w4_linear HBM GB/s (M=1 decode) & TFLOP/s (prefill) vs roofline"
WORKLOAD = ("Llama-3-8B decode linears, M=1, int4 g=32, W~N(0,0.02) with 0.1% outliers x10, X~N(0,1) bf16; "
            "one step = q,k,v,o,gate,up,down of 32 blocks (224 linears, 4.36 GB packed)")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# --------------------------------------------------------------------------- helpers

def linear_bytes(M, N, K, g):
    """Algorithmic bytes of one w4_linear: packed codes + qparams + X + Y."""
    return N * K // 2 + 4 * N * K // g + 2 * M * K + 2 * M * N


def quantize_bytes(N, K, g, bits=4):
    return 2 * N * K + N * K * bits // 8 + 4 * N * K // g


def linear_bytes_bits(M, N, K, g, bits):
    """Algorithmic bytes of one linear on `bits`-bit codes."""
    return N * K * bits // 8 + 4 * N * K // g + 2 * M * K + 2 * M * N


def replica_gbs(bytes_per_step, steps, world, ms):
    """Whole-job GB/s of `world` replicas that each ran `steps` steps of `bytes_per_step`
    algorithmic bytes, timed as the slowest rank's `ms` (weak scaling: per-GPU work is fixed)."""
    return bytes_per_step * steps * world / (ms * 1e-3) / 1e9


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


def source_sha(paths):
    """First 16 hex digits of the sha256 of the files' contents, concatenated in order."""
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, keyed by (kernel, shape),
    valid only while the kernel source still has the hash it was captured with."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    out = {}
    if not os.path.exists(p):
        return out
    for line in open(p):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kernel, shape, src, sha, nbytes = line.split()
        paths = [os.path.join(ROOT, f) for f in src.split(",")]  # every source the kernel is built from
        if all(os.path.exists(f) for f in paths) and source_sha(paths) == sha:
            out[(kernel, shape)] = float(nbytes)
    return out


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the GPU works."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [s for s, p in zip(sm, power) if p > 0.25 * max(power)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


class Dist:
    """Rank bookkeeping; the N>1 case runs N independent replicas (no data-path collective)."""

    def __init__(self, backend):
        import torch.distributed as dist
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.dist = dist
        self.on = self.world > 1
        if self.on and not dist.is_initialized():
            dist.init_process_group(backend=backend)

    def barrier(self):
        if self.on:
            self.dist.barrier()

    def max(self, x: float, device=None) -> float:
        if not self.on:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.on and self.dist.is_initialized():
            self.dist.destroy_process_group()


# --------------------------------------------------------------------------- GPU arm

def quantize_linears(cases, device, w4, wl):
    """Quantize each case's weights on the GPU (bf16 freed right after)."""
    import torch
    out = []
    for c in cases:
        W = wl.gen_weight(c.N, c.K, c.w_seed, outliers=c.outliers, device=device)
        Wq, sc, of = w4.w4_quantize(W, c.group_size)
        del W
        out.append((Wq, sc, of))
    torch.cuda.synchronize(device)
    return out


class LinearStack:
    """Packed weights, inputs and outputs of a sequence of linears, with all X in
    one device buffer and all Y in another (one copy each way per step)."""

    def __init__(self, cases, device, w4, wl, packed=None, layout="canonical", workspace=None, bias=False):
        import torch
        self.cases = cases
        self.device = device
        self.packed = packed if packed is not None else quantize_linears(cases, device, w4, wl)
        self.layout = layout
        # decode layout: the same weights rearranged once by w4_repack (not timed)
        self.repacked = ([w4.w4_repack(Wq, sc, of, c.group_size) for c, (Wq, sc, of) in zip(cases, self.packed)]
                         if layout == "decode" else None)
        xs = sum(c.M * c.K for c in cases)
        ys = sum(c.M * c.N for c in cases)
        self.X = torch.empty(xs, dtype=torch.bfloat16, device=device)
        self.Y = torch.empty(ys, dtype=torch.bfloat16, device=device)
        self.xv, self.yv = [], []
        xo = yo = 0
        for c in cases:
            self.xv.append(self.X[xo:xo + c.M * c.K].view(c.M, c.K))
            self.yv.append(self.Y[yo:yo + c.M * c.N].view(c.M, c.N))
            self.xv[-1].copy_(wl.gen_activation(c.M, c.K, c.x_seed, device=device))
            xo += c.M * c.K
            yo += c.M * c.N
        need = max(w4.w4_linear_workspace_bytes(c.M, c.N, c.K, c.group_size) for c in cases)
        self.ws = workspace if workspace is not None else w4.Workspace(device, need)
        self.bytes = sum(linear_bytes(c.M, c.N, c.K, c.group_size) for c in cases)
        self.flops = sum(2 * c.M * c.N * c.K for c in cases)
        self.w4 = w4
        # a bf16 bias per output row of every linear (N(0, 1), seeded by the weight seed), read once
        # per call: 2N more algorithmic bytes
        self.bias = ([wl.gen_activation(1, c.N, c.w_seed + 2_000_000, device=device).view(c.N) for c in cases]
                     if bias else None)
        if bias:
            self.bytes += sum(2 * c.N for c in cases)

    def run(self):
        if self.repacked is not None:
            for x, y, rp in zip(self.xv, self.yv, self.repacked):
                self.w4.w4_linear_repacked(x, rp, out=y, workspace=self.ws)
            return
        if self.bias is not None:
            for c, x, y, (Wq, sc, of), b in zip(self.cases, self.xv, self.yv, self.packed, self.bias):
                self.w4.w4_linear_bias(x, Wq, sc, of, c.group_size, b, out=y, workspace=self.ws)
            return
        for c, x, y, (Wq, sc, of) in zip(self.cases, self.xv, self.yv, self.packed):
            self.w4.w4_linear(x, Wq, sc, of, c.group_size, out=y, workspace=self.ws)

    def capture(self, stream):
        import torch
        with torch.cuda.stream(stream):
            self.run()  # warm-up on the capture stream (kernel attributes set, nothing allocated)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                self.run()
        return g


def device_fault(w4, device):
    """None if no libw4 kernel gave up a bounded wait since the last check, else its detail
    (a timed-out kernel's output is undefined, so the numbers timed over it are not reported)."""
    try:
        w4.w4_device_fault(device)
        return None
    except w4.W4Error as e:
        return str(e)


def time_region(fn, steps, warmup, stream, dist, device):
    """W untimed steps, then K steps between events on `stream`, barrier + sync on both sides;
    returns the max over ranks of the elapsed milliseconds."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(device)
    dist.barrier()
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize(device)
    dist.barrier()
    ms = start.elapsed_time(end)
    return dist.max(ms, device)


def time_each(fn, iters, stream, flush=None):
    """Median event time of single calls, optionally flushing L2 before each."""
    import torch
    ts = []
    for _ in range(iters):
        if flush is not None:
            flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def gpu_arm(args):
    import torch
    import bit_weight_quantization_02_b300 as w4
    from bit_weight_quantization_02_b300 import workloads as wl

    dist = Dist("nccl")
    device = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(device)
    w4.load_library()
    peaks = load_peaks()
    traffic = load_traffic()
    stream = torch.cuda.Stream(device)
    clocks = ClockSampler(dist.local_rank).start()

    # ---- headline: M=1 decode through 32 blocks of Llama-3-8B linears (g=32)
    cases = [c for layer in range(args.layers) for c in wl.config2(layer)]
    stack = LinearStack(cases, device, w4, wl)
    graph = stack.capture(stream)
    with torch.cuda.stream(stream):
        ms = time_region(graph.replay, args.steps, args.warmup, stream, dist, device)
    step_ms = ms / args.steps
    value = replica_gbs(stack.bytes, args.steps, dist.world, ms)
    launches = len(cases) * args.steps
    # dominant kernel: the stream-K decode kernel is the only kernel of the step (M=1
    # always takes it), so its average launch is the step time over the launches
    achieved = stack.bytes / (step_ms * 1e-3) / 1e9
    tr = traffic.get(("stream_kernel", "llama3_8b_decode_step"))
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": (round(tr / len(cases)) if tr is not None else None),
                "algorithmic_bytes_per_launch": round(stack.bytes / len(cases)),
                "peak_source": f"{peaks['source']} copy bandwidth (MEASURED_PEAKS hbm_gbs)"
                if peaks["source"] == "measured" else "fallback 6.4 TB/s",
                "frac_of_nominal_8TBs": round(achieved / 8000.0, 4)}

    # ---- end to end through the public API with host buffers: pinned X -> device,
    # the captured linears, Y -> pinned host, every step
    xh = torch.empty(stack.X.shape, dtype=torch.bfloat16, pin_memory=True)
    xh.copy_(stack.X)
    yh = torch.empty(stack.Y.shape, dtype=torch.bfloat16, pin_memory=True)

    def e2e_step():
        stack.X.copy_(xh, non_blocking=True)
        graph.replay()
        yh.copy_(stack.Y, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_ms = time_region(e2e_step, args.steps, args.warmup, stream, dist, device)
    e2e_val = replica_gbs(stack.bytes, args.steps, dist.world, e2e_ms)

    def e2e_eager_step():
        stack.X.copy_(xh, non_blocking=True)
        stack.run()
        yh.copy_(stack.Y, non_blocking=True)

    eager_steps = max(3, args.steps // 10)
    with torch.cuda.stream(stream):
        eager_ms = time_region(e2e_eager_step, eager_steps, 2, stream, dist, device)
    faults = [f for f in [device_fault(w4, device)] if f]

    # the same step without a workspace: w4_linear's call with no workspace (the SM-pair kernel)
    nows = LinearStack(cases, device, w4, wl, packed=stack.packed, workspace=w4.Workspace(device))
    nows_graph = nows.capture(stream)
    with torch.cuda.stream(stream):
        nows_ms = time_region(nows_graph.replay, args.steps, args.warmup, stream, dist, device)
    nows_gbs = replica_gbs(nows.bytes, args.steps, dist.world, nows_ms)
    no_workspace = {"value": round(nows_gbs, 1), "unit": "GB/s", "ms_per_step": round(nows_ms / args.steps, 4),
                    "frac_of_hbm_peak": round(nows_gbs / peaks["hbm_gbs"], 4),
                    "time_vs_workspace_step": round(nows_ms / ms, 3), "kernel": "pair_kernel (w4_linear, no workspace)",
                    "how": "the headline step's 224 w4_linear calls with no workspace passed (thread-block clusters "
                           "of two SMs split K and add their partial sums in shared memory), CUDA graph"}
    del nows_graph, nows
    faults += [f for f in [device_fault(w4, device)] if f]

    e2e = {"value": round(e2e_val, 1), "unit": "GB/s", "h2d_bytes_per_step": stack.X.numel() * 2,
           "d2h_bytes_per_step": stack.Y.numel() * 2, "ms_per_step": round(e2e_ms / args.steps, 4),
           "how": "pinned X -> device, CUDA graph of the 224 w4_linear calls, Y -> pinned host, per step",
           "eager_python_calls": {"value": round(replica_gbs(stack.bytes, eager_steps, dist.world, eager_ms), 1),
                                  "ms_per_step": round(eager_ms / eager_steps, 4)}}

    rows = {}
    if not args.headline_only:
        # the same step on the same weights rearranged once by w4_repack (decode layout)
        dl = LinearStack(cases, device, w4, wl, packed=stack.packed, layout="decode")
        dl_graph = dl.capture(stream)
        with torch.cuda.stream(stream):
            dl_ms = time_region(dl_graph.replay, args.steps, args.warmup, stream, dist, device)
        dl_gbs = replica_gbs(dl.bytes, args.steps, dist.world, dl_ms)
        rows["decode_layout_step"] = {"unit": "GB/s", "value": round(dl_gbs, 1),
                                      "ms_per_step": round(dl_ms / args.steps, 4),
                                      "frac_of_hbm_peak": round(dl_gbs / peaks["hbm_gbs"], 4),
                                      "kernel": "decode_kernel (w4_linear_repacked)",
                                      "how": "the headline step with every weight in the decode layout "
                                             "(w4_repack once, untimed), CUDA graph of the 224 calls"}
        del dl_graph, dl
        # the same step with a bf16 bias on every linear (w4_linear_bias: added to the fp32 sum
        # in each kernel's epilogue, before the one rounding)
        bs = LinearStack(cases, device, w4, wl, packed=stack.packed, bias=True)
        bs_graph = bs.capture(stream)
        with torch.cuda.stream(stream):
            bs_ms = time_region(bs_graph.replay, args.steps, args.warmup, stream, dist, device)
        bs_gbs = replica_gbs(bs.bytes, args.steps, dist.world, bs_ms)
        rows["decode_step_bias"] = {"unit": "GB/s", "value": round(bs_gbs, 1),
                                    "ms_per_step": round(bs_ms / args.steps, 4),
                                    "frac_of_hbm_peak": round(bs_gbs / peaks["hbm_gbs"], 4),
                                    "time_vs_no_bias": round(bs_ms / ms, 3),
                                    "kernel": "stream_kernel (w4_linear_bias)",
                                    "how": "the headline step with a bf16 bias on each of the 224 linears "
                                           "(2N more bytes a call), CUDA graph"}
        del bs_graph, bs
        rows.update(int8_rows(args, w4, wl, device, stream, dist, peaks, cases, stack, ms))
        # the same step with the weights that share an input merged row-wise, as serving stacks
        # store them (q|k|v: 6144 x 4096, gate|up: 28672 x 4096): 4 launches per block instead of
        # 7, the same codes, scales and offsets per output row (fresh seeded weights of those shapes)
        merged = [wl.LinearCase(f"L{layer}.{n}", N, K, 32, 1, wl.weight_seed(6, layer, i), outliers=True)
                  for layer in range(args.layers)
                  for i, (n, N, K) in enumerate((("qkv", 6144, 4096), ("o", 4096, 4096),
                                                 ("gate_up", 28672, 4096), ("down", 4096, 14336)))]
        mg = LinearStack(merged, device, w4, wl)
        mg_graph = mg.capture(stream)
        with torch.cuda.stream(stream):
            mg_ms = time_region(mg_graph.replay, args.steps, args.warmup, stream, dist, device)
        mg_gbs = replica_gbs(mg.bytes, args.steps, dist.world, mg_ms)
        rows["decode_step_merged_qkv_gateup"] = {
            "unit": "GB/s", "value": round(mg_gbs, 1), "ms_per_step": round(mg_ms / args.steps, 4),
            "frac_of_hbm_peak": round(mg_gbs / peaks["hbm_gbs"], 4), "launches_per_step": len(merged),
            "kernel": "stream_kernel (w4_linear)",
            "how": "the headline step's weights with q|k|v and gate|up merged row-wise (one w4_linear per "
                   "merged matrix), CUDA graph of the 128 calls"}
        del mg_graph, mg
        rows.update(other_rows(args, w4, wl, device, stream, peaks, dist))
        faults += [f for f in [device_fault(w4, device)] if f]

    step_bytes = stack.bytes
    del graph, stack
    clk = clocks.stop()
    cpu = None
    if dist.rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample(args.cpu_seconds)

    prefill, batched = summary_rows(rows, peaks)
    if dist.rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": dist.world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded; random-init Llama-3-8B-shaped weights)",
                "config": {"workload": WORKLOAD if args.layers == 32 else f"{args.layers}-block profiling cut of: " + WORKLOAD,
                           "l2": f"inputs larger than L2 ({step_bytes / 1e9:.2f} GB of packed weights per step)",
                           "group_size": 32, "M": 1, "linears_per_step": len(cases),
                           "parallelism": "replicas" if dist.world > 1 else "single GPU"},
                "roofline": roofline, "prefill": prefill, "batched": batched, "no_workspace": no_workspace,
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
                "clocks": clk, "peaks": {k: peaks.get(k) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained",
                                                                     "source")},
                "device_fault": faults[0] if faults else None,
                "rows": rows}
        if faults:  # a kernel gave up a bounded wait: its outputs, and so these numbers, are not valid
            line["value"] = None
            line["e2e"]["value"] = None
        print(json.dumps(line), flush=True)
    dist.close()


def int8_rows(args, w4, wl, device, stream, dist, peaks, cases, stack, ws_ms):
    """The headline step on int8 activations (w4_quantize_activation_i8 + w4_linear_i8, one
    scale per tensor): with the codes made beforehand (the linear alone) and with the
    quantization inside the step (the whole dynamic path, two launches a linear); and the
    M = 2048 prefill of the gate projection (quantize, widen, tensor-core GEMM)."""
    import torch
    out = {}
    xq = [w4.w4_quantize_activation_i8(x) for x in stack.xv]
    need = max(w4.w4_linear_i8_workspace_bytes(c.M, c.N, c.K, c.group_size) for c in cases)
    ws = w4.Workspace(device, need)
    qws = w4.Workspace(device, 4096)

    def lin_only():
        for c, (q, s_), y, (Wq, sc, of) in zip(cases, xq, stack.yv, stack.packed):
            w4.w4_linear_i8(q, s_, False, Wq, sc, of, c.group_size, out=y, workspace=ws)

    def dynamic():
        for c, x, (q, s_), y, (Wq, sc, of) in zip(cases, stack.xv, xq, stack.yv, stack.packed):
            w4.w4_quantize_activation_i8(x, False, out=(q, s_), workspace=qws)
            w4.w4_linear_i8(q, s_, False, Wq, sc, of, c.group_size, out=y, workspace=ws)

    dws = w4.Workspace(device, max(w4.w4_linear_i8_dynamic_workspace_bytes(c.M, c.N, c.K, c.group_size)
                                   for c in cases))

    def fused():
        for c, x, y, (Wq, sc, of) in zip(cases, stack.xv, stack.yv, stack.packed):
            w4.w4_linear_i8_dynamic(x, Wq, sc, of, c.group_size, out=y, workspace=dws)

    act_bytes = sum(2 * c.M * c.K + c.M * c.K + 4 for c in cases)  # X read, codes written, the scale
    for name, fn, extra, launches in (("decode_step_int8_codes", lin_only, 0, 1),
                                      ("decode_step_int8_dynamic", dynamic, act_bytes, 2),
                                      ("decode_step_int8_one_call", fused, sum(2 * c.M * c.K for c in cases), 1)):
        with torch.cuda.stream(stream):
            fn()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            t = time_region(g.replay, args.steps, args.warmup, stream, dist, device)
        # the linear reads int8 codes: M K fewer bytes of X than the bf16 linear
        lin_bytes = stack.bytes - sum(c.M * c.K for c in cases)
        gbs = replica_gbs(lin_bytes + extra, args.steps, dist.world, t)
        out[name] = {"unit": "GB/s", "value": round(gbs, 1), "ms_per_step": round(t / args.steps, 4),
                     "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4), "time_vs_bf16_step": round(t / ws_ms, 3),
                     "launches_per_step": launches * len(cases),
                     "kernel": ("stream_kernel quantizing bf16 X itself (w4_linear_i8_dynamic)" if name.endswith("one_call")
                                else "stream_kernel on int8 codes (w4_linear_i8)" +
                                (" + act_rows_kernel (w4_quantize_activation_i8)" if launches == 2 else "")),
                     "how": "the headline step's 224 linears on int8 activation codes, one scale per tensor, CUDA graph" +
                            ("; each linear's activations quantized inside the step" if launches == 2 else
                             "; one call a linear: the kernel quantizes its bf16 X" if name.endswith("one_call") else
                             "; codes made before the timed region")}
        del g
    # prefill: the gate projection at M = 2048 on int8 activations, L2 flushed before each call
    M, N, K, gs = 2048, 14336, 4096, 32
    W = wl.gen_weight(N, K, seed=wl.weight_seed(4, 0, 0), outliers=False, device=device)
    Wq, sc, of = w4.w4_quantize(W, gs)
    del W
    X = wl.gen_activation(M, K, seed=wl.weight_seed(4, 0, 0) + 1, device=device)
    q, s_ = w4.w4_quantize_activation_i8(X, per_token=True)
    pws = w4.Workspace(device, w4.w4_linear_i8_workspace_bytes(M, N, K, gs))
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)

    def pre():
        w4.w4_quantize_activation_i8(X, True, out=(q, s_))
        w4.w4_linear_i8(q, s_, True, Wq, sc, of, gs, out=Y, workspace=pws)
    torch.cuda.synchronize(device)  # the inputs were made on the default stream
    with torch.cuda.stream(stream):
        pre()
        ts = time_each(pre, 10, stream, flush=lambda: flush.zero_())
    tf = 2 * M * N * K / (ts * 1e-3) / 1e12
    out["prefill_int8_dynamic"] = {"unit": "TFLOP/s", "M": M, "N": N, "K": K, "g": gs, "ms": round(ts, 4),
                                   "tflops": round(tf, 1), "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                                   "kernel": "act_rows_kernel + widen_kernel + gemm_kernel (tcgen05, bf16 operands "
                                             "holding the int8 codes exactly)",
                                   "how": "per-token int8 quantization of X, the codes widened to bf16, the "
                                          "tensor-core GEMM with the activation scale in its epilogue; L2 flushed"}
    del flush, pws, Y, q, X
    return out


def summary_rows(rows, peaks):
    """Compact prefill (TFLOP/s) and batched-decode (GB/s) results for the top of the JSON line."""
    pre = rows.get("prefill_gemm", {}).get("cases", [])
    prefill = {"unit": "TFLOP/s", "kernel": "gemm_kernel (tcgen05, persistent, stream-K tail with the default workspace)",
               "peak": peaks["bf16_tflops"],
               "peak_source": "MEASURED_PEAKS bf16_tflops (burst)", "l2": "flushed before every call",
               "cases": [{"M": c["M"], "N": c["N"], "K": c["K"], "g": 32, "tflops": c["tflops"],
                          "frac": c["frac_of_bf16_peak"]} for c in pre]} if pre else None
    b3 = [c for c in rows.get("batched_decode_g64", {}).get("cases", []) if c.get("layout", "canonical") == "canonical"]
    # with a workspace first; the no-workspace rows say so in their kernel name
    batched = {"unit": "GB/s", "peak": peaks["hbm_gbs"], "peak_source": "MEASURED_PEAKS hbm_gbs (copy)",
               "l2": "graph of calls over weight copies > 4x L2",
               "cases": [{"M": c.get("M"), "N": c.get("N"), "K": c.get("K"), "g": 64, "kernel": c.get("kernel"),
                          "gbs": c.get("gbs"), "frac": c.get("frac_of_hbm_peak")} for c in b3]} if b3 else None
    return prefill, batched


def _rotated_graph_row(c, w4, wl, device, stream, dist, peaks, layout="canonical", no_workspace=False, kernel=None):
    """Time one linear shape: a graph of back-to-back calls over weight copies totalling
    more than 4x L2 (so every call streams its weights from HBM); `layout` "decode" times
    w4_linear_repacked on w4_repack's rearrangement of the same weights."""
    import torch
    (Wq, sc, of), = quantize_linears([c], device, w4, wl)
    copies = max(2, int(4 * 126e6 // (c.N * c.K * 0.5625)) + 1)
    if layout == "decode":
        reps = [w4.w4_repack(Wq, sc, of, c.group_size) for _ in range(copies)]
    else:
        reps = [(Wq.clone(), sc.clone(), of.clone()) for _ in range(copies)]
    X = wl.gen_activation(c.M, c.K, c.x_seed, device=device)
    Y = torch.empty((c.M, c.N), dtype=torch.bfloat16, device=device)
    ws = w4.Workspace(device) if no_workspace else w4.Workspace(device).reserve_for(c.M, c.N, c.K, c.group_size)
    it = {"i": 0}

    def one():
        r = reps[it["i"] % copies]
        it["i"] += 1
        if layout == "decode":
            w4.w4_linear_repacked(X, r, out=Y, workspace=ws)
        elif kernel is not None:
            w4.w4_linear_ex(X, *r, c.group_size, kernel, out=Y, workspace=ws)
        else:
            w4.w4_linear(X, *r, c.group_size, out=Y, workspace=ws)

    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        one()
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(copies):
                one()
        t = time_region(g.replay, 20, 3, stream, dist, device) / (20 * copies)
    gbs = linear_bytes(c.M, c.N, c.K, c.group_size) / (t * 1e-3) / 1e9
    del reps, Wq, sc, of, g
    return {"M": c.M, "N": c.N, "K": c.K, "g": c.group_size, "layout": layout, "workspace": not no_workspace,
            "us": round(t * 1e3, 2),
            "gbs": round(gbs, 1),
            "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4),
            "tflops": round(2 * c.M * c.N * c.K / (t * 1e-3) / 1e12, 2)}


def _code_width_rows(w4, wl, device, stream, dist, peaks, flush, only_bits=0):
    """2- and 8-bit codes (8 bits in groups of 128, 2 bits in groups of 32) on Llama-3-8B shapes:
    quantize (L2 flushed), decode at M = 1 and 16 (graphs of back-to-back calls over weight copies
    totalling > 4x L2) and prefill at M = 2048 (L2 flushed)."""
    import torch
    cases = []
    for b, g in ((8, 128), (2, 32)):
        if only_bits and b != only_bits:
            continue
        N, K = 14336, 4096
        W = wl.gen_weight(N, K, wl.weight_seed(7, 0, b), outliers=True, device=device)
        with torch.cuda.stream(stream):
            out = w4.w4_quantize_bits(W, g, b)
            t = time_each(lambda: w4.w4_quantize_bits(W, g, b, out=out), 20, stream, flush)
        qb = quantize_bytes(N, K, g, b)
        cases.append({"bits": b, "g": g, "op": "quantize", "N": N, "K": K, "us": round(t * 1e3, 2),
                      "gbs": round(qb / (t * 1e-3) / 1e9, 1), "frac_of_hbm_peak": round(qb / (t * 1e-3) / 1e9 /
                                                                                     peaks["hbm_gbs"], 4)})
        del W, out
        for (N, K) in ((14336, 4096), (4096, 14336)):
            W = wl.gen_weight(N, K, wl.weight_seed(7, 1, b), outliers=True, device=device)
            Wq, sc, of = w4.w4_quantize_bits(W, g, b)
            del W
            per = N * K * b // 8 + 4 * N * K // g
            copies = max(2, int(4 * 126e6 // per) + 1)
            reps = [(Wq.clone(), sc.clone(), of.clone()) for _ in range(copies)]
            for M in (1, 16):
                X = wl.gen_activation(M, K, 8 + M, device=device)
                Y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
                ws = w4.Workspace(device).reserve_for(M, N, K, g)
                it = {"i": 0}

                def one():
                    r = reps[it["i"] % copies]
                    it["i"] += 1
                    w4.w4_linear_bits(X, *r, g, b, out=Y, workspace=ws)

                with torch.cuda.stream(stream):
                    graph = torch.cuda.CUDAGraph()
                    one()
                    stream.synchronize()
                    with torch.cuda.graph(graph, stream=stream):
                        for _ in range(copies):
                            one()
                    t = time_region(graph.replay, 20, 3, stream, dist, device) / (20 * copies)
                by = linear_bytes_bits(M, N, K, g, b)
                gbs = by / (t * 1e-3) / 1e9
                cases.append({"bits": b, "g": g, "op": "linear", "kernel": "batch_kernel", "M": M, "N": N, "K": K,
                              "us": round(t * 1e3, 2), "gbs": round(gbs, 1),
                              "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4)})
                del graph
            del reps
            if (N, K) == (14336, 4096):
                M = 2048
                X = wl.gen_activation(M, K, 9, device=device)
                Y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
                with torch.cuda.stream(stream):
                    for _ in range(3):
                        w4.w4_linear_bits(X, Wq, sc, of, g, b, out=Y)
                    t = time_each(lambda: w4.w4_linear_bits(X, Wq, sc, of, g, b, out=Y), 10, stream, flush)
                tf = 2 * M * N * K / (t * 1e-3) / 1e12
                cases.append({"bits": b, "g": g, "op": "linear", "kernel": "gemm_kernel", "M": M, "N": N, "K": K,
                              "ms": round(t, 4), "tflops": round(tf, 1),
                              "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4)})
            del Wq, sc, of
    return {"cases": cases, "l2": "quantize and prefill: 512 MB flush before every call; decode: graphs over weight "
                                  "copies totalling > 4x L2"}


def other_rows(args, w4, wl, device, stream, peaks, dist, only=None):
    """Prefill GEMMs, batched decode, the g=128 stack, quantize / dequantize."""
    import torch
    rows = {}
    want = (lambda name: only is None or only == name)
    flush_buf = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device)

    def flush():
        flush_buf.fill_(1)

    # prefill (tcgen05 GEMM), L2 flushed before every timed call
    pre = []
    for c in (wl.config4() if want("prefill") else []):
        (Wq, sc, of), = quantize_linears([c], device, w4, wl)
        X = wl.gen_activation(c.M, c.K, c.x_seed, device=device)
        Y = torch.empty((c.M, c.N), dtype=torch.bfloat16, device=device)
        with torch.cuda.stream(stream):
            for _ in range(3):
                w4.w4_linear(X, Wq, sc, of, c.group_size, out=Y)
            t = time_each(lambda: w4.w4_linear(X, Wq, sc, of, c.group_size, out=Y), args.prefill_iters, stream, flush)
        tf = 2 * c.M * c.N * c.K / (t * 1e-3) / 1e12
        pre.append({"M": c.M, "N": c.N, "K": c.K, "ms": round(t, 4), "tflops": round(tf, 1),
                    "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                    "hbm_gbs": round(linear_bytes(c.M, c.N, c.K, c.group_size) / (t * 1e-3) / 1e9, 1)})
        del Wq, sc, of, X, Y
    best = max(pre, key=lambda r: r["tflops"]) if pre else {"tflops": 0.0}
    rows["prefill_gemm"] = {"unit": "TFLOP/s", "cases": pre,
                            "kernel": "gemm_kernel (tcgen05, TMEM accumulators, persistent, stream-K tail)",
                            "roofline": {"bound": "tensor", "achieved": best["tflops"], "peak": peaks["bf16_tflops"],
                                         "unit": "TFLOP/s", "frac": round(best["tflops"] / peaks["bf16_tflops"], 4),
                                         "traffic": None,
                                         "peak_source": "MEASURED_PEAKS bf16_tflops (burst, kernel timed alone)"},
                            "l2": "flushed (512 MB write) before every timed call"}

    # per-linear decode: each distinct Llama-3-8B shape at M=1 g=32, weights
    # rotated through copies totalling > 4x L2, back-to-back calls in a graph
    seen, dshape = set(), []
    for c in (wl.config2(0) if want("shapes") else []):
        if (c.N, c.K) in seen:
            continue
        seen.add((c.N, c.K))
        dshape.append(_rotated_graph_row(c, w4, wl, device, stream, dist, peaks))
        dshape.append(_rotated_graph_row(c, w4, wl, device, stream, dist, peaks, layout="decode"))
    rows["decode_shapes_g32"] = {"unit": "GB/s", "cases": dshape,
                                 "l2": "graph of back-to-back calls over weight copies totalling > 4x L2"}

    # batched decode, config 3 (g=64): weights rotated through copies totalling > 4x L2
    b3 = []
    for c in (wl.config3() if want("batched") else []):
        if args.batched_m and c.M != args.batched_m:
            continue
        b3.append(_rotated_graph_row(c, w4, wl, device, stream, dist, peaks))
        # the auto choice for the canonical layout: per-warp stream-K up to 4 tokens, block-shared X beyond
        b3[-1]["kernel"] = "stream_kernel" if c.M <= 4 else "batch_kernel"
        b3.append(_rotated_graph_row(c, w4, wl, device, stream, dist, peaks, layout="decode"))
        b3[-1]["kernel"] = "decode_kernel"
        if c.N == 4096 and c.M in (2, 16, 32):  # w4_linear without a workspace: the cluster split-K kernel
            b3.append(_rotated_graph_row(c, w4, wl, device, stream, dist, peaks, no_workspace=True))
            b3[-1]["kernel"] = "skinny_kernel (no workspace)"
        if c.M in (8, 16, 32):  # the tcgen05 batched-decode kernel, on request (not the automatic choice)
            b3.append(_rotated_graph_row(c, w4, wl, device, stream, dist, peaks, kernel=w4.KERNEL_TC_DECODE))
            b3[-1]["kernel"] = "tcdec_kernel (tcgen05, W4_KERNEL_TC_DECODE)"
    rows["batched_decode_g64"] = {"unit": "GB/s", "cases": b3,
                                  "l2": "graph of back-to-back calls over weight copies totalling > 4x L2"}

    if want("widths"):
        rows["other_code_widths"] = _code_width_rows(w4, wl, device, stream, dist, peaks, flush, args.widths_bits)

    # full 32-block stack at g=128: quantize every weight (all 6.98 B bf16 weights resident,
    # the 224 quantize calls back to back between two events), then M=1 and M=16 passes
    torch.cuda.synchronize(device)
    c5 = wl.config5(1) if want("stack") else []
    t0 = time.perf_counter()
    Ws = [wl.gen_weight(c.N, c.K, c.w_seed, device=device) for c in c5]
    packed = [(torch.empty((c.N, c.K // 2), dtype=torch.uint8, device=device),
               torch.empty((c.N, c.K // c.group_size), dtype=torch.bfloat16, device=device),
               torch.empty((c.N, c.K // c.group_size), dtype=torch.bfloat16, device=device)) for c in c5]
    qbytes = sum(quantize_bytes(c.N, c.K, c.group_size) for c in c5)

    def quantize_all():
        for c, W, out in zip(c5, Ws, packed):
            w4.w4_quantize(W, c.group_size, out=out)

    q_ms = q_eager_ms = 0.0
    if c5:
        with torch.cuda.stream(stream):
            q_eager_ms = time_region(quantize_all, 3, 3, stream, dist, device) / 3
            quantize_all()  # warm (capture-time checks need no CUDA call)
            stream.synchronize()
            qg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(qg, stream=stream):
                quantize_all()
            q_ms = time_region(qg.replay, 3, 3, stream, dist, device) / 3
            del qg
    del Ws
    setup_s = time.perf_counter() - t0
    stack_rows = {}
    if c5:
        stack_rows["quantize"] = {"weights": wl.config5_weight_count(), "ms": round(q_ms, 3),
                                  "gbs": round(qbytes / (q_ms * 1e-3) / 1e9, 1),
                                  "frac_of_hbm_peak": round(qbytes / (q_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                                  "algorithmic_bytes": qbytes, "setup_s": round(setup_s, 1),
                                  "how": "the 224 w4_quantize calls of the stack (13.96 GB of bf16 weights "
                                         "resident) in a CUDA graph, mean of 3 timed replays after 3 warm-up ones",
                                  "eager_python_calls": {"ms": round(q_eager_ms, 3),
                                                         "gbs": round(qbytes / (q_eager_ms * 1e-3) / 1e9, 1)}}
    for M, layout in (((1, "canonical"), (16, "canonical"), (1, "decode"), (16, "decode")) if c5 else ()):
        cases = wl.config5(M)
        st = LinearStack(cases, device, w4, wl, packed=packed, layout=layout)
        g = st.capture(stream)
        with torch.cuda.stream(stream):
            t = time_region(g.replay, 10, 3, stream, dist, device) / 10
        stack_rows[f"M{M}" if layout == "canonical" else f"M{M}_decode_layout"] = {
            "ms": round(t, 4), "gbs": round(st.bytes / (t * 1e-3) / 1e9, 1),
            "frac_of_hbm_peak": round(st.bytes / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "algorithmic_bytes": st.bytes}
        del g, st
    rows["llama3_8b_stack_g128"] = stack_rows
    del packed

    # dequantize throughput on the gate/up shape, L2 flushed
    if want("dequant"):
        c = wl.config2()[4]
        (Wq, sc, of), = quantize_linears([c], device, w4, wl)
        out = torch.empty((c.N, c.K), dtype=torch.bfloat16, device=device)
        with torch.cuda.stream(stream):
            t = time_each(lambda: w4.w4_dequantize(Wq, sc, of, c.group_size, out=out), 20, stream, flush)
        db = c.N * c.K // 2 + 4 * c.N * c.K // c.group_size + 2 * c.N * c.K
        rows["dequantize"] = {"N": c.N, "K": c.K, "g": c.group_size, "us": round(t * 1e3, 2),
                              "gbs": round(db / (t * 1e-3) / 1e9, 1),
                              "frac_of_hbm_peak": round(db / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
        del Wq, sc, of, out
    # 4-bit quantize throughput on the gate/up shape at every group size: back-to-back calls over
    # weight copies that together exceed L2 (single calls are too short for the event clock)
    if want("quantize"):
        c = wl.config2()[4]
        copies = max(1, args.quant_copies)
        Ws = [wl.gen_weight(c.N, c.K, seed=c.w_seed + i, outliers=c.outliers, device=device) for i in range(copies)]
        qcases = []
        for g in (32, 64, 128):
            outs = [w4.w4_quantize(W, g) for W in Ws]
            torch.cuda.synchronize(device)  # the copies and outputs were made on the default stream
            with torch.cuda.stream(stream):
                for W, o in zip(Ws, outs):
                    w4.w4_quantize(W, g, out=o)
                t = time_each(lambda: [w4.w4_quantize(W, g, out=o) for W, o in zip(Ws, outs)], 5, stream) / copies
            qb = 2 * c.N * c.K + c.N * c.K // 2 + 4 * c.N * c.K // g
            qcases.append({"g": g, "us": round(t * 1e3, 2), "gbs": round(qb / (t * 1e-3) / 1e9, 1),
                           "frac_of_hbm_peak": round(qb / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)})
            del outs
        rows["quantize"] = {"N": c.N, "K": c.K, "bits": 4, "copies": copies, "cases": qcases,
                            "l2": f"{copies} weight copies of {2 * c.N * c.K / 1e6:.0f} MB quantized back to back"}
        del Ws
    del flush_buf
    return rows


# --------------------------------------------------------------------------- CPU oracle

def _oracle_decode_inputs(cases):
    import numpy as np
    import oracle
    from bit_weight_quantization_02_b300 import workloads as wl

    def bits(t):
        return t.contiguous().view(__import__("torch").int16).numpy().view(np.uint16)

    prepared = []
    for c in cases:
        W = bits(wl.gen_weight(c.N, c.K, c.w_seed, outliers=c.outliers))
        prepared.append((c, bits(wl.gen_activation(c.M, c.K, c.x_seed)), oracle.ref_quantize(W, c.group_size)))
    return prepared


def cpu_baseline_sample(seconds):
    """The oracle, as it stands (plain C, fp64 accumulation), on the host's cores: the headline
    metric on one block's 7 decode linears, single-threaded and on every core (OpenMP over
    output rows; the results do not depend on the thread count), w4_quantize's work on the
    gate matrix, and a bounded sample of every config with the extrapolations labelled."""
    import numpy as np
    import torch
    import oracle
    from bit_weight_quantization_02_b300 import workloads as wl

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    cores = oracle.set_threads(0)
    prepared = _oracle_decode_inputs(wl.config2(0))

    def linear_pass_rate(threads, budget):
        oracle.set_threads(threads)
        nbytes, el, passes = 0, 0.0, 0
        while el < budget or passes == 0:
            for c, X, (Wq, sc, of) in prepared:
                t = time.perf_counter()
                oracle.ref_linear(X, Wq, sc, of, c.group_size)
                el += time.perf_counter() - t
                nbytes += linear_bytes(c.M, c.N, c.K, c.group_size)
            passes += 1
        return nbytes / el / 1e9, passes, el

    single, p1, t1 = linear_pass_rate(1, 0.35 * seconds)
    multi, pn, tn = linear_pass_rate(0, 0.1 * seconds)

    def quant_rate(W, g, threads):
        oracle.set_threads(threads)
        t = time.perf_counter()
        oracle.ref_quantize(W, g)
        return time.perf_counter() - t

    gate = wl.config2()[4]
    Wg = bits(wl.gen_weight(gate.N, gate.K, gate.w_seed, outliers=True))
    qb = quantize_bytes(gate.N, gate.K, 32)
    q1, qn = quant_rate(Wg, 32, 1), quant_rate(Wg, 32, 0)
    del Wg

    # every config, on every core (one sample each; scaled where noted)
    oracle.set_threads(0)
    per = {}

    def lin_time(c, M=None, rows=None):
        W = bits(wl.gen_weight(c.N, c.K, c.w_seed, outliers=c.outliers))
        t = time.perf_counter()
        q = oracle.ref_quantize(W, c.group_size)
        tq = time.perf_counter() - t
        X = bits(wl.gen_activation(M or c.M, c.K, c.x_seed))
        if rows is not None:
            X = X[:rows]
        t = time.perf_counter()
        oracle.ref_linear(X, *q, c.group_size)
        return tq, time.perf_counter() - t

    c1 = wl.config1()[0]
    tq, tl = lin_time(c1)
    per["config1"] = {"quantize_ms": round(tq * 1e3, 3), "linear_ms": round(tl * 1e3, 3), "scaled": False}
    per["config2"] = {"linear_gbs": round(multi, 4), "quantize_gbs_gate": round(qb / qn / 1e9, 4), "scaled": False,
                      "note": "one block's 7 linears are the whole config"}
    down3 = [c for c in wl.config3() if c.N == 4096 and c.M in (2, 32)]
    c3 = {}
    for c in down3:
        tq, tl = lin_time(c)
        c3[f"M{c.M}"] = {"quantize_ms": round(tq * 1e3, 1), "linear_ms": round(tl * 1e3, 1)}
    per["config3_down_g64"] = dict(c3, scaled=False, note="the other M and the up shape scale with M*N*K")
    c4 = wl.config4()[0]
    tq, tl = lin_time(c4, rows=64)
    per["config4_gate_g32"] = {"quantize_ms": round(tq * 1e3, 1), "linear_ms_64_tokens": round(tl * 1e3, 1),
                               "linear_s_extrapolated_M2048": round(tl * 2048 / 64, 1),
                               "linear_s_extrapolated_M8192": round(tl * 8192 / 64, 1), "scaled": True,
                               "note": "64 of the tokens timed; the full M extrapolated linearly (labelled)"}
    c5 = wl.config5(1)[:7]  # one block at g=128
    tq5 = tl5 = 0.0
    for c in c5:
        a, b = lin_time(c)
        tq5 += a
        tl5 += b
    per["config5_g128"] = {"quantize_s_one_block": round(tq5, 2), "linear_M1_s_one_block": round(tl5, 2),
                           "quantize_s_extrapolated_32_blocks": round(32 * tq5, 1),
                           "linear_M1_s_extrapolated_32_blocks": round(32 * tl5, 1), "scaled": True,
                           "note": "one of the 32 blocks timed, the stack extrapolated x32 (labelled)"}
    oracle.set_threads(1)
    return {"value": round(multi, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{pn} pass(es) of the 7 M=1 g=32 decode linears of one Llama-3-8B block on {cores} "
                      f"threads ({tn:.1f} s; plain C, fp64 accumulation, OpenMP over output rows)",
            "single_thread": {"value": round(single, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"{p1} pass(es) of the same 7 linears ({t1:.1f} s)"},
            "quantize": {"unit": "GB/s", "shape": [gate.N, gate.K], "group_size": 32,
                         "single_thread": round(qb / q1 / 1e9, 4), "all_cores": round(qb / qn / 1e9, 4),
                         "cores": cores},
            "per_config": per, "host_cores_available": os.cpu_count()}


def reference_arm(args):
    """The CPU oracle on the headline workload: one step = one linear of the 224 (the 7
    shapes in turn), timed on the host; rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    from bit_weight_quantization_02_b300 import workloads as wl
    prepared = _oracle_decode_inputs(wl.config2(0))
    cores = oracle.set_threads(0)  # every host core (OpenMP over output rows)

    def step(i):
        c, X, (Wq, sc, of) = prepared[i % len(prepared)]
        oracle.ref_linear(X, Wq, sc, of, c.group_size)
        return linear_bytes(c.M, c.N, c.K, c.group_size)

    for i in range(args.warmup):
        step(i)
    nbytes = 0
    t = time.perf_counter()
    for i in range(args.steps):
        nbytes += step(i)
    el = time.perf_counter() - t
    value = nbytes / el / 1e9
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; random-init Llama-3-8B-shaped weights)",
            "config": {"workload": WORKLOAD, "group_size": 32, "M": 1},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": "one of the 7 decode linears of a block per step, in turn "
                                       f"(C oracle on {cores} threads: dequantize + fp64 dot products)"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- main

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["libw4", "reference"], default="libw4")
    ap.add_argument("--headline-only", action="store_true", help="skip the secondary rows")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--prefill-iters", type=int, default=10)
    ap.add_argument("--section", choices=["all", "prefill", "shapes", "batched", "widths", "stack", "dequant", "quantize"],
                    default="all",
                    help="all = the benchmark; the others run one secondary row alone (for profiling) and print it")
    ap.add_argument("--batched-m", type=int, default=0,
                    help="with --section batched: only the cases with this many tokens (for profiling)")
    ap.add_argument("--widths-bits", type=int, default=0, choices=[0, 2, 8],
                    help="with --section widths: only this code width (for profiling)")
    ap.add_argument("--quant-copies", type=int, default=8,
                    help="with --section quantize: weight copies quantized back to back (fewer only for profiling)")
    ap.add_argument("--layers", type=int, default=32,
                    help="Llama-3-8B blocks in the headline step (32 = the whole model; fewer only for profiling)")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be at least 3")
    return a


def section_only(args):
    import torch
    import bit_weight_quantization_02_b300 as w4
    from bit_weight_quantization_02_b300 import workloads as wl
    dist = Dist("nccl")
    device = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(device)
    w4.load_library()
    rows = other_rows(args, w4, wl, device, torch.cuda.Stream(device), load_peaks(), dist, only=args.section)
    if dist.rank == 0:
        print(json.dumps({"section": args.section, "rows": rows}), flush=True)
    dist.close()


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        reference_arm(args)
    elif args.section != "all":
        section_only(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
