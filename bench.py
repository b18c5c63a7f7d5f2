#!/usr/bin/env python3
"""Throughput of the BitNet b1.58 W2A8 path on B300.

Default line (N=1): the 100B-class layer stream, the largest configuration
that fits one GPU: 30 distinct BitLinear layers of 28672 x 8192 ternary
weights (58.7 MB of packed 2-bit codes each, 1.76 GB per pass, 14x the L2),
bf16 activations quantised per token inside the streaming kernel.  One pass
= one token through the 30 layers; one step = a decode of `--tokens` tokens
(192 by default, so that 20 timed steps last about a second).  `value` is
packed-weight GB/s.  The same line carries a `prefill` object: the prefill
GEMM workload (M = 2048 tokens against 6912 x 2560 and 2560 x 6912), in
TOPS, timed in the same run.  Weights are packed once before timing (the
offline step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl reference]

Prints one JSON line (rank 0).  Under torchrun the ranks split every matrix
by output rows (each rank streams its N / world rows of every layer, x is
replicated, each rank keeps its slice of y: no collective on the data path);
`--replicas` runs independent copies of the whole stack instead.
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
sys.path.insert(0, ROOT)

METRIC = "W2A8 GEMV packed-weight GB/s (% of HBM peak); prefill GEMM int8 TOPS (% peak)"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0

# DRAM bytes (read + write) per launch of the dominant kernel from one ncu
# capture of the current kernel version, keyed by the step's shape; a step of
# another shape, or a kernel changed since its capture, reports null.  The
# last capture of the 28672 x 8192 launch (58.797 MB, the algorithmic bytes
# within 0.1 %: profiles/gemv_ldg_kernel_100b_stream_m1.md) predates the
# kernel's 32-bit row-range arithmetic, so that shape has no entry.
MEASURED_TRAFFIC = {}

# Output rows of each prefill matrix the CPU oracle computes per sample pass
# (all 2048 tokens, the whole K), to keep its timing bounded.
PREFILL_ORACLE_ROWS = 32


L2_BYTES = 126e6  # B300 L2


def default_layers(workload):
    """Copies in the stack: 30 layers for the model-shaped stacks; for the
    single-matrix workloads enough distinct copies that one step streams
    three times the L2 (so every timed step reads its weights from HBM)."""
    from ternary_weight_05_b300 import synth

    if workload in ("gateup-sweep", "bitlinear-1024"):
        L = synth.workload(workload).layers[0]
        return max(30, -(-int(3 * L2_BYTES) // (L.N * L.K // 4)))
    return 30


def l2_note(wbytes):
    """How the timed steps meet the L2 rule, stated from the stack's size."""
    if wbytes > L2_BYTES:
        return "inputs larger than L2 (packed stack %.0f MB > 126 MB L2)" % (wbytes / 1e6)
    return ("L2-resident: packed stack %.1f MB fits the 126 MB L2, an L2-hot figure (--layers grows it)"
            % (wbytes / 1e6))


def metric_unit(workload):
    """(unit, divisor of the per-second amount) of the metric for a workload."""
    return ("TOPS", 1e12) if workload == "prefill-2048" else ("GB/s", 1e9)


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="100b-stream",
                    choices=["2b-decode", "100b-stream", "gateup-sweep", "prefill-2048", "bitlinear-1024",
                             "ffn-2b-decode"])
    ap.add_argument("--layers", type=int, default=None,
                    help="matrices (or layers) in the stack; default: 30, or for the single-matrix workloads "
                         "enough copies to hold 3x the L2")
    ap.add_argument("--M", type=int, default=None, help="tokens (decode workloads)")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--unfused", action="store_true",
                    help="decode step as quant_act + w2a8_gemv (two calls) instead of the fused bitlinear call")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=None,
                    help="reference arm: seconds of oracle work per step (default: 150 s over warm-up and "
                         "steps, 1 to 20 s each)")
    ap.add_argument("--group", type=int, default=0,
                    help="group-wise weight scales: G consecutive weights of a row per scale (0: one beta per matrix)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="decode workloads: tokens per step, each one pass over the stack (default: 192 for "
                         "100b-stream, so that 20 steps last about a second; 1 otherwise)")
    ap.add_argument("--no-prefill", action="store_true",
                    help="100b-stream: leave out the prefill GEMM object of the line")
    ap.add_argument("--replicas", action="store_true",
                    help="N > 1: every rank runs the whole stack (independent replicas) instead of its rows")
    args = ap.parse_args(argv)
    if args.layers is None:
        args.layers = default_layers(args.workload)
    if args.tokens is None:
        args.tokens = 192 if args.workload == "100b-stream" else 1
    return args


def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1400.0, "fallback"


# ---------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during timing."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ workloads --

def decode_layers(args):
    from ternary_weight_05_b300 import synth

    if args.workload == "2b-decode":
        wl = synth.workload("2b-decode")
        layers = [(L, rep) for rep in range(args.layers) for L in wl.layers]
        M = args.M or 1
    elif args.workload == "100b-stream":
        wl = synth.workload("100b-stream")
        layers = [(L, 0) for L in wl.layers[: args.layers]]
        M = args.M or 1
    elif args.workload == "gateup-sweep":
        wl = synth.workload("gateup-sweep")
        layers = [(wl.layers[0], r) for r in range(max(1, args.layers))]
        M = args.M or 1
    elif args.workload == "bitlinear-1024":
        wl = synth.workload("bitlinear-1024")
        layers = [(wl.layers[0], r) for r in range(max(1, args.layers))]
        M = 1
    else:
        raise ValueError(args.workload)
    return wl, layers, M


def build_stack(args, dev, rank, world=1):
    """Packs every weight matrix on the device (offline step, not timed).
    With world > 1 (row split) each rank keeps the packed rows of its range
    of every matrix and computes that slice of y."""
    import torch

    import ternary_weight_05_b300 as tw
    from ternary_weight_05_b300 import shard, synth

    wl, layers, M = decode_layers(args)
    split = world > 1 and not args.replicas
    stack = []
    for L, rep in layers:
        W = synth.weights_torch(L.N, L.K, L.w_dist, L.w_scale, L.w_seed + 1000 * rep, dev)
        if args.group:
            packed, beta, _ = tw.pack_weights_grouped(W, args.group)  # beta: [N, K/G] group scales
        else:
            packed, beta, _ = tw.pack_weights(W)
        del W
        r0, r1 = shard.row_bounds(L.N, world, rank) if split else (0, L.N)
        if split:
            packed = shard.packed_rows(packed, L.K, r0, r1).clone()
            if args.group:
                beta = beta[r0:r1].clone()
        # the activations: the same on every rank when the rows are split,
        # an independent token stream per replica otherwise
        xs = L.x_seed + 1000 * rep + (0 if split else 7919 * rank)
        x = synth.acts_torch(M, L.K, L.x_dist, xs, dev, outlier_p=L.outlier_p)
        if not L.x_bf16:
            x = x.float()
        n = r1 - r0
        stack.append(dict(L=L, n=n, r0=r0, packed=packed, beta=beta, x=x, M=M,
                          xq=torch.empty((M, L.K), dtype=torch.int8, device=dev),
                          s=torch.empty(M, dtype=torch.float32, device=dev),
                          y=torch.empty((M, n), dtype=torch.float32, device=dev)))
    torch.cuda.synchronize(dev)
    return wl, stack, M


def decode_layer_fn(ws, fused, G):
    """One BitLinear of a decode stack entry as the benchmark runs it: the
    fused call (quantisation inside the streaming kernel), or quant_act and
    the matmul (`quant` False: the matmul alone)."""
    import ternary_weight_05_b300 as tw

    def layer(e, quant):
        L, n = e["L"], e["n"]
        if fused and G:
            tw.bitlinear_grouped(e["x"], e["packed"], e["beta"], n, L.K, G, out=e["y"], workspace=ws)
        elif fused:
            tw.bitlinear(e["x"], e["packed"], e["beta"], n, L.K, out=e["y"], workspace=ws)
        else:
            if quant:
                tw.quant_act(e["x"], out=(e["xq"], e["s"]))
            if G:
                tw.w2a8_grouped(e["xq"], e["s"], e["packed"], e["beta"], n, L.K, G, out=e["y"])
            else:
                tw.w2a8_gemv(e["xq"], e["s"], e["packed"], e["beta"], n, L.K, out=e["y"], workspace=ws)

    return layer


def passes_per_graph(tokens):
    """Passes over the stack captured in one graph: a step's passes are then
    tokens / ppg replays of it."""
    return max(d for d in (16, 8, 4, 2, 1) if tokens % d == 0)


def capture_passes(stack, ws, fused, G, ppg, stream):
    """The benchmark's CUDA graph: ppg passes over the stack's BitLinears
    (launched with the calling thread's PDL setting), captured on `stream`."""
    import torch

    layer = decode_layer_fn(ws, fused, G)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(ppg):
            for e in stack:
                if e["n"] > 0:
                    layer(e, True)
    return graph


def max_over_ranks(values, device):
    """Element-wise maximum over the ranks of per-rank floats (the slowest
    rank's times); the values themselves on one rank."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def init_dist():
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    return world, rank, dev


def run_native(args):
    import torch
    import torch.distributed as dist

    import ternary_weight_05_b300 as tw

    world, rank, dev = init_dist()
    hbm_peak, bf16_peak, bf16_sust, peak_src = load_peaks()
    if args.workload == "prefill-2048":
        return run_prefill(args, dev, rank, world, bf16_peak, peak_src)
    if args.workload == "ffn-2b-decode":
        return run_ffn(args, dev, rank, world, hbm_peak, peak_src)

    wl, stack, M = build_stack(args, dev, rank, world)
    split = world > 1 and not args.replicas
    fused = not args.unfused
    G = args.group
    T = args.tokens
    max_ws = max(max(tw.gemv_workspace_bytes(M, max(e["n"], 1), e["L"].K),
                     tw.bitlinear_workspace_bytes(M, max(e["n"], 1), e["L"].K)) for e in stack)
    ws = torch.zeros(max_ws, dtype=torch.uint8, device=dev)
    # weight bytes this rank streams per pass: packed codes (+ fp32 group scales)
    wbytes = sum(e["n"] * e["L"].K // 4 + (4 * e["n"] * (e["L"].K // G) if G else 0) for e in stack)
    # the whole job's per pass: every rank's rows (split) or every replica's stack
    job_bytes = (sum(e["L"].N * e["L"].K // 4 + (4 * e["L"].N * (e["L"].K // G) if G else 0) for e in stack)
                 * (1 if split else world))
    xes = stack[0]["x"].element_size()
    if fused:
        # fused BitLinear kernel: weights + x (bf16/fp32) + w_scale + y
        gemv_bytes = wbytes + sum(xes * M * e["L"].K + (0 if G else 4) + 4 * M * e["n"] for e in stack)
    else:
        # GEMV: weights + x_q + scales + w_scale + y
        gemv_bytes = wbytes + sum(M * e["L"].K + 4 * M + (0 if G else 4) + 4 * M * e["n"] for e in stack)
    active = [e for e in stack if e["n"] > 0]
    layer = decode_layer_fn(ws, fused, G)

    def one_pass():
        for e in active:
            layer(e, True)

    ppg = passes_per_graph(T)

    tw.set_pdl(not args.no_pdl)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        one_pass()
        torch.cuda.synchronize(dev)
        graph = None if args.no_graph else capture_passes(stack, ws, fused, G, ppg, stream)

        def step():
            if graph is not None:
                for _ in range(T // ppg):
                    graph.replay()
            else:
                for _ in range(T):
                    one_pass()

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        clocks = ClockSampler(dev.index or 0)
        clocks.start()
        time.sleep(0.3)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms_total = e0.elapsed_time(e1)
        passes = args.steps * T

        if fused:
            # the fused step is nothing but the GEMV kernel launches: their
            # duration is the timed region's
            gemv_ms, n_meas = ms_total, passes
        else:
            # the GEMV launches alone: a graph of the stack's GEMV calls (same
            # inputs, same launch configuration), replayed between two events
            gemv_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gemv_graph, stream=stream):
                for e in active:
                    layer(e, False)
            for _ in range(2):
                gemv_graph.replay()
            n_meas = max(3, args.steps)
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            for _ in range(n_meas):
                gemv_graph.replay()
            g1.record(stream)
            torch.cuda.synchronize(dev)
            gemv_ms = g0.elapsed_time(g1)
        gemv_launches = n_meas * len(active)
        clk = clocks.stop()

        # end to end through the public API: per pass, the layers' activations
        # from pinned host memory in one copy, one bitlinear call per layer
        # (PDL on, as a user enables it), every output back to pinned host
        # memory in one copy.  Two sets of buffers, the copies on their own
        # streams ordered by events: a pass's readback runs while the next
        # pass computes, as a serving loop pipelines its tokens.
        xsz = [e["x"].numel() for e in active]
        ysz = [e["y"].numel() for e in active]
        hx = torch.cat([e["x"].reshape(-1) for e in active]).cpu().pin_memory()
        hy = [torch.empty(sum(ysz), dtype=torch.float32).pin_memory() for _ in range(2)]
        dx = [torch.empty_like(hx, device=dev) for _ in range(2)]
        dy = [torch.empty(sum(ysz), dtype=torch.float32, device=dev) for _ in range(2)]
        xv, yv = [[], []], [[], []]
        for b in range(2):
            ox, oy = 0, 0
            for e, nx, ny in zip(active, xsz, ysz):
                xv[b].append(dx[b][ox:ox + nx].view(e["x"].shape))
                yv[b].append(dy[b][oy:oy + ny].view(e["y"].shape))
                ox += nx
                oy += ny
        h2d = hx.numel() * hx.element_size()
        d2h = hy[0].numel() * hy[0].element_size()
        h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        x_ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]  # the pass's kernels: x read, y written
        y_free = [torch.cuda.Event() for _ in range(2)]
        n_pass = [0]

        def e2e_pass():
            b = n_pass[0] % 2
            if n_pass[0] >= 2:  # buffer set b was last used two passes ago
                h2d_stream.wait_event(done[b])
                stream.wait_event(y_free[b])
            with torch.cuda.stream(h2d_stream):
                dx[b].copy_(hx, non_blocking=True)
                x_ready[b].record(h2d_stream)
            stream.wait_event(x_ready[b])
            for e, xd, yd in zip(active, xv[b], yv[b]):
                if G:
                    tw.bitlinear_grouped(xd, e["packed"], e["beta"], e["n"], e["L"].K, G, out=yd, workspace=ws)
                else:
                    tw.bitlinear(xd, e["packed"], e["beta"], e["n"], e["L"].K, out=yd, workspace=ws)
            done[b].record(stream)
            d2h_stream.wait_event(done[b])
            with torch.cuda.stream(d2h_stream):
                hy[b].copy_(dy[b], non_blocking=True)
                y_free[b].record(d2h_stream)
            n_pass[0] += 1

        for _ in range(2):
            e2e_pass()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(args.steps * T):
            e2e_pass()
        torch.cuda.synchronize(dev)
        e2e_s = time.perf_counter() - t0
    tw.check_device_error(stream)
    tw.set_pdl(False)

    ms_step = ms_total / args.steps
    if world > 1:  # max over ranks
        ms_step, e2e_s = max_over_ranks([ms_step, e2e_s], dev)
    value = job_bytes * T / (ms_step * 1e-3) / 1e9
    e2e_val = job_bytes * T * args.steps / e2e_s / 1e9
    achieved = gemv_bytes * n_meas / (gemv_ms * 1e-3) / 1e9
    # kernels per BitLinear: fused M <= 2: 1; fused M >= 3: prep + tensor-core GEMV;
    # unfused: quant_act (+ prep for M >= 3) + GEMV
    if G:
        # fused M <= 2: one streaming kernel; M >= 3 (fused or not): the prep
        # kernel + the grouped tensor-core GEMV (64 tokens per chunk)
        per_layer = 1 if (fused and M <= 2) else 2
        kname = ("gemv_ldg_kernel grouped form" if M <= 2 else "gemv_mma_grouped_kernel (+prep)") + \
            (" (fused quant)" if fused else "")
    else:
        per_layer = (1 if M <= 2 else 2) if fused else (2 if M <= 2 else 3)
        kname = ("gemv_ldg_kernel" if M <= 2 else "gemv_mma_kernel (+prep)") + (" (fused quant)" if fused else "")
    if split:
        parallelism = f"rows split over {world} ranks (each streams N/{world} rows of every layer; x replicated, " \
                      "y left sharded: no collective)"
    else:
        parallelism = f"replicas x{world}"
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "strong" if split else "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic (seeded, weights and activations drawn on device)",
        "config": {"workload": f"{wl.name}: {wl.description}", "layers_in_stack": len(stack), "M": M,
                   "tokens_per_step": T,
                   "step": f"{T} pass(es) over the stack, one token each; "
                           + ("fused bitlinear" if fused else "quant_act + w2a8_gemv") + " per layer"
                           + (f" with group-wise scales, G={G} (weight bytes include the fp32 scales)" if G else ""),
                   "packed_weight_bytes_per_pass": job_bytes, "graph": not args.no_graph,
                   "passes_per_graph": ppg if not args.no_graph else None, "pdl": not args.no_pdl,
                   "l2": l2_note(wbytes),
                   "parallelism": parallelism},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4),
                     "traffic": MEASURED_TRAFFIC.get((args.workload, M, fused, G)) if not split else None,
                     "algorithmic_bytes_per_launch": round(gemv_bytes / len(active)),
                     "kernel": kname, "peak_source": peak_src + " HBM copy",
                     "launches_timed": gemv_launches, "avg_launch_us": round(1e3 * gemv_ms / gemv_launches, 3)},
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d * T,
                "d2h_bytes_per_step": d2h * T},
        "gpu_launches": per_layer * len(active) * T * args.steps,
        "clocks": clk,
    }
    if args.workload == "100b-stream" and not args.no_prefill:
        # the other half of the metric, in the same run: the prefill GEMM
        line["prefill"] = measure_prefill(args, dev, rank, world, bf16_peak, peak_src, sub=True)
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(args)
        if "prefill" in line:
            line["prefill"]["cpu_baseline"] = cpu_baseline(args, workload="prefill-2048",
                                                           seconds=args.cpu_seconds / 2, one_thread=False)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def graph_of(fn, stream):
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def time_replays(graph, n, stream):
    import torch

    for _ in range(2):
        graph.replay()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def run_ffn(args, dev, rank, world, hbm_peak, peak_src):
    """Feed-forward decode: per layer silu(gate(h)) * up(h) from the fused
    gate+up matrix (one call, one streaming kernel for M <= 2), then the down
    BitLinear on that product.  Every layer has its own weights and h."""
    import torch
    import torch.distributed as dist

    import ternary_weight_05_b300 as tw
    from ternary_weight_05_b300 import synth

    wl = synth.workload("ffn-2b-decode")
    gu, dn = wl.layers
    I, D = gu.N // 2, gu.K
    M = args.M or 1
    stack = []
    for r in range(args.layers):
        W = synth.weights_torch(gu.N, gu.K, gu.w_dist, gu.w_scale, gu.w_seed + 1000 * r, dev)
        pgu, bgu, _ = tw.pack_weights(W)
        W = synth.weights_torch(dn.N, dn.K, dn.w_dist, dn.w_scale, dn.w_seed + 1000 * r, dev)
        pd, bd, _ = tw.pack_weights(W)
        del W
        x = synth.acts_torch(M, D, gu.x_dist, gu.x_seed + 1000 * r + 7919 * rank, dev, outlier_p=gu.outlier_p)
        stack.append(dict(pg=pgu[:I], pu=pgu[I:], bgu=bgu, pd=pd, bd=bd, x=x,
                          a=torch.empty((M, I), dtype=torch.float32, device=dev),
                          y=torch.empty((M, D), dtype=torch.float32, device=dev)))
    torch.cuda.synchronize(dev)
    ws = torch.zeros(max(tw.bitlinear_swiglu_workspace_bytes(M, I, D), tw.bitlinear_workspace_bytes(M, D, I)),
                     dtype=torch.uint8, device=dev)
    wbytes = args.layers * (gu.N * gu.K // 4 + dn.N * dn.K // 4)
    xes = stack[0]["x"].element_size()
    # algorithmic bytes of the gate/up SwiGLU kernel: both matrices, h, two
    # scales, the product a
    swiglu_bytes = 2 * I * D // 4 + xes * M * D + 8 + 4 * M * I

    def swiglu_all():
        for e in stack:
            tw.bitlinear_swiglu(e["x"], e["pg"], e["bgu"], e["pu"], e["bgu"], I, D, out=e["a"], workspace=ws)

    def down_all():
        for e in stack:
            tw.bitlinear(e["a"], e["pd"], e["bd"], D, I, out=e["y"], workspace=ws)

    def step():
        for e in stack:
            tw.bitlinear_swiglu(e["x"], e["pg"], e["bgu"], e["pu"], e["bgu"], I, D, out=e["a"], workspace=ws)
            tw.bitlinear(e["a"], e["pd"], e["bd"], D, I, out=e["y"], workspace=ws)

    tw.set_pdl(not args.no_pdl)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        step()
        torch.cuda.synchronize(dev)
        graph = graph_of(step, stream)
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        clocks = ClockSampler(dev.index or 0)
        clocks.start()
        time.sleep(0.3)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms_total = e0.elapsed_time(e1)
        # the dominant kernel (gate/up SwiGLU) and the down BitLinear, each
        # alone in a graph over the whole stack, same launch configuration
        n_meas = max(3, args.steps)
        sw_ms = time_replays(graph_of(swiglu_all, stream), n_meas, stream)
        dn_ms = time_replays(graph_of(down_all, stream), n_meas, stream)
        clk = clocks.stop()

        tw.set_pdl(False)
        hx = [e["x"].cpu().pin_memory() for e in stack]
        hy = [torch.empty((M, D), dtype=torch.float32).pin_memory() for _ in stack]
        h2d = sum(t.numel() * t.element_size() for t in hx)
        d2h = sum(t.numel() * t.element_size() for t in hy)

        def e2e_step():
            for e, xh, yh in zip(stack, hx, hy):
                xd = xh.to(dev, non_blocking=True)
                a = tw.bitlinear_swiglu(xd, e["pg"], e["bgu"], e["pu"], e["bgu"], I, D)
                yh.copy_(tw.bitlinear(a, e["pd"], e["bd"], D, I), non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        torch.cuda.synchronize(dev)
        e2e_s = time.perf_counter() - t0
    tw.check_device_error(stream)

    ms_step = ms_total / args.steps
    if world > 1:
        ms_step, e2e_s = max_over_ranks([ms_step, e2e_s], dev)
    value = world * wbytes / (ms_step * 1e-3) / 1e9
    achieved = swiglu_bytes * args.layers * n_meas / (sw_ms * 1e-3) / 1e9
    down_bytes = dn.N * dn.K // 4 + 4 * M * I + 4 + 4 * M * D
    # kernels per layer: M <= 2: the SwiGLU streaming kernel + the down
    # streaming kernel; M >= 3: gate (prep + GEMV), up (prep + GEMV),
    # elementwise product, down (prep + GEMV)
    per_layer = 2 if M <= 2 else 7
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic (seeded, weights and activations drawn on device)",
        "config": {"workload": f"{wl.name}: {wl.description}", "layers_in_stack": args.layers, "M": M,
                   "step": "per layer: bitlinear_swiglu (gate+up) then bitlinear (down)",
                   "packed_weight_bytes_per_step": wbytes, "graph": True, "pdl": not args.no_pdl,
                   "l2": l2_note(wbytes),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": None,
                     "kernel": "gemv_ldg_kernel SwiGLU form (gate+up, fused quant)" if M <= 2
                     else "gate/up BitLinears + swiglu_kernel", "peak_source": peak_src,
                     "launches_timed": args.layers * n_meas,
                     "avg_launch_us": round(1e3 * sw_ms / (args.layers * n_meas), 3)},
        "down_kernel": {"achieved": round(down_bytes * args.layers * n_meas / (dn_ms * 1e-3) / 1e9, 1),
                        "unit": "GB/s", "avg_launch_us": round(1e3 * dn_ms / (args.layers * n_meas), 3)},
        "e2e": {"value": round(world * wbytes * args.steps / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": per_layer * args.layers * args.steps,
        "clocks": clk,
    }
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(args)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def measure_prefill(args, dev, rank, world, bf16_peak, peak_src, sub=False):
    """Prefill: per step the fused BitLinear (quantisation into the tensor-core
    operand layout, then the tcgen05 GEMM) for both M=2048 matrices.  L2 is
    flushed (256 MB write) before every step, outside the timed spans.  With
    the rows split over ranks each rank computes its rows of both matrices.

    Returns the figures: value (TOPS of the whole job), ms per step, the GEMM
    roofline (prep + GEMM kernels alone, CUDA events), e2e through the public
    API with host buffers, clocks.  With sub=True (the prefill object of the
    default line) it uses at least 10 steps and 3 warm-up steps of its own."""
    import torch

    import ternary_weight_05_b300 as tw
    from ternary_weight_05_b300 import shard, synth

    wl = synth.workload("prefill-2048")
    M = args.M if (args.M and not sub) else 2048
    steps = max(args.steps, 10) if sub else args.steps
    warmup = max(args.warmup, 3) if sub else args.warmup
    split = world > 1 and not args.replicas
    mats = []
    for L in wl.layers:
        W = synth.weights_torch(L.N, L.K, L.w_dist, L.w_scale, L.w_seed, dev)
        packed, beta, _ = tw.pack_weights(W)
        del W
        r0, r1 = shard.row_bounds(L.N, world, rank) if split else (0, L.N)
        if split:
            packed = shard.packed_rows(packed, L.K, r0, r1).clone()
        n = r1 - r0
        x = synth.acts_torch(M, L.K, L.x_dist, L.x_seed + (0 if split else 7919 * rank), dev)
        mats.append(dict(L=L, n=n, packed=packed, beta=beta, x=x,
                         xq=torch.empty((M, L.K), dtype=torch.int8, device=dev),
                         s=torch.empty(M, dtype=torch.float32, device=dev),
                         y=torch.empty((M, n), dtype=torch.float32, device=dev),
                         ws=torch.empty(tw.gemm_workspace_bytes(M, n, L.K), dtype=torch.uint8, device=dev),
                         wsb=torch.zeros(tw.bitlinear_workspace_bytes(M, n, L.K), dtype=torch.uint8, device=dev)))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flops = sum(2.0 * M * m["n"] * m["L"].K for m in mats)
    flops_job = sum(2.0 * M * m["L"].N * m["L"].K for m in mats) * (1 if split else world)
    tw.set_pdl(not args.no_pdl)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        def step():
            for m in mats:
                if args.unfused:
                    tw.quant_act(m["x"], out=(m["xq"], m["s"]))
                    tw.w2a8_gemm(m["xq"], m["s"], m["packed"], m["beta"], m["n"], m["L"].K, out=m["y"],
                                 workspace=m["ws"])
                else:
                    tw.bitlinear(m["x"], m["packed"], m["beta"], m["n"], m["L"].K, out=m["y"], workspace=m["wsb"])

        def gemm_only():
            for m in mats:
                tw.w2a8_gemm(m["xq"], m["s"], m["packed"], m["beta"], m["n"], m["L"].K, out=m["y"],
                             workspace=m["ws"])

        for _ in range(warmup):
            step()
        torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        clocks = None
        if not sub:
            clocks = ClockSampler(dev.index or 0)
            clocks.start()
            time.sleep(0.3)
        spans, gspans = [], []
        for _ in range(steps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step()
            b.record(stream)
            spans.append((a, b))
        for m in mats:  # int8 activations for the GEMM-only timing
            tw.quant_act(m["x"], out=(m["xq"], m["s"]))
        for _ in range(steps):
            flush.fill_(2)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            gemm_only()
            b.record(stream)
            gspans.append((a, b))
        torch.cuda.synchronize(dev)
        clk = clocks.stop() if clocks is not None else None
        ms_step = sum(a.elapsed_time(b) for a, b in spans) / steps
        ms_gemm = sum(a.elapsed_time(b) for a, b in gspans) / steps
        # end to end: host activations in, host outputs out, public API
        hx = [m["x"].cpu().pin_memory() for m in mats]
        hy = [torch.empty(m["y"].shape, dtype=torch.float32).pin_memory() for m in mats]
        dx = [torch.empty_like(m["x"]) for m in mats]

        def e2e_step():
            for m, xh, xd, yh in zip(mats, hx, dx, hy):
                xd.copy_(xh, non_blocking=True)
                tw.bitlinear(xd, m["packed"], m["beta"], m["n"], m["L"].K, out=m["y"], workspace=m["wsb"])
                yh.copy_(m["y"], non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(steps):
            e2e_step()
        torch.cuda.synchronize(dev)
        e2e_s = (time.perf_counter() - t0) / steps
    tw.check_device_error(stream)
    tw.set_pdl(False)
    if world > 1:
        ms_step, e2e_s = max_over_ranks([ms_step, e2e_s], dev)
    value = flops_job / (ms_step * 1e-3) / 1e12
    achieved = flops / (ms_gemm * 1e-3) / 1e12
    res = {
        "workload": f"{wl.name}: {wl.description}", "M": M,
        "matrices": [f"{m['L'].N}x{m['L'].K}" for m in mats],
        "value": round(value, 2), "unit": "TOPS", "steps": steps, "warmup": warmup,
        "ms_per_step": round(ms_step, 4), "l2": "flushed before every step (256 MB write)",
        "step": "quant_act + w2a8_gemm per matrix" if args.unfused else "fused bitlinear per matrix",
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": round(achieved / bf16_peak, 4), "traffic": None,
                     "kernel": "gemm_tc_kernel (+prep)", "ms_per_call_pair": round(ms_gemm, 4),
                     "peak_source": peak_src + " bf16 dense burst (the GEMM runs kind::f16 MMAs; tcgen05 "
                                               "kind::i8 does not exist on sm_103a)"},
        "e2e": {"value": round(flops_job / e2e_s / 1e12, 2), "unit": "TOPS",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hx),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in hy)},
        "gpu_launches": (6 if args.unfused else 4) * steps,
    }
    if clk is not None:
        res["clocks"] = clk
    return res


def run_prefill(args, dev, rank, world, bf16_peak, peak_src):
    """The prefill workload as the whole line (--workload prefill-2048)."""
    import torch.distributed as dist

    r = measure_prefill(args, dev, rank, world, bf16_peak, peak_src)
    split = world > 1 and not args.replicas
    line = {
        "metric": METRIC, "value": r["value"], "unit": "TOPS", "n_gpus": world, "steps": r["steps"],
        "warmup": r["warmup"], "ms_per_step": r["ms_per_step"], "higher_is_better": True,
        "scaling": "strong" if split else "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded, drawn on device)",
        "config": {"workload": r["workload"], "M": r["M"], "matrices": r["matrices"], "l2": r["l2"],
                   "step": r["step"], "pdl": not args.no_pdl,
                   "parallelism": f"rows split over {world} ranks" if split else f"replicas x{world}"},
        "roofline": r["roofline"], "e2e": r["e2e"], "gpu_launches": r["gpu_launches"], "clocks": r["clocks"],
    }
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(args)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# ------------------------------------------------------------ CPU oracle --

def oracle_sample(args):
    """One layer of the workload for the oracle (bounded sample): a list of
    (name, amount, callable running the oracle on it), the amount in the
    metric's numerator (packed weight bytes; flops for the prefill GEMM)."""
    import numpy as np

    import oracle
    from ternary_weight_05_b300 import synth

    def host_packed(L, rep=0):
        W = synth.weights_np(L.N, L.K, L.w_dist, L.w_scale, seed=L.w_seed + 1000 * rep)
        packed, beta, _ = oracle.pack_weights(W)
        return packed, beta

    if args.workload == "prefill-2048":
        # every token, the first PREFILL_ORACLE_ROWS output rows of each matrix
        wl = synth.workload("prefill-2048")
        M = 2048
        sample = []
        for L in wl.layers:
            packed, beta = host_packed(L)
            _, x = synth.acts_np(M, L.K, L.x_dist, seed=L.x_seed, outlier_p=L.outlier_p, bf16=L.x_bf16)
            R = PREFILL_ORACLE_ROWS
            sample.append((f"{L.name}[:{R}]", 2 * M * R * L.K,
                           lambda threads, L=L, p=packed[:R * L.K // 4], b=beta, x=x, R=R: oracle.bitlinear(
                               x, p, b, R, L.K, threads=threads)))
        return sample, M
    if args.workload == "ffn-2b-decode":
        wl = synth.workload("ffn-2b-decode")
        gu, dn = wl.layers
        I, D, M = gu.N // 2, gu.K, args.M or 1
        pgu, bgu = host_packed(gu)
        pd, bd = host_packed(dn)
        _, x = synth.acts_np(M, D, gu.x_dist, seed=gu.x_seed, outlier_p=gu.outlier_p)

        def ffn(threads):
            h = I * D // 4  # the oracle's packed matrix is flat: gate rows, then up rows
            a, *_ = oracle.bitlinear_swiglu(x, pgu[:h], bgu, pgu[h:], bgu, I, D, threads=threads)
            oracle.bitlinear(a.astype(np.float32), pd, bd, D, I, threads=threads)

        return [("gate_up+down", gu.N * gu.K // 4 + dn.N * dn.K // 4, ffn)], M
    wl, layers, M = decode_layers(args)
    n = len(wl.layers) if args.workload == "2b-decode" else 1
    sample = []
    G = args.group
    for L, rep in layers[:n]:
        _, x = synth.acts_np(M, L.K, L.x_dist, seed=L.x_seed + 1000 * rep, outlier_p=L.outlier_p, bf16=L.x_bf16)
        if G:
            W = synth.weights_np(L.N, L.K, L.w_dist, L.w_scale, seed=L.w_seed + 1000 * rep)
            packed, ws, _ = oracle.pack_weights_grouped(W, G)
            sample.append((L.name, L.N * L.K // 4 + 4 * L.N * (L.K // G),
                           lambda threads, L=L, p=packed, w=ws, x=x: oracle.bitlinear_grouped(
                               x, p, w, L.N, L.K, G, threads=threads)))
            continue
        packed, beta = host_packed(L, rep)
        sample.append((L.name, L.N * L.K // 4,
                       lambda threads, L=L, p=packed, b=beta, x=x: oracle.bitlinear(x, p, b, L.N, L.K,
                                                                                    threads=threads)))
    return sample, M


def time_oracle(sample, seconds, threads, div=1e9):
    done, t0, passes = 0, time.perf_counter(), 0
    while True:
        for _, amount, fn in sample:
            fn(threads)
            done += amount
        passes += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return done / el / div, el, passes


def cpu_baseline(args, workload=None, seconds=None, one_thread=True):
    """The oracle, as it stands, on the host's cores over a bounded sample of
    the workload (and on one thread, for the oracle's own scaling)."""
    if workload is not None:
        args = argparse.Namespace(**{**vars(args), "workload": workload, "M": None})
    seconds = args.cpu_seconds if seconds is None else seconds
    unit, div = metric_unit(args.workload)
    try:
        sample, M = oracle_sample(args)
        cores = os.cpu_count() or 1
        v, el, passes = time_oracle(sample, seconds, cores, div)
        names = ",".join(name for name, *_ in sample)
        res = {"value": round(v, 6), "unit": unit, "cores": cores, "kind": "oracle",
               "sample": f"{passes} pass(es) over one layer ({names}; M={M}) in {el:.1f} s, "
                         f"rows split over {cores} threads"}
        if one_thread:
            # the same sample on one thread, for the scaling of the oracle itself
            v1, el1, passes1 = time_oracle(sample, min(6.0, seconds / 2), 1, div)
            res["value_1thread"] = round(v1, 6)
            res["sample_1thread"] = f"{passes1} pass(es) over the same layer in {el1:.1f} s on one thread"
        return res
    except Exception as ex:  # the baseline must never break the GPU line
        return {"value": None, "unit": unit, "cores": os.cpu_count(), "kind": "oracle", "sample": f"failed: {ex}"}


def run_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    sample, M = oracle_sample(args)
    unit, div = metric_unit(args.workload)
    cores = os.cpu_count() or 1
    per_step = args.ref_step_seconds or max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        time_oracle(sample, per_step / 4, cores, div)
    vals = []
    for _ in range(args.steps):
        v, _, _ = time_oracle(sample, per_step, cores, div)
        vals.append(v)
    value = statistics.median(vals)
    amount = sum(a for _, a, _ in sample)
    names = ",".join(name for name, *_ in sample)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": unit, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * amount / (value * div), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded numpy PCG64)",
        "config": {"workload": args.workload, "M": M, "sample": f"one layer ({names}) per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": f"each step: >= {per_step:.1f} s of passes over one layer ({names}), "
                                   f"rows split over {cores} threads"},
        "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if args.workload == "100b-stream" and not args.no_prefill:
        # the prefill half of the metric: the oracle on its bounded sample
        pf = cpu_baseline(args, workload="prefill-2048", seconds=min(10.0, per_step), one_thread=False)
        line["prefill"] = {"workload": "prefill-2048", "value": pf["value"], "unit": pf["unit"],
                           "cpu_baseline": pf}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
