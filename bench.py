"""Benchmark of the MoE layer forward pass on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config mixtral|qwen_prefill|qwen_decode|deepseek|toy] [--tokens T]

A step is one moe_layer_forward over one batch of synthetic tokens (router, top-k,
gate drop, permutation, grouped SwiGLU FFN, shared expert, combine).  Timing: CUDA
events on the launching stream around each step, with an L2 flush between steps outside
the events (a 512 MiB write, then a 512 MiB read of another buffer, so the previous
step's data is evicted and no dirty lines are left behind); W untimed warm-up steps; max over ranks.  With
N > 1 (torchrun) every rank runs an independent replica on its own GPU (the layer has
no exchange step on one GPU): weak scaling, value = all tokens / slowest rank's time.

The default workload is the largest one, the DeepSeek-shaped layer (T=16384, H=7168,
256 routed experts top-8 with the 0.05 gate drop, one shared expert).  The same line
carries the decode half of the metric: the Qwen3-shaped layer at T = 1, 8, 32 and 64
tokens, each replayed from a CUDA graph ("decode_sweep"; --no-decode-sweep skips it).

Extra keys: "roofline" for the dominant kernel (the grouped gate/up GEMM, timed alone
through moe_expert_gate_up, against the measured peaks), "layer_roofline" (the whole layer
against the measured and the nominal GB300 peaks, 2.25 PFLOP/s dense bf16 and 8 TB/s),
"cpu_baseline" (the CPU oracle on a bounded token sample), "e2e" (the same metric with
host buffers: every step's H2D of x and D2H of y inside the timed region; for prefill
layers whose weights exceed L2 the copies of neighbouring steps run on copy streams while a
step computes, and the serial figure is kept beside it), "stages_us" (route /
permute / gate_up / down / shared / combine, timed one by one), "gpu_launches" (the
library's own launch counter over the timed region), "clocks" (SM clock and clock-event
reasons sampled during the timed region: NVML every 10 ms, else nvidia-smi every 200 ms).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

FLUSH_BYTES = 512 << 20
L2_BYTES = 129 << 20  # GB300's L2 (126.5 MiB reported; rounded up)
PROFILES_DIR = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = [os.path.join(ROOT, "mixture_experts_layer_04_gb300", "csrc", f)
                  for f in ("gemm_tc.cu", "common.cuh")]
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# nominal GB300 peaks, the ones the layer's targets are stated against
NOMINAL_TFLOPS = 2250.0
NOMINAL_GBS = 8000.0
DECODE_SWEEP = (1, 8, 32, 64)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="deepseek", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--tokens", type=int, default=None, help="token count (decode sweeps)")
    ap.add_argument("--cpu-sample", type=int, default=None, help="tokens in the CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", dest="graph", action="store_true", default=None,
                    help="replay the layer from a CUDA graph (default: on for T <= 128)")
    ap.add_argument("--no-graph", dest="graph", action="store_false")
    ap.add_argument("--fused-combine", dest="fused", action="store_true", default=None,
                    help="fuse the combine into the down GEMM (MOE_FLAG_FUSED_COMBINE; "
                         "default for K >= 8)")
    ap.add_argument("--gather-combine", dest="fused", action="store_false")
    ap.add_argument("--fp8", action="store_true",
                    help="also time the FP8 (E4M3) gate/up: the token-row quantiser and the "
                         "kind::f8f6f4 grouped GEMM (the layer itself stays bf16)")
    ap.add_argument("--capacity", action="store_true",
                    help="capacity-limited routing (MOE_FLAG_CAPACITY: ceil(1.2 T K / E) per expert)")
    ap.add_argument("--time-row-gather", action="store_true",
                    help="also time the row-gather gate/up variant as a stage")
    ap.add_argument("--no-decode-sweep", action="store_true",
                    help="skip the Qwen3-shaped decode sweep (T = 1, 8, 32, 64)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, world, dev):
    """The largest of every rank's value (the slowest replica sets the job's time)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_seed(shape, rank):
    """Each replica draws its own token batch (and weights) from seed + rank."""
    return shape.seed + rank


def load_peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    return FALLBACK_PEAKS, "fallback"


class ClockSampler:
    """SM clock and clock-event reasons sampled while the timed region runs. Through NVML
    (ctypes on the driver's libnvidia-ml) every 10 ms where it loads, else from nvidia-smi
    every 200 ms. Only samples taken between entering and leaving the region count; if the
    region is shorter than one nvidia-smi period, the first sample after it stands in."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # clock-event reason bits of the NVML API
    NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                    0x40: "hw_thermal_slowdown"}

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.nvml = None
        self.samples = []  # (monotonic time, sm MHz, max MHz, reason names)
        self.source = None
        self.t0 = self.t1 = None
        self.stop = threading.Event()

    def _nvml_open(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return False
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
                lib.nvmlShutdown()
                return False
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError):
            return False
        self.nvml = (lib, h, reasons, ctypes)
        return True

    def _nvml_loop(self):
        lib, h, reasons, ctypes = self.nvml
        sm, mx, bits = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            ok = (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0 and
                  lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and
                  reasons(h, ctypes.byref(bits)) == 0)
            if ok:
                names = [n for b, n in self.NVML_REASONS.items() if bits.value & b]
                self.samples.append((time.monotonic(), float(sm.value), float(mx.value), names))
            self.stop.wait(0.01)

    def _smi_loop(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.strip().split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            active = [n for n, v in zip(names, parts[5:9]) if v.lower() == "active"]
            self.samples.append((time.monotonic(), sm, mx, active))

    def __enter__(self):
        if self._nvml_open():
            self.source = "nvml, every 10 ms"
            self.thread = threading.Thread(target=self._nvml_loop, daemon=True)
            self.thread.start()
        else:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "200"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi, every 200 ms"
                self.thread = threading.Thread(target=self._smi_loop, daemon=True)
                self.thread.start()
            except (OSError, FileNotFoundError):
                self.proc = None
        self.t0 = time.monotonic()
        return self

    def __exit__(self, *a):
        self.t1 = time.monotonic()
        if self.nvml is not None:
            self.stop.set()
            self.thread.join(timeout=1)
            self.nvml[0].nvmlShutdown()
        elif self.proc is not None:
            if not any(self.t0 <= t <= self.t1 for t, *_ in self.samples):
                time.sleep(0.25)  # the region was shorter than one period: take the next
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        inside = [x for x in self.samples if self.t0 <= x[0] <= self.t1]
        if not inside:
            inside = [x for x in self.samples if x[0] > self.t1][:1]
        sm = [x[1] for x in inside]
        reasons = sorted({n for x in inside for n in x[3]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": inside[-1][2] if inside else None,
                "reasons": reasons, "samples": len(sm), "source": self.source}


def gate_up_kernel(shape, T):
    """The gate/up kernel the layer launches (mirrors the library's choice): CTA pairs with
    256-row tiles for groups of >= 384 rows per expert on average (the gate/up GEMM's
    threshold), else single CTAs with 128-row tiles; decode-sized batches (T <= 128) put
    the weights on the MMA's 128-row side."""
    if shape.dtype != "bf16":
        return "tf32x3_gemm_kernel<SwiGLU> (moe_expert_gate_up)"
    if T <= 128:
        bt = 16 if T <= 16 else 32 if T <= 32 else 64
        return f"tc_grouped_gemm_kernel<{bt},SwiGLU,swap> (moe_expert_gate_up)"
    rows = T * shape.K // shape.E
    if rows >= 384 or (rows >= 256 and (shape.H >= 4096 or shape.I >= 4096)):
        return "tc_pair_gemm_kernel<SwiGLU> (moe_expert_gate_up)"
    return "tc_grouped_gemm_kernel<256,SwiGLU> (moe_expert_gate_up)"


def recorded_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` on `workload` from a committed ncu summary under
    profiles/, or None when there is none or the kernel sources changed since it was taken
    (the summary records a hash of the kernel sources)."""
    import glob
    import hashlib
    import re

    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    digest = h.hexdigest()[:16]
    pat = re.compile(r"traffic: workload=(\S+) kernel=(\S+) bytes_per_launch=(\d+) source_sha256=(\w+)")
    for path in sorted(glob.glob(os.path.join(PROFILES_DIR, "*.md"))):
        with open(path) as fh:
            for m in pat.finditer(fh.read()):
                if m.group(1) == workload and m.group(2) == kernel and m.group(4) == digest:
                    return int(m.group(3))
    return None


def algorithmic(shape, T, counts):
    """FLOPs and bytes the layer must do (not the dense work it avoids)."""
    M = int(counts.sum())
    touched = int((counts > 0).sum())
    b = 2 if shape.dtype == "bf16" else 4
    H, E, I, Is = shape.H, shape.E, shape.I, shape.I_shared
    flops = 2 * T * E * H + 6 * H * I * M + 6 * H * Is * T
    byts = T * H * b + E * H * b + 3 * H * I * b * touched + 3 * H * Is * b + T * H * b
    gate_up_flops = 4 * H * I * M
    gate_up_bytes = T * H * b + 2 * I * H * b * touched + M * I * b  # x rows read once
    return dict(M=M, touched=touched, flops=flops, bytes=byts, gate_up_flops=gate_up_flops,
                gate_up_bytes=gate_up_bytes)


def run_ours(args, rank, world, local):
    import mixture_experts_layer_04_gb300 as moe

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    moe.load()
    shape = synth.WORKLOADS[args.config]
    T = args.tokens if args.tokens is not None else shape.T
    inp = synth.make_inputs(shape.with_(seed=replica_seed(shape, rank)), device=dev, T=T)
    dt = moe.BF16 if shape.dtype == "bf16" else moe.F32
    # default: the fp32 scatter-add combine fused into the down GEMM when each token has
    # many (K >= 8) contributions to add, the deterministic gather combine otherwise
    fused = bool(args.fused) if args.fused is not None else (shape.K >= 8 and shape.dtype == "bf16")
    flags = (moe.FLAG_FUSED_COMBINE if fused else 0) | (moe.FLAG_CAPACITY if args.capacity else 0)
    cfg = moe.MoEConfig.make(T, shape.H, shape.E, shape.K, shape.I, shape.I_shared, shape.theta, dt,
                             flags)
    ws = torch.empty(moe.workspace_size(cfg), dtype=torch.uint8, device=dev)
    y = torch.empty(T, shape.H, dtype=shape.torch_dtype, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_rd = torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read another one: the inputs of the previous
        # step are evicted and no dirty lines are left for the timed kernels to write back
        flush.zero_()
        flush_rd.sum()
    stream = torch.cuda.current_stream(dev)

    def step():
        moe.layer_forward(cfg, inp["x"], inp["w_router"], inp["router_bias"], inp["w_gate_up"],
                          inp["w_down"], inp.get("w_shared_gate_up"), inp.get("w_shared_down"),
                          y, None, ws, stream=stream)

    def timed(fn, n):
        fn()  # untimed first call: module loading and one-time set-up stay out of the mean
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a, b in evs:
            flush_l2()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in evs]

    for _ in range(args.warmup):
        flush_l2()
        step()
    moe.sync_check(stream)

    # Decode-sized layers are launch-bound: capture the whole layer once in a CUDA graph
    # (every kernel, with its programmatic-dependent-launch edges) and replay it.
    use_graph = args.graph if args.graph is not None else T <= 128
    layer_step = step
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        c0 = moe.kernel_launch_count()
        with torch.cuda.graph(graph):
            moe.layer_forward(cfg, inp["x"], inp["w_router"], inp["router_bias"], inp["w_gate_up"],
                              inp["w_down"], inp.get("w_shared_gate_up"), inp.get("w_shared_down"),
                              y, None, ws, stream=torch.cuda.current_stream(dev))
        graph_launches = moe.kernel_launch_count() - c0
        layer_step = graph.replay
        for _ in range(3):
            flush_l2()
            layer_step()
        torch.cuda.synchronize(dev)

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        n0 = moe.kernel_launch_count()
        t_wall0 = time.perf_counter()
        times = timed(layer_step, args.steps)
        t_wall = time.perf_counter() - t_wall0
        # the library's own launch counter (timed() makes one untimed call before the K
        # timed ones); a graph replays the launches counted at its capture
        per_step = ((moe.kernel_launch_count() - n0) / (args.steps + 1) if not use_graph
                    else graph_launches)
        launches = per_step * args.steps
    if world > 1:
        torch.distributed.barrier()
    moe.sync_check(stream)
    ms = max_over_ranks(statistics.mean(times), world, dev)

    # routing statistics of this batch (counts come from the layer's own workspace)
    views = moe.workspace_views(cfg, ws)
    off = views["counts"] - ws.data_ptr()
    counts = ws[off:off + 4 * shape.E].view(torch.int32).cpu().numpy()
    alg = algorithmic(shape, T, counts)

    # per-stage times (M1: route, permute, expert GEMMs and combine measured separately)
    stages = {}
    E, K, H_ = shape.E, shape.K, shape.H
    logits = torch.empty(T, E, dtype=torch.float32, device=dev)
    ids = torch.empty(T, K, dtype=torch.int32, device=dev)
    w = torch.empty(T, K, dtype=torch.float32, device=dev)
    counts_t = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * K, dtype=torch.int32, device=dev)
    inv = torch.empty(T * K, dtype=torch.int32, device=dev)
    x_perm = torch.empty(T * K, H_, dtype=shape.torch_dtype, device=dev)
    h = torch.empty(T * K, shape.I, dtype=shape.torch_dtype, device=dev)
    out_perm = torch.empty(T * K, H_, dtype=torch.float32, device=dev)
    nst = max(3, min(args.steps, 10))
    stages["route"] = timed(lambda: moe.route(cfg, inp["x"], inp["w_router"], inp["router_bias"],
                                              logits, ids, w, stream=stream), nst)
    stages["permute"] = timed(lambda: moe.permute(cfg, inp["x"], ids, counts_t, offsets, perm, inv,
                                                  x_perm, ws, stream=stream), nst)
    gate_up_times = timed(lambda: moe.expert_gate_up(cfg, x_perm, offsets, inp["w_gate_up"], h, ws,
                                                     stream=stream), max(args.steps, 5))
    stages["gate_up"] = gate_up_times
    gu_kernel = gate_up_kernel(shape, T)
    if shape.dtype == "bf16" and args.time_row_gather:
        # the row-gather variant (not used by the layer), for comparison
        stages["gate_up_gather"] = timed(lambda: moe.expert_gate_up_gather(
            cfg, inp["x"], perm, offsets, inp["w_gate_up"], h, ws, stream=stream), nst)
    fp8 = None
    if args.fp8 and shape.dtype == "bf16" and H_ % 128 == 0:
        # weights quantised once (outside the timing), token rows per step
        wq = torch.empty(E, 2 * shape.I, H_, dtype=torch.uint8, device=dev)
        wsc = torch.empty(E, 2 * shape.I, dtype=torch.float32, device=dev)
        moe.quantize_fp8(inp["w_gate_up"].reshape(E * 2 * shape.I, H_), wq, wsc, stream=stream)
        xq = torch.empty(T * K, H_, dtype=torch.uint8, device=dev)
        xs = torch.empty(T * K, dtype=torch.float32, device=dev)
        stages["quantize_x_fp8"] = timed(lambda: moe.quantize_fp8(x_perm, xq, xs, stream=stream), nst)
        fp8 = timed(lambda: moe.expert_gate_up_fp8(cfg, xq, xs, offsets, wq, wsc, h, ws,
                                                  stream=stream), max(args.steps, 5))
        stages["gate_up_fp8"] = fp8
        if H_ % 128 == 0 and shape.I % 128 == 0:
            # the whole layer with FP8 experts (moe_layer_forward_fp8): the fused combine as
            # above for prefill; decode-sized layers gather (its fp32 sum would cost a zeroing
            # and a rounding launch)
            cfg8 = moe.MoEConfig.make(T, H_, E, K, shape.I, shape.I_shared, shape.theta, dt,
                                      moe.FLAG_FP8 | (moe.FLAG_CAPACITY if args.capacity else 0) |
                                      (moe.FLAG_FUSED_COMBINE if fused and T > 128 else 0))
            ws8 = torch.empty(moe.workspace_size(cfg8), dtype=torch.uint8, device=dev)
            wdq = torch.empty(E, H_, shape.I, dtype=torch.uint8, device=dev)
            wds = torch.empty(E, H_, dtype=torch.float32, device=dev)
            moe.quantize_fp8(inp["w_down"].reshape(E * H_, shape.I), wdq, wds, stream=stream)
            def fp8_layer(st=stream):
                moe.layer_forward_fp8(cfg8, inp["x"], inp["w_router"], inp["router_bias"], wq,
                                      wsc, wdq, wds, inp.get("w_shared_gate_up"),
                                      inp.get("w_shared_down"), y, None, ws8, stream=st)
            fp8_step = fp8_layer
            if T <= 128:  # like the bf16 layer: decode-sized layers replay a CUDA graph
                fp8_layer()
                torch.cuda.synchronize(dev)
                graph8 = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph8):
                    fp8_layer(torch.cuda.current_stream(dev))
                fp8_step = graph8.replay
            stages["layer_fp8"] = timed(fp8_step, nst)
    stages["down"] = timed(lambda: moe.expert_down(cfg, h, offsets, inp["w_down"], out_perm, ws,
                                                   stream=stream), nst)
    shared_out = None
    if shape.I_shared:
        one = moe.MoEConfig.make(T, H_, 1, 1, shape.I_shared, 0, 0.0, dt)
        ws1 = torch.empty(moe.workspace_size(one), dtype=torch.uint8, device=dev)
        one_off = torch.tensor([0, T], dtype=torch.int32, device=dev)
        hs = torch.empty(T, shape.I_shared, dtype=shape.torch_dtype, device=dev)
        shared_out = torch.empty(T, H_, dtype=torch.float32, device=dev)
        stages["shared"] = timed(lambda: (
            moe.expert_gate_up(one, inp["x"], one_off, inp["w_shared_gate_up"].unsqueeze(0), hs, ws1,
                               stream=stream),
            moe.expert_down(one, hs, one_off, inp["w_shared_down"].unsqueeze(0), shared_out, ws1,
                            stream=stream)), nst)
    stages["combine"] = timed(lambda: moe.combine(cfg, out_perm, inv, w, shared_out, y, None,
                                                  stream=stream), nst)
    moe.sync_check(stream)
    stages_us = {k: round(1e3 * statistics.mean(v), 2) for k, v in stages.items()}

    # roofline of the dominant kernel (grouped gate/up GEMM, timed alone)
    peaks, peak_kind = load_peaks()
    gu_s = statistics.mean(gate_up_times) / 1e3
    decode = T <= 256
    if decode:
        achieved = alg["gate_up_bytes"] / gu_s / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4)}
    else:
        achieved = alg["gate_up_flops"] / gu_s / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4)}
    roof["traffic"] = recorded_traffic(args.config if args.tokens is None else
                                       f"{args.config}-T{T}", "gate_up")
    roof["kernel"] = gu_kernel
    roof["peak_source"] = peak_kind

    # the FP8 gate/up variant (--fp8): E4M3 operands; the FP8 tensor peak is the measured
    # bf16 peak times the nominal FP8/bf16 ratio (4.5 / 2.25 PFLOP/s)
    fp8_roof = None
    if fp8 is not None:
        f8_s = statistics.mean(fp8) / 1e3
        if decode:
            f8_bytes = (T * H_ + 2 * shape.I * H_ * alg["touched"] + alg["M"] * shape.I * 2 +
                        4 * (T * K + 2 * shape.I * alg["touched"]))
            a8 = f8_bytes / f8_s / 1e9
            fp8_roof = {"bound": "hbm", "achieved": round(a8, 1), "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": round(a8 / peaks["hbm_gbs"], 4)}
        else:
            pk8 = 2.0 * peaks["bf16_tflops"]
            a8 = alg["gate_up_flops"] / f8_s / 1e12
            fp8_roof = {"bound": "tensor", "achieved": round(a8, 1), "peak": round(pk8, 1),
                        "unit": "TFLOP/s", "frac": round(a8 / pk8, 4),
                        "peak_note": "2 x measured bf16 (nominal fp8/bf16 ratio)"}
        fp8_roof["us"] = round(f8_s * 1e6, 2)
        fp8_roof["kernel"] = "tc_grouped_gemm_kernel<...,SwiGLU,F8> (moe_expert_gate_up_fp8)"

    # whole-layer roofline: the slower of FLOPs at the bf16 peak and bytes at HBM speed,
    # against the measured peaks and against the nominal GB300 peaks
    t_roof = max(alg["flops"] / (peaks["bf16_tflops"] * 1e12), alg["bytes"] / (peaks["hbm_gbs"] * 1e9))
    layer_frac = t_roof / (ms / 1e3)
    t_nom = max(alg["flops"] / (NOMINAL_TFLOPS * 1e12), alg["bytes"] / (NOMINAL_GBS * 1e9))
    layer_bound = "tensor" if alg["flops"] / NOMINAL_TFLOPS / 1e12 >= alg["bytes"] / NOMINAL_GBS / 1e9 \
        else "hbm"

    # end to end through the public API with host buffers (x in, y out, pinned)
    x_host = inp["x"].cpu().pin_memory()
    y_host = torch.empty(T, H_, dtype=shape.torch_dtype).pin_memory()
    x_dev = torch.empty_like(inp["x"])

    def e2e_step():
        x_dev.copy_(x_host, non_blocking=True)
        moe.layer_forward(cfg, x_dev, inp["w_router"], inp["router_bias"], inp["w_gate_up"],
                          inp["w_down"], inp.get("w_shared_gate_up"), inp.get("w_shared_down"),
                          y, None, ws, stream=stream)
        y_host.copy_(y, non_blocking=True)

    for _ in range(2):
        e2e_step()
    e2e_run = e2e_step
    if use_graph:
        # decode-sized layers: the copies and the layer replay as one CUDA graph, as the
        # device-only timing above does for the layer alone
        torch.cuda.synchronize(dev)
        graph_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_e2e):
            x_dev.copy_(x_host, non_blocking=True)
            moe.layer_forward(cfg, x_dev, inp["w_router"], inp["router_bias"], inp["w_gate_up"],
                              inp["w_down"], inp.get("w_shared_gate_up"), inp.get("w_shared_down"),
                              y, None, ws, stream=torch.cuda.current_stream(dev))
            y_host.copy_(y, non_blocking=True)
        e2e_run = graph_e2e.replay
        for _ in range(2):
            e2e_run()
    e2e_times = timed(e2e_run, args.steps)
    e2e_serial_ms = max_over_ranks(statistics.mean(e2e_times), world, dev)
    e2e_ms = e2e_serial_ms
    moe.sync_check(stream)

    # Pipelined end to end (prefill layers whose weights are larger than L2, so no flush is
    # needed between steps): each step still copies its x in from pinned host memory and its
    # y out, on two copy streams, with two device buffers each, so that step i+1's copy-in
    # and step i-1's copy-out run while step i's layer computes.  Timed over all K steps
    # from the first copy-in to the last copy-out.
    weight_bytes = sum(t.numel() * t.element_size() for k, t in inp.items() if k.startswith("w_"))
    pipelined = not use_graph and weight_bytes > 2 * L2_BYTES
    if pipelined:
        y_ref = y_host.clone()  # the serial steps' output
        h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        xs_host = [x_host, x_host.clone().pin_memory()]
        ys_host = [y_host, torch.empty_like(y_host).pin_memory()]
        xs_dev = [x_dev, torch.empty_like(x_dev)]
        ys_dev = [y, torch.empty_like(y)]
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_comp = [torch.cuda.Event(), torch.cuda.Event()]
        ev_out = [torch.cuda.Event(), torch.cuda.Event()]

        def pipeline(n):
            for i in range(n):
                b = i % 2
                if i >= 2:
                    h2d.wait_event(ev_comp[b])    # step i-2's layer has read xs_dev[b]
                with torch.cuda.stream(h2d):
                    xs_dev[b].copy_(xs_host[b], non_blocking=True)
                ev_in[b].record(h2d)
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_out[b])  # step i-2's y has left ys_dev[b]
                moe.layer_forward(cfg, xs_dev[b], inp["w_router"], inp["router_bias"],
                                  inp["w_gate_up"], inp["w_down"], inp.get("w_shared_gate_up"),
                                  inp.get("w_shared_down"), ys_dev[b], None, ws, stream=stream)
                ev_comp[b].record(stream)
                d2h.wait_event(ev_comp[b])
                with torch.cuda.stream(d2h):
                    ys_host[b].copy_(ys_dev[b], non_blocking=True)
                ev_out[b].record(d2h)

        pipeline(max(6, 2 * args.warmup))  # the copy paths settle over the first steps
        torch.cuda.synchronize(dev)
        t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_a.record(h2d)
        pipeline(args.steps)
        t_b.record(d2h)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(t_a.elapsed_time(t_b) / args.steps, world, dev)
        moe.sync_check(stream)
        # both buffers hold a full layer output: equal to the serial one up to the fused
        # combine's order of fp32 additions (at most a last-bit flip of the bf16 rounding)
        tol = 1e-2 * float(y_ref.float().abs().max())
        for yb in ys_host:
            assert float((yb.float() - y_ref.float()).abs().max()) <= tol, "pipelined output"

    res = {
        "metric": "MoE-layer tokens/s (prefill) & us/layer (decode), % of TC/HBM roofline",
        "value": round(T * world / (ms / 1e3), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "us_per_layer": round(ms * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": shape.dtype,
        "data": "synthetic (seeded; x~N(0,1), W_r~N(0,1/H), expert W~N(0,0.02))",
        "config": {"workload": args.config, "T": T, "H": shape.H, "E": shape.E, "K": shape.K,
                   "I": shape.I, "I_shared": shape.I_shared, "theta": shape.theta,
                   "router_bias": shape.bias,
                   "routing": "capacity ceil(1.2 T K / E) per expert" if args.capacity else "top-k",
                   "l2": "flushed between steps: 512 MiB write, then 512 MiB read of another buffer",
                   "parallelism": "replicas" if world > 1 else "single-gpu",
                   "cuda_graph": bool(use_graph),
                   "combine": "fused scatter-add (fp32, order not fixed)" if fused else "gather (deterministic)",
                   "kept_assignments": alg["M"], "experts_touched": alg["touched"],
                   "group_rows_max": int(counts.max()), "empty_experts": int((counts == 0).sum())},
        "roofline": roof,
        **({"fp8_gate_up": fp8_roof} if fp8_roof is not None else {}),
        "layer_roofline": {"bound": layer_bound,
                           "t_roofline_us": round(t_roof * 1e6, 2), "frac": round(layer_frac, 4),
                           "peaks": peak_kind,
                           "t_roofline_nominal_us": round(t_nom * 1e6, 2),
                           "frac_nominal": round(t_nom / (ms / 1e3), 4),
                           "nominal_peaks": {"tflops_bf16": NOMINAL_TFLOPS, "hbm_gbs": NOMINAL_GBS},
                           "target_frac_nominal": 0.6 if layer_bound == "tensor" else 0.7,
                           "flops": alg["flops"], "bytes": alg["bytes"]},
        "stages_us": stages_us,
        "e2e": {"value": round(T * world / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
                "d2h_bytes_per_step": y_host.numel() * y_host.element_size(),
                "cuda_graph": bool(use_graph),
                "pipelined": bool(pipelined),
                **({"overlap": "copy-in of step i+1 and copy-out of step i-1 on two copy "
                               "streams during step i's layer; two device buffers each; no L2 "
                               "flush (weights larger than L2)",
                    "serial_value": round(T * world / (e2e_serial_ms / 1e3), 1),
                    "serial_ms_per_step": round(e2e_serial_ms, 4)} if pipelined else {})},
        "gpu_launches": int(launches),
        "gpu_launches_source": "moe_kernel_launch_count() over the timed steps (graph: launches "
                               "captured x replays)",
        "clocks": clk.summary(),
        "wall_s_timed_region": round(t_wall, 3),
    }
    if not args.no_decode_sweep and args.config != "qwen_decode" and args.tokens is None:
        res["decode_sweep"] = decode_sweep(args, moe, dev, stream, timed, peaks)
    return res, shape, T, inp


def decode_sweep(args, moe, dev, stream, timed, peaks):
    """The decode half of the metric: the Qwen3-shaped layer (H=2048, E=128, top-8, I=768,
    per-expert logit bias) at T = 1, 8, 32 and 64 tokens, each replayed from a CUDA graph
    with L2 flushed between replays.  Per T: us per layer, the layer against its HBM
    roofline (measured copy bandwidth and nominal 8 TB/s), and the gate/up GEMM alone
    (its algorithmic bytes / its time, against the measured copy bandwidth)."""
    shape = synth.WORKLOADS["qwen_decode"]
    out = {}
    for T in DECODE_SWEEP:
        inp = synth.make_inputs(shape, device=dev, T=T)
        fused = shape.K >= 8
        cfg = moe.MoEConfig.make(T, shape.H, shape.E, shape.K, shape.I, shape.I_shared,
                                 shape.theta, moe.BF16, moe.FLAG_FUSED_COMBINE if fused else 0)
        ws = torch.empty(moe.workspace_size(cfg), dtype=torch.uint8, device=dev)
        y = torch.empty(T, shape.H, dtype=shape.torch_dtype, device=dev)

        def layer(st):
            moe.layer_forward(cfg, inp["x"], inp["w_router"], inp["router_bias"],
                              inp["w_gate_up"], inp["w_down"], None, None, y, None, ws, stream=st)

        for _ in range(3):
            layer(stream)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        c0 = moe.kernel_launch_count()
        with torch.cuda.graph(graph):
            layer(torch.cuda.current_stream(dev))
        n_launch = moe.kernel_launch_count() - c0
        for _ in range(3):
            graph.replay()
        t_layer = statistics.mean(timed(graph.replay, max(args.steps, 10))) / 1e3
        moe.sync_check(stream)
        # routing and dispatch of this batch, then the gate/up GEMM alone
        E, K, H_, I = shape.E, shape.K, shape.H, shape.I
        logits = torch.empty(T, E, dtype=torch.float32, device=dev)
        ids = torch.empty(T, K, dtype=torch.int32, device=dev)
        w = torch.empty(T, K, dtype=torch.float32, device=dev)
        counts = torch.empty(E, dtype=torch.int32, device=dev)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(T * K, dtype=torch.int32, device=dev)
        inv = torch.empty(T * K, dtype=torch.int32, device=dev)
        x_perm = torch.empty(T * K, H_, dtype=shape.torch_dtype, device=dev)
        h = torch.empty(T * K, I, dtype=shape.torch_dtype, device=dev)
        moe.route(cfg, inp["x"], inp["w_router"], inp["router_bias"], logits, ids, w, stream=stream)
        moe.permute(cfg, inp["x"], ids, counts, offsets, perm, inv, x_perm, ws, stream=stream)
        t_gu = statistics.mean(timed(lambda: moe.expert_gate_up(
            cfg, x_perm, offsets, inp["w_gate_up"], h, ws, stream=stream), max(args.steps, 10))) / 1e3
        moe.sync_check(stream)
        alg = algorithmic(shape, T, counts.cpu().numpy())
        gu_gbs = alg["gate_up_bytes"] / t_gu / 1e9
        out[f"T{T}"] = {
            "us_per_layer": round(t_layer * 1e6, 2),
            "layer_bytes": alg["bytes"], "experts_touched": alg["touched"],
            "layer_gbs": round(alg["bytes"] / t_layer / 1e9, 1),
            "layer_frac_measured_hbm": round(alg["bytes"] / t_layer / 1e9 / peaks["hbm_gbs"], 4),
            "layer_frac_nominal_hbm": round(alg["bytes"] / t_layer / 1e9 / NOMINAL_GBS, 4),
            "gate_up_us": round(t_gu * 1e6, 2), "gate_up_gbs": round(gu_gbs, 1),
            "gate_up_frac_measured_hbm": round(gu_gbs / peaks["hbm_gbs"], 4),
            "launches_per_layer": int(n_launch),
        }
        del graph
    return {"workload": "qwen_decode (H=2048, E=128, K=8, I=768, N(0,1) expert bias)",
            "timing": "CUDA-graph replay, L2 flushed between replays", "target_frac_nominal_hbm": 0.7,
            **out}


def oracle_sample(shape, T, inp, n_tokens, seed=0):
    """Run the CPU oracle on a bounded token sample; returns (seconds, tokens)."""
    import oracle
    from synth import to_numpy_f64 as f64

    class Lazy:
        def __init__(self, w):
            self.w = w

        def __getitem__(self, e):
            return f64(self.w[int(e)])

    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(T, size=min(T, n_tokens), replace=False))
    x = f64(inp["x"][torch.from_numpy(toks).to(inp["x"].device)])
    bias = inp["router_bias"].cpu().numpy() if inp["router_bias"] is not None else None
    sh = {}
    if shape.I_shared:
        sh = dict(w_shared_gate_up=f64(inp["w_shared_gate_up"]), w_shared_down=f64(inp["w_shared_down"]))
    t0 = time.perf_counter()
    oracle.moe_layer_tokens(x, f64(inp["w_router"]), Lazy(inp["w_gate_up"]), Lazy(inp["w_down"]),
                            shape.K, shape.theta, bias, **sh)
    return time.perf_counter() - t0, len(toks)


def default_sample(shape, T):
    return min(T, {"toy": 256, "mixtral": 16, "qwen_prefill": 256, "qwen_decode": 64,
                   "deepseek": 8}.get(shape.name, 32))


def main():
    args = parse()
    rank, world, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group(backend="nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        # The reference arm is the CPU oracle as it stands (rank 0 only).
        if rank != 0:
            return
        shape = synth.WORKLOADS[args.config]
        T = args.tokens if args.tokens is not None else shape.T
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        inp = synth.make_inputs(shape, device=dev, T=T)
        n = args.cpu_sample or default_sample(shape, T)
        for _ in range(args.warmup):
            oracle_sample(shape, T, inp, max(1, n // 4), seed=99)
        secs = [oracle_sample(shape, T, inp, n, seed=s)[0] for s in range(args.steps)]
        rate = n / statistics.mean(secs)
        res = {"impl": "reference",
               "metric": "MoE-layer tokens/s (prefill) & us/layer (decode), % of TC/HBM roofline",
               "value": round(rate, 3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": round(1e3 * statistics.mean(secs), 2),
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
               "dtype": "f64", "data": "synthetic",
               "config": {"workload": args.config, "T": T},
               "cpu_baseline": {"value": round(rate, 3), "unit": "tokens/s",
                                "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{n} random tokens of the {T}-token batch per step"},
               "e2e": {"value": round(rate, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                       "d2h_bytes_per_step": 0}}
        print(json.dumps(res))
        return
    res, shape, T, inp = run_ours(args, rank, world, local)
    if rank == 0 and not args.no_cpu_baseline:
        n = args.cpu_sample or default_sample(shape, T)
        secs, nt = oracle_sample(shape, T, inp, n)
        res["cpu_baseline"] = {"value": round(nt / secs, 3), "unit": "tokens/s",
                               "cores": os.cpu_count(), "kind": "oracle",
                               "sample": f"{nt} random tokens of the {T}-token batch, float64 numpy"}
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
