#!/usr/bin/env python3
"""Benchmark of the W4A16 linear layer on B300.

Default workload (one step): the Llama-2-7B-shaped decode sweep at batch 1 --
32 layers x 7 linear layers (q, k, v, o 4096x4096; gate, up 11008x4096; down
4096x11008), each with its own seeded weights (N(0, 0.02), round-to-nearest
asymmetric uint4, group 128): 224 GEMVs streaming 3.37 GB of packed weights,
far more than the 126 MB L2, so every step reads cold weights from HBM. The
headline schedule streams the whole sweep in one persistent launch of the
library's chained decode product (w4a16_chain_*); every GEMV reads its own
precomputed synthetic activations, so no GEMV waits for another. The same
launch with a decoder's data dependencies (q, k, v after the previous
layer's down; o after q..v; gate, up after o; down after gate and up) and
the per-launch schedules are reported beside it. The launch is captured in a
CUDA graph through the public API and replayed once per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload llama2-7b|llama70b|sweep8192] [--schedule S]
    python bench.py --profile-case gemv|gemm|stream --case N K M [--calls C]
                    [--layers L] [--act] [--bits B]

Prints one JSON line (rank 0). `value` is GEMV throughput in algorithmic GB/s
(packed codes + fp16 scales + 4-bit zeros + activations + outputs per GEMV)
summed over the ranks; with N > 1 every rank runs an independent replica
(weak scaling: the path has no cross-GPU exchange). Extra keys carry the other
workloads: the single 256x512 linear (microseconds per call), the 8192x8192
batch sweep with its group-size and symmetric variants, the Llama-70B-shaped
weight stream, and the prefill GEMM (M = 2048, GPTQ act order) on the tensor
cores with an fp16 cuBLAS GEMM on the same shapes for reference.
`--impl reference` times the CPU oracle (NumPy fp64 dequantize-then-matmul)
on a bounded sample of the same workload.

`--profile-case` makes a few calls of one entry point on one seeded layer (or,
for `stream`, one chained launch over L copies of it) and exits 0 when the
device reports no pipeline timeout: a small, fixed command for a profiler
that skips the first calls (-s) and captures the next few (-c).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A16 GEMV achieved HBM GB/s (% of 8 TB/s) at batch 1; GEMM TFLOP/s"
NOMINAL_HBM_GBPS = 8000.0
WORKLOAD_7B = ("llama2-7b decode sweep, batch 1: 32 layers x (q,k,v,o 4096x4096; gate,up 11008x4096; "
               "down 4096x11008), 224 GEMVs per step")
WORKLOAD_70B = ("llama-70b decode weight stream, batch 1: 80 layers x (q,o 8192x8192; k,v 1024x8192; "
                "gate,up 28672x8192; down 8192x28672), 560 GEMVs per step, all weights resident")
# Fallback peaks (one earlier B300 measurement) when the measured file is absent.
FALLBACK_HBM_GBPS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0
# ncu DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of
# the headline kernel of each schedule on the Llama-2-7B sweep (4-bit codes),
# {schedule: {"source_sha1", "bytes_per_launch"}}; valid only for the kernel
# sources it was taken on (STREAM_SOURCES for the stream and chain schedules,
# GEMV_SOURCES for the others).
GEMV_TRAFFIC = {"stream": {"source_sha1": "85b8ae41e753fdf8b76379834e376e6423165865", "bytes_per_launch": 3364989952 + 5612032}}
SCHEDULE_TEXT = {
    "stream": ("stream: the step is one persistent launch of the chained decode product (decode_stream_kernel); "
               "each GEMV reads its own precomputed activations, so none waits for another"),
    "chain": ("chain: the step is one persistent launch; q, k, v wait for the previous layer's down, o for "
              "q..v, gate and up for o, down for gate and up (device completion counters)"),
    "decode": ("decode: one launch per GEMV; k, v and up do not wait for the GEMV before them (same input); "
               "q, o, gate, down wait for their predecessor (programmatic dependent launch)"),
    "grouped": ("grouped: q,k,v in one launch and gate,up in one launch (w4a16_gemv_grouped, same input), o and "
                "down alone: 4 launches per layer, each waiting for the one before (programmatic dependent launch)"),
}
GEMV_SOURCES = ("gemv_impl.cuh", "k_gemv.cu", "k_gemv_b4.cu")
STREAM_SOURCES = ("decode_stream.cuh", "stream_geom.h", "gemv_impl.cuh", "chain.cu", "k_gemv_b4.cu")
SCHEDULES = ("stream", "chain", "grouped", "decode", "dependent", "independent")
NOMINAL_FP16_TFLOPS = 2250.0
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="llama2-7b", choices=["llama2-7b", "llama70b", "sweep8192"])
    p.add_argument("--no-gemm", action="store_true")
    p.add_argument("--no-shapes", action="store_true")
    p.add_argument("--no-gptq", action="store_true")
    p.add_argument("--bits", type=int, default=4, choices=[3, 4, 8], help="code width of every packed linear")
    p.add_argument("--schedule", default="stream", choices=list(SCHEDULES),
                   help="headline schedule: one persistent launch per step (without or with the decoder's "
                        "dependencies), grouped launches, or one launch per GEMV")
    p.add_argument("--schedules", default=",".join(SCHEDULES),
                   help="comma-separated schedules to capture and time (the headline one is always included)")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the other workloads (single linear, 8192x8192 sweep, 70B stream)")
    p.add_argument("--profile-case", choices=["gemv", "gemm", "stream"], default=None)
    p.add_argument("--case", type=int, nargs=3, metavar=("N", "K", "M"), default=(4096, 4096, 1))
    p.add_argument("--calls", type=int, default=3)
    p.add_argument("--layers", type=int, default=8, help="--profile-case stream: copies of the layer")
    p.add_argument("--time-calls", type=int, default=0,
                   help="--profile-case, outside a profiler: time this many more calls back to back")
    p.add_argument("--act", action="store_true", help="--profile-case gemm: GPTQ act order")
    return p.parse_args()


def gemv_bytes(N: int, K: int, M: int = 1, g: int = 128, sym: bool = False, bits: int = 4) -> int:
    G = K // g
    zero_bits = 8 if bits == 8 else 4  # 3-bit zero points are stored as nibbles
    return N * K * bits // 8 + N * G * 2 + (0 if sym else N * G * zero_bits // 8) + M * K * 2 + M * N * 2


def max_over_ranks(torch, dist, value: float, device) -> float:
    """The slowest rank's time (every rank gets it); the value itself on one process."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reference_rank_runs(rank: int) -> bool:
    """The reference arm (the CPU oracle) runs and prints on rank 0 only."""
    return rank == 0


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBPS, FALLBACK_BF16_TFLOPS, "fallback"


def source_sha1(names) -> str:
    h = hashlib.sha1()
    for name in names:
        with open(os.path.join(ROOT, "weight_only_bit_04_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


class _Nvml:
    """The few NVML queries the clock sampler needs, through the nvidia-ml-py
    module when it is installed, else straight from the driver's
    libnvidia-ml.so.1 with ctypes."""

    CLOCK_SM = 1  # NVML_CLOCK_SM

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.py = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.py = pynvml
            return
        except ImportError:
            pass
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def handle(self, uuid, index):
        if self.py is not None:
            try:
                return self.py.nvmlDeviceGetHandleByUUID(uuid)
            except Exception:
                return self.py.nvmlDeviceGetHandleByIndex(index)
        h = self.ct.c_void_p()
        if uuid is None or self.lib.nvmlDeviceGetHandleByUUID(self.ct.c_char_p(uuid.encode()), self.ct.byref(h)) != 0:
            if self.lib.nvmlDeviceGetHandleByIndex_v2(self.ct.c_uint(index), self.ct.byref(h)) != 0:
                raise RuntimeError("no NVML handle")
        return h

    def clock(self, h, maximum=False):
        if self.py is not None:
            fn = self.py.nvmlDeviceGetMaxClockInfo if maximum else self.py.nvmlDeviceGetClockInfo
            return float(fn(h, self.py.NVML_CLOCK_SM))
        v = self.ct.c_uint()
        fn = self.lib.nvmlDeviceGetMaxClockInfo if maximum else self.lib.nvmlDeviceGetClockInfo
        if fn(h, self.ct.c_int(self.CLOCK_SM), self.ct.byref(v)) != 0:
            raise RuntimeError("clock query failed")
        return float(v.value)

    def reasons(self, h):
        if self.py is not None:
            fn = getattr(self.py, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.py.nvmlDeviceGetCurrentClocksThrottleReasons
            return int(fn(h))
        v = self.ct.c_ulonglong()
        if self._reasons(h, self.ct.byref(v)) != 0:
            raise RuntimeError("reasons query failed")
        return int(v.value)


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons of one GPU
    every `period` seconds on a host thread (NVML), from __enter__ to
    __exit__; `summary()` keeps the samples taken while `timed` was set."""

    REASONS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40), ("sw_thermal_slowdown", 0x20),
               ("sw_power_cap", 0x4), ("hw_power_brake", 0x80))

    def __init__(self, torch, device, period=0.0005):
        import threading
        self.period = period
        self.samples = []  # (timed, sm_mhz, reasons bitmask)
        self.max_mhz = None
        self.timed = False
        self.error = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None
        try:
            if torch is None:
                raise RuntimeError("no device")
            self._nvml = _Nvml()
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            self._handle = self._nvml.handle(uuid, device.index or 0)
            self.max_mhz = self._nvml.clock(self._handle, maximum=True)
        except Exception as e:  # reported in the summary
            self.error = f"NVML unavailable: {type(e).__name__}: {e}"
            self._handle = None

    def _run(self):
        nv, h = self._nvml, self._handle
        while not self._stop.is_set():
            try:
                mhz = nv.clock(h)
                reasons = nv.reasons(h)
                self.samples.append((self.timed, mhz, reasons))
            except Exception as e:
                self.error = f"NVML query failed: {type(e).__name__}"
                return
            time.sleep(self.period)

    def __enter__(self):
        import threading
        if self._handle is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=5)
        return False

    def summary(self):
        timed = [(m, r) for t, m, r in self.samples if t]
        if not timed:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"],
                    "error": self.error or "no sample fell inside the timed region"}
        reasons = sorted({name for _, r in timed for name, bit in self.REASONS if r & bit})
        return {"sm_mhz": statistics.median(m for m, _ in timed), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(timed), "min_mhz": min(m for m, _ in timed),
                "source": f"NVML every {self.period * 1e3:g} ms during the timed region"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def build_stack(torch, W, synth, dev, workload, bits=4):
    """Pack every linear of the decode stack on the GPU (RTN, asymmetric, g128)."""
    if workload == "llama70b":
        linears, nlayers, frac, tag = synth.LLAMA_70B_LINEARS, synth.LLAMA_70B_LAYERS, synth.LLAMA_70B_OUTLIER_FRAC, "llama70b"
    else:
        linears, nlayers, frac, tag = synth.LLAMA2_7B_LINEARS, synth.LLAMA2_7B_LAYERS, synth.LLAMA2_7B_OUTLIER_FRAC, "llama2-7b"
    layers = []
    for layer in range(nlayers):
        lins = []
        for name, N, K in linears:
            fmt = W.make_format(N, K, 128, False, False, bits=bits)
            w = synth.weights_cuda(N, K, synth.seed_for(tag, layer, name, "w"), device=dev)
            q, s, z = W.quantize_rtn(fmt, w)
            packed = W.pack(fmt, q, s, z)
            del w, q, s, z
            lins.append((name, fmt, packed))
        layers.append(lins)
    Ks = sorted({K for _, _, K in linears})
    xs = {K: synth.activations_cuda(1, K, frac, synth.seed_for(tag, "x", K), device=dev) for K in Ks}
    # all outputs of a step in one buffer, so the end-to-end run reads them back in one copy
    sizes = [fmt.N for lins in layers for _, fmt, _ in lins]
    yall = torch.empty(sum(sizes), dtype=torch.float16, device=dev)
    ys, off = [], 0
    for lins in layers:
        row = []
        for _, fmt, _ in lins:
            row.append(yall[off:off + fmt.N].view(1, fmt.N))
            off += fmt.N
        ys.append(row)
    torch.cuda.synchronize()
    return layers, xs, ys, yall


def warm_graph(torch, graph, stream, reps):
    """Untimed replays on the timing stream, finished before the timed region starts."""
    with torch.cuda.stream(stream):
        for _ in range(reps):
            graph.replay()
    torch.cuda.synchronize()


def time_graph(torch, graph, stream, reps):
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def per_shape(torch, W, layers, xs, dev):
    """Each distinct layer shape on its own: a graph of one launch per layer
    (32 or 80 distinct weight copies, so the weights are cold in L2)."""
    res = {}
    names = [n for n, _, _ in layers[0]]
    seen = set()
    for j, name in enumerate(names):
        fmt = layers[0][j][1]
        key = f"{fmt.N}x{fmt.K}"
        if key in seen:
            continue
        seen.add(key)
        y = torch.empty((1, fmt.N), dtype=torch.float16, device=dev)
        stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(stream):
            for lins in layers:
                W.gemv(fmt, lins[j][2], xs[fmt.K], out=y, weights_ready=True)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for lins in layers:
                W.gemv(fmt, lins[j][2], xs[fmt.K], out=y, weights_ready=True)
        warm_graph(torch, g, stream, 3)
        ms = time_graph(torch, g, stream, 20) / len(layers)
        nb = gemv_bytes(fmt.N, fmt.K, bits=fmt.bits)
        res[key] = {"us": round(ms * 1e3, 2), "GB/s": round(nb / (ms * 1e-3) / 1e9, 1), "linears": name}
        del g
    return res


def run_ours(args, rank, world, local_rank):
    import torch
    from weight_only_bit_04_b300 import synth
    from weight_only_bit_04_b300 import w4a16 as W
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    if args.workload == "sweep8192":
        run_sweep8192(torch, W, synth, dev, args, rank, world, dist)
        return

    layers, xs, ys, yall = build_stack(torch, W, synth, dev, args.workload, args.bits)
    wanted = [x for x in args.schedules.split(",") if x]
    scheds = tuple(x for x in SCHEDULES if x == args.schedule or x in wanted)
    step = time_stack(torch, W, dev, layers, xs, ys, yall, args, dist, world, local_rank, schedules=scheds)
    shapes = None if args.no_shapes else per_shape(torch, W, layers, xs, dev)
    del layers, xs, ys, yall
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    gemm = None
    if not args.no_gemm and args.workload == "llama2-7b":
        gemm = run_gemm(torch, W, synth, dev, args)
    gptq = None
    if not args.no_gptq and args.workload == "llama2-7b" and args.bits == 4:
        gptq = run_gptq(torch, W, synth, dev)
    extra = {}
    if not args.no_extra and args.workload == "llama2-7b" and args.bits == 4:
        extra["single_linear_256x512"] = run_single_linear(torch, W, synth, dev)
        extra["sweep_8192x8192"] = sweep8192_rows(torch, W, synth, dev, variants=True)
        torch.cuda.empty_cache()
        extra["llama70b_stream"] = run_70b(torch, W, synth, dev, args, dist, world, local_rank)
        torch.cuda.empty_cache()

    if rank == 0:
        hbm, bf16, peak_kind = measured_peaks()
        ms = step["ms"]
        launches = {"stream": 1, "chain": 1, "grouped": 4 * step["n_layers"]}.get(args.schedule, step["n_launch"])
        traffic = None
        ref = GEMV_TRAFFIC.get(args.schedule)
        srcs = STREAM_SOURCES if args.schedule in ("stream", "chain") else GEMV_SOURCES
        if args.bits == 4 and ref and ref["source_sha1"] == source_sha1(srcs):
            traffic = ref["bytes_per_launch"]
        step_bytes = step["step_bytes"]
        per_rank = step_bytes / (ms * 1e-3) / 1e9
        if args.workload == "llama70b":
            workload = WORKLOAD_70B
            frac = synth.LLAMA_70B_OUTLIER_FRAC
        else:
            workload = WORKLOAD_7B
            frac = synth.LLAMA2_7B_OUTLIER_FRAC
        kernel = {"stream": "decode_stream_kernel (one persistent launch per step, after a counter reset)",
                  "chain": "decode_stream_kernel (one persistent launch per step, after a counter reset)",
                  "grouped": "gemv_kernel (every launch of the step; q,k,v and gate,up grouped)"}.get(
                      args.schedule, "gemv_kernel (every launch of the step)")
        line = {
            "metric": METRIC if args.bits == 4 else METRIC.replace("W4A16", f"W{args.bits}A16"),
            "value": round(step["value"], 1),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "fp16",
            "precision": f"fp16 activations x uint{args.bits} weights (fp16 scales), fp32 accumulate",
            "data": (f"synthetic: seeded N(0,0.02) weights RTN-quantized on the GPU, N(0,1) fp16 activations "
                     f"with {100 * frac:g}% outlier channels x20"),
            "config": {"workload": workload,
                       "M": 1, "group_size": 128, "scheme": f"asymmetric uint{args.bits}, fp16 scales",
                       "bytes_per_step": step_bytes, "gemvs_per_step": step["n_launch"],
                       "l2": f"inputs larger than L2 ({step_bytes / 1e9:.2f} GB of packed weights per step vs 126 MB L2)",
                       "timing": "CUDA graph replay per step, CUDA events on the launching stream",
                       "schedule": SCHEDULE_TEXT[args.schedule],
                       "parallelism": f"replicas x{world}"},
            "pct_of_nominal_hbm": round(100 * per_rank / NOMINAL_HBM_GBPS, 1),
            "roofline": {"bound": "hbm", "achieved": round(per_rank, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(per_rank / hbm, 4), "traffic": traffic,
                         "avg_launch_us": round(ms * 1e3 / launches, 3),
                         "alg_bytes_per_launch": round(step_bytes / launches),
                         "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                         "kernel": kernel},
            "e2e": step["e2e"],
            "gpu_launches": launches * args.steps,
            "clocks": step["clocks"],
            "decode_step_with_dependencies": step["schedules"].get("chain"),
            "schedules": step["schedules"],
            "per_shape": shapes,
            "gemm": gemm,
            "gptq": gptq,
        }
        line.update(extra)
        line["cpu_baseline"] = cpu_baseline(world)
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def chain_of(W, layers, xs, ys, deps):
    """The step as one chained launch: without waits, or with a decoder's
    data dependencies (q, k, v after the previous layer's down; o after q..v;
    gate, up after o; down after gate and up)."""
    chain_layers = []
    for li, lins in enumerate(layers):
        base = li * len(lins)
        idx = {n: base + j for j, (n, _, _) in enumerate(lins)}
        for j, (name, fmt, packed) in enumerate(lins):
            wait = None
            if deps:
                if name in ("q", "k", "v"):
                    wait = None if li == 0 else (base - 1, base - 1)
                elif name == "o":
                    wait = (idx["q"], idx["v"])
                elif name in ("gate", "up"):
                    wait = (idx["o"], idx["o"])
                else:
                    wait = (idx["gate"], idx["up"])
            chain_layers.append((fmt, packed, xs[fmt.K], ys[li][j], wait))
    return W.Chain(chain_layers, 1)


def time_stack(torch, W, dev, layers, xs, ys, yall, args, dist, world, local_rank, schedules=SCHEDULES, e2e=True):
    """Every schedule of the sweep captured in a graph; the headline one timed
    with exactly `steps` replays (barrier + synchronize on both sides, clocks
    sampled), the others after it, and the end-to-end step."""
    n_launch = sum(len(l) for l in layers)
    step_bytes = sum(gemv_bytes(fmt.N, fmt.K, bits=fmt.bits) for lins in layers for _, fmt, _ in lins)
    # Per-launch schedules. "decode": the launches that read the same
    # activations as the one before (k and v after q, up after gate) do not
    # wait for it; every other GEMV waits for its predecessor (programmatic
    # dependent launch, weights streamed early). "dependent": every GEMV
    # waits. "independent": none waits. "grouped": q,k,v and gate,up share
    # launches, every launch waits for the one before.
    same_input = {"k", "v", "up"}
    chains = {"stream": chain_of(W, layers, xs, ys, False), "chain": chain_of(W, layers, xs, ys, True)}

    def sweep(schedule):
        for li, lins in enumerate(layers):
            if schedule == "grouped":
                by = {name: (j, fmt, packed) for j, (name, fmt, packed) in enumerate(lins)}
                for group in (("q", "k", "v"), ("o",), ("gate", "up"), ("down",)):
                    sel = [by[n] for n in group if n in by]
                    if len(sel) == 1:
                        j, fmt, packed = sel[0]
                        W.gemv(fmt, packed, xs[fmt.K], out=ys[li][j], weights_ready=True)
                    else:
                        W.gemv_grouped([f for _, f, _ in sel], [p for _, _, p in sel], xs[sel[0][1].K],
                                       outs=[ys[li][j] for j, _, _ in sel], weights_ready=True)
                continue
            for j, (name, fmt, packed) in enumerate(lins):
                ready = schedule == "independent" or (schedule == "decode" and name in same_input)
                W.gemv(fmt, packed, xs[fmt.K], out=ys[li][j], weights_ready=True, inputs_ready=ready)

    stream = torch.cuda.Stream(device=dev)
    graphs = {}
    for schedule in schedules:
        run = (lambda c=chains[schedule]: c.run(stream)) if schedule in chains else (lambda s=schedule: sweep(s))
        with torch.cuda.stream(stream):
            run()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run()
        torch.cuda.synchronize()
        graphs[schedule] = g
    head = args.schedule if args.schedule in graphs else schedules[0]
    graph = graphs[head]

    # Warm-up, then exactly `steps` timed replays, barrier + synchronize on
    # both sides; clocks sampled from before the warm-up, kept for the timed region.
    with ClockSampler(torch, dev) as clk:
        warm_graph(torch, graph, stream, args.warmup)
        if dist:
            dist.barrier()
        clk.timed = True
        ms = time_graph(torch, graph, stream, args.steps)
        clk.timed = False
    if dist:
        dist.barrier()
    ms = max_over_ranks(torch, dist, ms, dev)
    value = world * step_bytes / (ms * 1e-3) / 1e9
    results = {head: {"ms_per_step": round(ms, 4), "GB/s": round(step_bytes / (ms * 1e-3) / 1e9, 1)}}
    # The other schedules, each over at least 100 replays after its warm-up.
    for schedule in schedules:
        if schedule == head:
            continue
        g = graphs[schedule]
        warm_graph(torch, g, stream, args.warmup)
        sms = time_graph(torch, g, stream, max(args.steps, 100))
        results[schedule] = {"ms_per_step": round(sms, 4), "GB/s": round(step_bytes / (sms * 1e-3) / 1e9, 1)}
    for name in chains:
        if name in results:
            results[name]["launches_per_step"] = 1
    if W.pipeline_timeouts() != 0:
        raise RuntimeError("a chained launch gave up a bounded wait: its outputs are undefined")

    e2e_rec = None
    if e2e:
        e2e_rec = time_e2e(torch, W, dev, layers, xs, ys, yall, graph, chains.get(head), head, stream, step_bytes,
                           args, dist, world)
    del graph, graphs, chains
    return {"ms": ms, "value": value, "step_bytes": step_bytes, "n_launch": n_launch, "n_layers": len(layers),
            "schedules": results, "clocks": clk.summary(), "e2e": e2e_rec}


def time_e2e(torch, W, dev, layers, xs, ys, yall, graph, chain, head, stream, step_bytes, args, dist, world):
    """End to end through the public API with host buffers: every step copies
    its inputs in from pinned host memory, runs, and copies every output back
    to pinned host memory, all inside the timed region. For the one-launch
    schedules the steps are pipelined over two input and two output buffers:
    step i + 1's inputs load (an input stream) and step i - 1's outputs read
    back (a copy stream) while step i computes, which is how a server streams
    independent steps; the per-launch schedules run one step at a time."""
    x_host = {K: x.cpu().pin_memory() for K, x in xs.items()}
    h2d = sum(x.numel() * x.element_size() for x in x_host.values())
    d2h = yall.numel() * yall.element_size()
    if chain is None:
        y_host = torch.empty(yall.shape, dtype=yall.dtype).pin_memory()

        def e2e_step(i):
            with torch.cuda.stream(stream):
                for K, x in xs.items():
                    x.copy_(x_host[K], non_blocking=True)
                graph.replay()
                y_host.copy_(yall, non_blocking=True)
            stream.synchronize()
        overlap = "none: inputs in, the step, outputs out, then a host synchronization, every step"
    else:
        # a second input and output buffer set and its own chained launch
        xs2 = {K: torch.empty_like(x) for K, x in xs.items()}
        for K in xs:
            xs2[K].copy_(xs[K])
        yall2 = torch.empty_like(yall)
        ys2, off = [], 0
        for row in ys:
            r2 = []
            for y in row:
                r2.append(yall2[off:off + y.shape[1]].view(1, y.shape[1]))
                off += y.shape[1]
            ys2.append(r2)
        chain2 = chain_of(W, layers, xs2, ys2, head == "chain")
        with torch.cuda.stream(stream):
            chain2.run(stream)
        torch.cuda.synchronize()
        graph2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph2, stream=stream):
            chain2.run(stream)
        torch.cuda.synchronize()
        graphs2, xins, youts = (graph, graph2), (xs, xs2), (yall, yall2)
        y_host = [torch.empty(yall.shape, dtype=yall.dtype).pin_memory() for _ in range(2)]
        in_stream = torch.cuda.Stream(device=dev)
        copy_stream = torch.cuda.Stream(device=dev)
        loaded = [torch.cuda.Event(), torch.cuda.Event()]
        computed = [torch.cuda.Event(), torch.cuda.Event()]
        copied = [torch.cuda.Event(), torch.cuda.Event()]

        def e2e_step(i):
            b = i & 1
            with torch.cuda.stream(in_stream):
                in_stream.wait_event(computed[b])  # step i - 2 has read input set b
                for K, x in xins[b].items():
                    x.copy_(x_host[K], non_blocking=True)
                loaded[b].record(in_stream)
            with torch.cuda.stream(stream):
                stream.wait_event(loaded[b])
                stream.wait_event(copied[b])  # output set b of step i - 2 is read back
                graphs2[b].replay()
                computed[b].record(stream)
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(computed[b])
                y_host[b].copy_(youts[b], non_blocking=True)
                copied[b].record(copy_stream)
        overlap = ("two input and two output buffer sets: step i+1's inputs load (input stream) and step "
                   "i-1's outputs read back (copy stream) while step i computes; every step's input and "
                   "output copies are inside the timed region")

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    e2e_ms = max_over_ranks(torch, dist, e2e_ms, dev)
    rec = {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
           "overlap": overlap}
    if chain is not None:
        # the same steps one at a time: inputs in, the step, outputs out, then a
        # host synchronization before the next step (nothing overlaps)
        n = min(args.steps, 50)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        t0 = time.perf_counter()
        for i in range(n):
            e2e_step(i)
            torch.cuda.synchronize()
        serial_ms = max_over_ranks(torch, dist, (time.perf_counter() - t0) * 1e3 / n, dev)
        rec["serial"] = {"value": round(world * step_bytes / (serial_ms * 1e-3) / 1e9, 1), "ms_per_step":
                         round(serial_ms, 4), "steps": n,
                         "how": "each step's copies and launch, then a host synchronization, step after step"}
    return rec


def run_70b(torch, W, synth, dev, args, dist, world, local_rank):
    """The Llama-70B-shaped weight stream at batch 1 (80 layers, ~37 GB
    packed, resident): the step as one chained launch, without and with the
    decoder's dependencies."""
    layers, xs, ys, yall = build_stack(torch, W, synth, dev, "llama70b", 4)
    step = time_stack(torch, W, dev, layers, xs, ys, yall, args, dist, world, local_rank,
                      schedules=("stream", "chain"), e2e=False)
    del layers, xs, ys, yall
    rec = {"workload": WORKLOAD_70B, "us_per_step": round(step["ms"] * 1e3, 1), "GB/s": round(step["value"], 1),
           "bytes_per_step": step["step_bytes"], "schedules": step["schedules"], "clocks": step["clocks"],
           "schedule": SCHEDULE_TEXT["stream"]}
    c = step["schedules"].get("chain")
    if c:
        rec["with_dependencies"] = {"us_per_step": round(c["ms_per_step"] * 1e3, 1), "GB/s": c["GB/s"]}
    return rec


def run_single_linear(torch, W, synth, dev):
    """The single 256x512 linear at batch 1 (asymmetric uint4, group 128):
    microseconds per w4a16_gemv call, L2 flushed before each call."""
    N, K = 256, 512
    fmt = W.make_format(N, K, 128, False, False)
    w = synth.weights_cuda(N, K, synth.seed_for("single", "w"), device=dev)
    q, s, z = W.quantize_rtn(fmt, w)
    packed = W.pack(fmt, q, s, z)
    x = synth.activations_cuda(1, K, 0.01, synth.seed_for("single", "x"), device=dev)
    y = torch.empty((1, N), dtype=torch.float16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ms = timed_calls(torch, lambda: W.gemv(fmt, packed, x, out=y), 50, flush)
    return {"shape": f"{N}x{K}", "M": 1, "us": round(ms * 1e3, 2),
            "GB/s": round(gemv_bytes(N, K) / (ms * 1e-3) / 1e9, 1),
            "timing": "median of 50 calls, CUDA events, L2 flushed before each (launch latency dominates)"}


def timed_calls(torch, fn, reps, flush):
    """Median of `reps` calls timed one by one with CUDA events, L2 flushed before each."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return float(np.median(ts))


def run_gemm(torch, W, synth, dev, args):
    """Prefill GEMM with GPTQ act order (M = 2048) on the two 7B MLP shapes,
    and an fp16 cuBLAS GEMM (torch.matmul on the dequantized weights) on the
    same shapes as a reference point."""
    M = synth.PREFILL_M
    res = {}
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    total_flop, total_ms, total_cublas = 0.0, 0.0, 0.0
    for N, K in synth.PREFILL_SHAPES:
        x = synth.activations_cuda(M, K, 0.01, synth.seed_for("prefill", "x", N, K), device=dev)
        gidx = synth.act_order_g_idx(x.float().cpu().numpy(), 128)
        fmt = W.make_format(N, K, 128, False, True, bits=args.bits)
        w = synth.weights_cuda(N, K, synth.seed_for("prefill", "w", N, K), device=dev)
        q, s, z = W.quantize_rtn(fmt, w, gidx)
        packed = W.pack(fmt, q, s, z, gidx)
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
        ws = torch.empty(max(W.gemm_workspace_bytes(fmt, M), 16), dtype=torch.uint8, device=dev)
        ms = timed_calls(torch, lambda: W.gemm(fmt, packed, x, out=y, workspace=ws), max(args.steps // 10, 10), flush)
        w_hat = W.dequant(fmt, packed)
        ms_cublas = timed_calls(torch, lambda: torch.matmul(x, w_hat.t()), max(args.steps // 10, 10), flush)
        flop = 2.0 * M * N * K
        res[f"{N}x{K}"] = {"us": round(ms * 1e3, 1), "tflops": round(flop / ms / 1e9, 1),
                           "cublas_fp16_us": round(ms_cublas * 1e3, 1),
                           "cublas_fp16_tflops": round(flop / ms_cublas / 1e9, 1)}
        total_flop += flop
        total_ms += ms
        total_cublas += ms_cublas
        del w, q, s, z, w_hat
    _, bf16, kind = measured_peaks()
    tf = total_flop / total_ms / 1e9
    res.update({"tflops": round(tf, 1), "unit": "TFLOP/s", "M": M, "act_order": True,
                "pct_of_nominal_fp16": round(100 * tf / NOMINAL_FP16_TFLOPS, 1),
                "nominal_fp16_tflops": NOMINAL_FP16_TFLOPS,
                "includes": "act-order activation gather kernel + tcgen05 GEMM kernel",
                "l2": "flushed (256 MB write) before every timed call",
                "cublas_fp16_tflops": round(total_flop / total_cublas / 1e9, 1),
                "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": bf16, "unit": "TFLOP/s",
                             "frac": round(tf / bf16, 4),
                             "peak_source": f"{kind} cuBLAS bf16 burst (MEASURED_PEAKS.json bf16_tflops); "
                                            "fp16 and bf16 dense rates are equal"}})
    # A bounded wait that gave up leaves some output tile unwritten: the
    # record is then not a valid measurement.
    timeouts = W.pipeline_timeouts()
    res["valid"] = timeouts == 0
    if timeouts:
        res["invalid"] = f"{timeouts} pipeline wait(s) gave up: outputs undefined, timings not valid"
    return res


NOMINAL_FP64_TFLOPS = 1.25


def run_gptq(torch, W, synth, dev):
    """GPTQ of one 4096 x 4096 projection with act order on 2048 calibration
    tokens (fp64 on the device), timed with CUDA events after one warm-up."""
    N = K = 4096
    T = 2048
    w = synth.weights_cuda(N, K, synth.seed_for("gptq-bench", "w"), device=dev)
    x = synth.activations_cuda(T, K, 0.01, synth.seed_for("gptq-bench", "x"), device=dev)
    fmt = W.make_format(N, K, 128, False, True)
    W.gptq(fmt, w, x)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    W.gptq(fmt, w, x)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    # multiply-adds: H = 2 x^T x (T K^2), Cholesky (K^3 / 3), triangular inverse (K^3 / 6), column loop (N K^2 / 2)
    fma = T * K * K + K ** 3 / 3 + K ** 3 / 6 + N * K * K / 2
    tf = 2 * fma / (ms * 1e-3) / 1e12
    return {"layer": f"{N}x{K}", "calib_tokens": T, "act_order": True, "ms": round(ms, 1),
            "fp64_tflops": round(tf, 3), "of_nominal_fp64": round(tf / NOMINAL_FP64_TFLOPS, 3),
            "peak_source": "nominal B300 FP64 1.25 TFLOP/s (no measured fp64 peak)"}


def sweep8192_rows(torch, W, synth, dev, variants=False):
    """8192x8192 uint4 weight, M in {1..128}: the GEMV for M <= 16 (16
    distinct weight copies, 560 MB, so that launches read cold weights), the
    GEMM for M >= 16 (L2 flushed before each call). With `variants`, also the
    GEMV at M = 1 and 16 for group sizes 32 and 64 and for the symmetric
    scheme (zero fixed at 8), and for every variant at M = 1 and 16 the 16
    copies as one chained launch (the decode stream), per copy."""
    N = K = 8192
    copies = 16
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def packs_for(g, sym):
        fmt = W.make_format(N, K, g, sym, False)
        w = synth.weights_cuda(N, K, synth.seed_for("sweep8192", "w"), device=dev)
        q, s, z = W.quantize_rtn(fmt, w)
        p0 = W.pack(fmt, q, s, z)
        del w, q, s, z
        return fmt, [p0] + [p0.clone() for _ in range(copies - 1)]

    def gemv_us(fmt, packs, x, y):
        stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(stream):
            for p in packs:
                W.gemv(fmt, p, x, out=y, weights_ready=True)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for p in packs:
                W.gemv(fmt, p, x, out=y, weights_ready=True)
        warm_graph(torch, g, stream, 3)
        ms = time_graph(torch, g, stream, 20) / copies
        del g
        return ms

    def stream_us(fmt, packs, x, M):
        """The copies as one chained launch (the decode stream), per copy."""
        ys = [torch.empty((M, N), dtype=torch.float16, device=dev) for _ in packs]
        chain = W.Chain([(fmt, p, x, y, None) for p, y in zip(packs, ys)], M)
        stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(stream):
            chain.run(stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            chain.run(stream)
        warm_graph(torch, g, stream, 3)
        ms = time_graph(torch, g, stream, 20) / copies
        del g, chain
        return ms

    def stream_row(fmt, packs, M, g, sym):
        x = synth.activations_cuda(M, K, 0.01, synth.seed_for("sweep8192", "x", M), device=dev)
        nbytes = gemv_bytes(N, K, M, g=g, sym=sym)
        ms = stream_us(fmt, packs, x, M)
        return {"M": M, "group_size": g, "scheme": "sym" if sym else "asym", "kernel": "stream",
                "us": round(ms * 1e3, 2), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
                "TFLOP/s": round(2.0 * M * N * K / ms / 1e9, 2)}

    rows = []
    fmt, packs = packs_for(128, False)
    if variants:
        for M in (1, 16):
            rows.append(stream_row(fmt, packs, M, 128, False))
    for M in synth.SWEEP_M:
        x = synth.activations_cuda(M, K, 0.01, synth.seed_for("sweep8192", "x", M), device=dev)
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
        nbytes = gemv_bytes(N, K, M)
        flop = 2.0 * M * N * K
        if M <= 16:
            ms = gemv_us(fmt, packs, x, y)
            rows.append({"M": M, "group_size": 128, "scheme": "asym", "kernel": "gemv", "us": round(ms * 1e3, 2),
                         "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1), "TFLOP/s": round(flop / ms / 1e9, 2)})
        if M >= 16:
            ms = timed_calls(torch, lambda: W.gemm(fmt, packs[0], x, out=y), 20, flush)
            rows.append({"M": M, "group_size": 128, "scheme": "asym", "kernel": "gemm", "us": round(ms * 1e3, 2),
                         "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1), "TFLOP/s": round(flop / ms / 1e9, 2)})
    del packs
    if variants:
        for g, sym in ((32, False), (64, False), (128, True)):
            fmt, packs = packs_for(g, sym)
            for M in (1, 16):
                x = synth.activations_cuda(M, K, 0.01, synth.seed_for("sweep8192", "x", M), device=dev)
                y = torch.empty((M, N), dtype=torch.float16, device=dev)
                nbytes = gemv_bytes(N, K, M, g=g, sym=sym)
                ms = gemv_us(fmt, packs, x, y)
                rows.append({"M": M, "group_size": g, "scheme": "sym" if sym else "asym", "kernel": "gemv",
                             "us": round(ms * 1e3, 2), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
                             "TFLOP/s": round(2.0 * M * N * K / ms / 1e9, 2)})
                rows.append(stream_row(fmt, packs, M, g, sym))
            del packs
    if W.pipeline_timeouts() != 0:
        raise RuntimeError("a GEMV or GEMM gave up a bounded wait: its outputs are undefined")
    return {"shape": "8192x8192", "rows": rows,
            "l2": "GEMV: 16 distinct weight copies (cold); GEMM: L2 flushed before each call"}


def run_sweep8192(torch, W, synth, dev, args, rank, world, dist):
    rec = sweep8192_rows(torch, W, synth, dev, variants=True)
    if rank == 0:
        hbm, bf16, kind = measured_peaks()
        m1 = rec["rows"][0]
        print(json.dumps({
            "metric": METRIC, "value": m1["GB/s"], "unit": "GB/s", "n_gpus": world, "steps": 20, "warmup": 3,
            "ms_per_step": m1["us"] / 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp16", "precision": "fp16 activations x uint4 weights (fp16 scales), fp32 accumulate",
            "data": "synthetic",
            "config": {"workload": "8192x8192 batch sweep M in {1..128}, asym uint4 g128 (value: M = 1 GEMV)",
                       "l2": rec["l2"]},
            "rows": rec["rows"], "peaks": {"hbm_gbs": hbm, "bf16_tflops": bf16, "source": kind}}), flush=True)


def run_profile_case(args):
    """A few calls of one entry point on one seeded layer (asymmetric, group
    128), for a profiler; exit status 0 when no bounded wait gave up."""
    import torch
    from weight_only_bit_04_b300 import synth
    from weight_only_bit_04_b300 import w4a16 as W
    N, K, M = args.case
    dev = torch.device("cuda", 0)
    x = synth.activations_cuda(M, K, 0.01, synth.seed_for("profile", "x", M, K), device=dev)
    gidx = synth.act_order_g_idx(x.float().cpu().numpy(), 128) if (args.act and args.profile_case == "gemm") else None
    fmt = W.make_format(N, K, 128, False, gidx is not None, bits=args.bits)
    q, s, z = W.quantize_rtn(fmt, synth.weights_cuda(N, K, synth.seed_for("profile", "w", N, K), device=dev), gidx)
    packed = W.pack(fmt, q, s, z, gidx)
    del q, s, z
    if args.profile_case == "stream":
        packs = [packed] + [packed.clone() for _ in range(args.layers - 1)]
        ys = [torch.empty((M, N), dtype=torch.float16, device=dev) for _ in packs]
        chain = W.Chain([(fmt, p, x, y, None) for p, y in zip(packs, ys)], M)
        call = chain.run
    else:
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
        if args.profile_case == "gemm":
            call = lambda: W.gemm(fmt, packed, x, out=y)  # noqa: E731
        else:
            call = lambda: W.gemv(fmt, packed, x, out=y)  # noqa: E731
    for _ in range(args.calls):
        call()
    torch.cuda.synchronize()
    line = f"{args.profile_case} {N}x{K} M={M} bits={args.bits}: {args.calls} calls"
    if args.time_calls > 0:
        # outside a profiler only: the calls back to back between two CUDA
        # events on the launching stream, so host work overlaps the GPU's
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.time_calls):
            call()
        e1.record(stream)
        e1.synchronize()
        ms = e0.elapsed_time(e1) / args.time_calls
        if args.profile_case == "gemm":
            rate = f"{2.0 * M * N * K / (ms * 1e-3) / 1e12:.1f} TFLOP/s (L2 not flushed)"
        else:
            nbytes = (args.layers if args.profile_case == "stream" else 1) * gemv_bytes(N, K, M, bits=args.bits)
            rate = f"{nbytes / (ms * 1e-3) / 1e9:.1f} GB/s"
        line += f"; {args.time_calls} more back to back: {ms * 1e3:.1f} us per call = {rate}"
    n = W.pipeline_timeouts()
    print(f"{line}; pipeline timeouts {n}")
    return 0 if n == 0 else 1


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------
def oracle_sample():
    """A bounded sample of the workload for the CPU oracle: the q (4096x4096)
    and down (4096x11008) linears of layer 0, quantized by the oracle."""
    from oracle import w4a16_oracle as O
    from weight_only_bit_04_b300 import synth
    sample = []
    for name, N, K in (("q", 4096, 4096), ("down", 4096, 11008)):
        Wt = synth.weights_np(N, K, synth.seed_for("llama2-7b-cpu", 0, name, "w"))
        x = synth.activations_np(1, K, synth.LLAMA2_7B_OUTLIER_FRAC, synth.seed_for("llama2-7b-cpu", "x", K))
        q, s, z = O.rtn_quantize(Wt, 128, False)
        sample.append((N, K, x, q, s, z))
    return sample


def time_oracle(sample, reps=1):
    from oracle import w4a16_oracle as O
    nbytes = 0
    t0 = time.perf_counter()
    for _ in range(reps):
        for N, K, x, q, s, z in sample:
            w_hat = O.dequant(q, s, z, 128)
            O.linear_ref(x, w_hat)
            nbytes += gemv_bytes(N, K)
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, dt


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(world):
    sample = oracle_sample()
    gbps, dt = time_oracle(sample)
    return {"value": round(gbps, 4), "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"2 of the 224 GEMVs per step (layer-0 q 4096x4096 and down 4096x11008), NumPy fp64 dequantize-then-matmul, {dt:.1f} s"}


def run_reference(args, rank, world):
    if not reference_rank_runs(rank):
        return
    sample = oracle_sample()
    for _ in range(min(args.warmup, 3)):
        time_oracle(sample[:1])
    steps = min(args.steps, 20)  # each step ~1 s of CPU work; keep the run within minutes
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(steps):
        time_oracle(sample[:1])
        nbytes += gemv_bytes(4096, 4096)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": min(args.warmup, 3),
        "ms_per_step": round(dt * 1e3 / steps, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic, same recipe as our arm",
        "config": {"workload": WORKLOAD_7B, "M": 1, "group_size": 128, "scheme": "asymmetric uint4, fp16 scales"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": ("each step a bounded sample of the workload: one 4096x4096 GEMV of it, "
                                    "NumPy fp64 dequantize-then-matmul")},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    world = max(world, 1)
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.profile_case:
        sys.exit(run_profile_case(args))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
