#!/usr/bin/env python3
"""Benchmark of the W4A16 linear layer on B300.

One step = the Llama-2-7B-shaped decode sweep at batch 1: 32 layers x 7 linear
layers (q, k, v, o 4096x4096; gate, up 11008x4096; down 4096x11008), each with
its own seeded weights (N(0, 0.02), round-to-nearest asymmetric uint4, group
128), i.e. 224 GEMV launches streaming 3.37 GB of packed weights -- far more
than the 126 MB L2, so every step reads cold weights from HBM. The launches of
one step are captured in a CUDA graph through the library's public API and
replayed once per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0). `value` is GEMV throughput in algorithmic GB/s
(packed codes + fp16 scales + 4-bit zeros + activations + outputs per launch)
summed over the ranks; with N > 1 every rank runs an independent replica
(weak scaling: the path has no cross-GPU exchange). The prefill GEMM TFLOP/s
are reported under "gemm" when the tensor-core GEMM is available.
`--impl reference` times the CPU oracle (NumPy fp64 dequantize-then-matmul) on
a bounded sample of the same workload.
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
# Fallback peaks (one earlier B300 measurement) when the measured file is absent.
FALLBACK_HBM_GBPS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0
# ncu DRAM traffic of the GEMV kernel, bytes per launch averaged over one
# layer's seven launches, valid only for the kernel source it was taken on.
GEMV_TRAFFIC = {"source_sha1": None, "bytes_per_launch": None}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-gemm", action="store_true")
    return p.parse_args()


def gemv_bytes(N: int, K: int, M: int = 1, g: int = 128, sym: bool = False) -> int:
    G = K // g
    return N * K // 2 + N * G * 2 + (0 if sym else N * G // 2) + M * K * 2 + M * N * 2


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBPS, FALLBACK_BF16_TFLOPS, "fallback"


def source_sha1(name: str) -> str:
    with open(os.path.join(ROOT, "weight_only_bit_04_b300", "csrc", name), "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)
        return False

    def summary(self):
        if not getattr(self, "samples", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def build_sweep(torch, W, synth, dev):
    """Pack the 224 linears of the Llama-2-7B-shaped stack on the GPU."""
    layers = []
    for layer in range(synth.LLAMA2_7B_LAYERS):
        lins = []
        for name, N, K in synth.LLAMA2_7B_LINEARS:
            fmt = W.make_format(N, K, 128, False, False)
            w = synth.weights_cuda(N, K, synth.seed_for("llama2-7b", layer, name, "w"), device=dev)
            q, s, z = W.quantize_rtn(fmt, w)
            packed = W.pack(fmt, q, s, z)
            del w, q, s, z
            lins.append((name, fmt, packed))
        layers.append(lins)
    xs = {K: synth.activations_cuda(1, K, synth.LLAMA2_7B_OUTLIER_FRAC, synth.seed_for("llama2-7b", "x", K),
                                    device=dev)
          for K in (4096, 11008)}
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

    layers, xs, ys, yall = build_sweep(torch, W, synth, dev)
    n_launch = sum(len(l) for l in layers)
    step_bytes = sum(gemv_bytes(fmt.N, fmt.K) for lins in layers for _, fmt, _ in lins)

    def sweep():
        for li, lins in enumerate(layers):
            for j, (name, fmt, packed) in enumerate(lins):
                W.gemv(fmt, packed, xs[fmt.K], out=ys[li][j], weights_ready=True)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        sweep()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        sweep()
    torch.cuda.synchronize()

    # Warm-up, then exactly `steps` timed replays, barrier + synchronize on both sides.
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        time.sleep(0.3)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = e0.elapsed_time(e1) / args.steps
    if dist:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    value = world * step_bytes / (ms * 1e-3) / 1e9

    # End to end through the public API with host buffers: pinned inputs copied
    # in, the step, every output copied back, all inside the timed region.
    x_host = {K: x.cpu().pin_memory() for K, x in xs.items()}
    y_host = torch.empty(yall.shape, dtype=yall.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in x_host.values())
    d2h = y_host.numel() * y_host.element_size()

    def e2e_step():
        with torch.cuda.stream(stream):
            for K, x in xs.items():
                x.copy_(x_host[K], non_blocking=True)
            graph.replay()
            y_host.copy_(yall, non_blocking=True)
        stream.synchronize()

    for _ in range(args.warmup):
        e2e_step()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    if dist:
        t = torch.tensor([e2e_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())
    e2e_value = world * step_bytes / (e2e_ms * 1e-3) / 1e9

    gemm = None
    if not args.no_gemm:
        gemm = run_gemm(torch, W, synth, dev, args)

    if rank == 0:
        hbm, bf16, peak_kind = measured_peaks()
        traffic = None
        if GEMV_TRAFFIC["source_sha1"] == source_sha1("k_gemv.cu"):
            traffic = GEMV_TRAFFIC["bytes_per_launch"]
        per_rank = step_bytes / (ms * 1e-3) / 1e9
        line = {
            "metric": METRIC,
            "value": round(value, 1),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "fp16 activations x uint4 weights, fp32 accumulate",
            "data": "synthetic: seeded N(0,0.02) weights RTN-quantized on the GPU, N(0,1) fp16 activations with 0.5% outlier channels x20",
            "config": {"workload": "llama2-7b decode sweep, batch 1: 32 layers x (q,k,v,o 4096x4096; gate,up 11008x4096; down 4096x11008), 224 GEMVs per step",
                       "M": 1, "group_size": 128, "scheme": "asymmetric uint4, fp16 scales",
                       "bytes_per_step": step_bytes, "launches_per_step": n_launch,
                       "l2": "inputs larger than L2 (3.37 GB of packed weights per step vs 126 MB L2)",
                       "timing": "CUDA graph replay per step, CUDA events on the launching stream",
                       "parallelism": f"replicas x{world}"},
            "pct_of_nominal_hbm": round(100 * per_rank / NOMINAL_HBM_GBPS, 1),
            "roofline": {"bound": "hbm", "achieved": round(per_rank, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(per_rank / hbm, 4), "traffic": traffic,
                         "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                         "kernel": "gemv_kernel (every launch of the step)"},
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": n_launch * args.steps,
            "clocks": clk.summary(),
            "gemm": gemm,
        }
        line["cpu_baseline"] = cpu_baseline(world)
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_gemm(torch, W, synth, dev, args):
    """Prefill GEMM with GPTQ act order (M = 2048) on the two 7B MLP shapes."""
    M = synth.PREFILL_M
    res = {}
    try:
        total_flop, total_ms = 0.0, 0.0
        for N, K in synth.PREFILL_SHAPES:
            x = synth.activations_cuda(M, K, 0.01, synth.seed_for("prefill", "x", N, K), device=dev)
            gidx = synth.act_order_g_idx(x.float().cpu().numpy(), 128)
            fmt = W.make_format(N, K, 128, False, True)
            w = synth.weights_cuda(N, K, synth.seed_for("prefill", "w", N, K), device=dev)
            q, s, z = W.quantize_rtn(fmt, w, gidx)
            packed = W.pack(fmt, q, s, z, gidx)
            y = torch.empty((M, N), dtype=torch.float16, device=dev)
            ws = torch.empty(max(W.gemm_workspace_bytes(fmt, M), 1), dtype=torch.uint8, device=dev)
            for _ in range(args.warmup):
                W.gemm(fmt, packed, x, out=y, workspace=ws)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.steps):
                W.gemm(fmt, packed, x, out=y, workspace=ws)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.steps
            flop = 2.0 * M * N * K
            res[f"{N}x{K}"] = {"ms": round(ms, 4), "tflops": round(flop / ms / 1e9, 1)}
            total_flop += flop
            total_ms += ms
        _, bf16, kind = measured_peaks()
        tf = total_flop / total_ms / 1e9
        res.update({"tflops": round(tf, 1), "unit": "TFLOP/s", "M": M, "act_order": True,
                    "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": bf16, "unit": "TFLOP/s",
                                 "frac": round(tf / bf16, 4),
                                 "peak_source": f"{kind} cuBLAS bf16 burst (fp16 tensor rate is the same)"}})
        return res
    except Exception as ex:  # the tensor-core GEMM may not be built on this revision
        return {"unavailable": str(ex)[:200]}


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
    if rank != 0:
        return
    sample = oracle_sample()
    for _ in range(args.warmup):
        time_oracle(sample[:1])
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        g, dt = time_oracle(sample[:1])
        nbytes += gemv_bytes(4096, 4096)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic, same recipe as our arm",
        "config": {"workload": "llama2-7b decode sweep, batch 1 (each step: the CPU oracle on one 4096x4096 GEMV of it)",
                   "M": 1, "group_size": 128, "scheme": "asymmetric uint4, fp16 scales"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": "one 4096x4096 GEMV of the sweep per step, NumPy fp64 dequantize-then-matmul"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.impl == "ours" and args.gpus == 1 else 1)))
    world = max(world, 1)
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
