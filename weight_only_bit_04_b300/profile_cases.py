"""Small, fixed invocations of the library for profiling one kernel at a time.

    python -m weight_only_bit_04_b300.profile_cases gemm N K M [--act] [--tile T] [--calls C]
    python -m weight_only_bit_04_b300.profile_cases gemv N K M [--ring | --async] [--shape S] [--ksplit S] [--calls C]

Each run packs one seeded layer (asymmetric uint4, group 128), makes `calls`
calls of the chosen entry point on the current stream and exits 0 when the
device reports no pipeline timeout. Meant to run under a profiler that skips
the first calls (`-s`) and captures the next few (`-c`).
"""

from __future__ import annotations

import argparse
import sys

import torch

from weight_only_bit_04_b300 import synth
from weight_only_bit_04_b300 import w4a16 as W


def main(argv=None) -> int:
    p = argparse.ArgumentParser()
    p.add_argument("kind", choices=["gemm", "gemv"])
    p.add_argument("N", type=int)
    p.add_argument("K", type=int)
    p.add_argument("M", type=int)
    p.add_argument("--act", action="store_true", help="GPTQ act order (gemm)")
    p.add_argument("--tile", type=int, default=0)
    p.add_argument("--gemm-ksplit", type=int, default=0)
    p.add_argument("--ring", action="store_true", help="register-ring GEMV kernel")
    p.add_argument("--async", dest="async_copy", action="store_true", help="asynchronous-copy GEMV kernel")
    p.add_argument("--shape", type=int, default=0)
    p.add_argument("--ksplit", type=int, default=0)
    p.add_argument("--calls", type=int, default=3)
    a = p.parse_args(argv)
    dev = torch.device("cuda", 0)
    x = synth.activations_cuda(a.M, a.K, 0.01, synth.seed_for("profile", "x", a.M, a.K), device=dev)
    gidx = synth.act_order_g_idx(x.float().cpu().numpy(), 128) if a.act else None
    fmt = W.make_format(a.N, a.K, 128, False, a.act)
    q, s, z = W.quantize_rtn(fmt, synth.weights_cuda(a.N, a.K, synth.seed_for("profile", "w", a.N, a.K), device=dev),
                             gidx)
    packed = W.pack(fmt, q, s, z, gidx)
    del q, s, z
    y = torch.empty((a.M, a.N), dtype=torch.float16, device=dev)
    for _ in range(a.calls):
        if a.kind == "gemm":
            W.gemm(fmt, packed, x, out=y, tile=a.tile, ksplit=a.gemm_ksplit)
        else:
            W.gemv(fmt, packed, x, out=y, shape=a.shape, ksplit=a.ksplit, register_ring=a.ring,
                   async_copy=a.async_copy)
    torch.cuda.synchronize()
    n = W.pipeline_timeouts()
    print(f"{a.kind} {a.N}x{a.K} M={a.M}: {a.calls} calls, pipeline timeouts {n}")
    return 0 if n == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
