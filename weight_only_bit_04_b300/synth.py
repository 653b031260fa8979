"""Seeded synthetic inputs for the W4A16 linear layer.

This module draws random numbers and nothing else: it holds none of the
quantization, packing, dequantization or matmul arithmetic. Both the tests
(which feed the CPU oracle and the CUDA path the same arrays) and the
benchmark use it.

Recipe (shapes and distributions of the workloads the pages discuss):

* Weights W [N, K]: N(0, 0.02) drawn in fp32, rounded to fp16.
* Activations x [M, K]: N(0, 1) in fp32; a seeded set of "outlier channels"
  (the same input channels for every token row, chosen without replacement)
  is multiplied by 20; then rounded to fp16. Such channels, a handful of
  inputs whose activations dwarf the rest, are what both calibration methods
  react to ("AWQ + GPTQ Quantization, in depth", section "Why small models lose
  more at 4 bits"; "LLM Quantization: INT8, GPTQ, and AWQ Explained", section
  "Round-to-nearest, and where it falls apart").
* Act order: a synthetic diag(H) with H = 2 X X^T over the workload's own
  activations, d_j = 2 * sum_t x[t, j]^2; columns are ranked by descending d
  (ties: lower column first) and column j goes to group rank(j) // g
  ("The two algorithms, compactly": under act order the columns are taken in
  descending order of their activation energy).

Seeds are derived from (workload, layer, linear, tensor) names so every run,
here or on another machine, draws the same numbers.
"""

from __future__ import annotations

import hashlib

import numpy as np

BASE_SEED = 20261202
W_STD = 0.02
OUTLIER_GAIN = 20.0

# Linear layers of one decoder block: name -> (N = out features, K = in features)
LLAMA2_7B_LINEARS = (
    ("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
    ("gate", 11008, 4096), ("up", 11008, 4096), ("down", 4096, 11008),
)
LLAMA2_7B_LAYERS = 32
LLAMA2_7B_OUTLIER_FRAC = 0.005

LLAMA_70B_LINEARS = (
    ("q", 8192, 8192), ("k", 1024, 8192), ("v", 1024, 8192), ("o", 8192, 8192),
    ("gate", 28672, 8192), ("up", 28672, 8192), ("down", 8192, 28672),
)
LLAMA_70B_LAYERS = 80
LLAMA_70B_OUTLIER_FRAC = 0.01

SINGLE_LINEAR = (256, 512)  # N x K, batch 1, 1% outliers
SWEEP_NK = (8192, 8192)
SWEEP_M = (1, 2, 4, 8, 16, 32, 64, 128)
PREFILL_SHAPES = ((11008, 4096), (4096, 11008))
PREFILL_M = 2048


def seed_for(*parts) -> int:
    """Stable 63-bit seed from BASE_SEED and any labels (str/int)."""
    h = hashlib.sha256(("%d|" % BASE_SEED + "|".join(str(p) for p in parts)).encode())
    return int.from_bytes(h.digest()[:8], "little") & ((1 << 63) - 1)


def outlier_count(K: int, frac: float) -> int:
    return int(round(frac * K))


# ---------------------------------------------------------------------------
# Host (NumPy PCG64) generators
# ---------------------------------------------------------------------------
def weights_np(N: int, K: int, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return (rng.standard_normal((N, K), dtype=np.float32) * np.float32(W_STD)).astype(np.float16)


def outlier_channels_np(K: int, frac: float, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed ^ 0x5EED))
    return np.sort(rng.choice(K, size=outlier_count(K, frac), replace=False))


def activations_np(M: int, K: int, frac: float, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((M, K), dtype=np.float32)
    x[:, outlier_channels_np(K, frac, seed)] *= np.float32(OUTLIER_GAIN)
    return x.astype(np.float16)


def act_order_g_idx(x: np.ndarray, group_size: int) -> np.ndarray:
    """Synthetic act-order map from d_j = 2 * sum_t x[t, j]^2 (fp64).

    Descending d, ties to the lower column index; g_idx[j] = rank(j) // g.
    """
    xd = np.asarray(x, dtype=np.float64)
    d = 2.0 * np.sum(xd * xd, axis=0)
    order = np.argsort(-d, kind="stable")
    rank = np.empty_like(order)
    rank[order] = np.arange(order.size)
    return (rank // group_size).astype(np.int32)


# ---------------------------------------------------------------------------
# Device (torch CUDA generator) generators for the large workloads
# ---------------------------------------------------------------------------
def weights_cuda(N: int, K: int, seed: int, device="cuda"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    w = torch.randn((N, K), generator=g, device=device, dtype=torch.float32)
    return (w * W_STD).to(torch.float16)


def activations_cuda(M: int, K: int, frac: float, seed: int, device="cuda"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    idx = torch.from_numpy(outlier_channels_np(K, frac, seed)).to(device)
    x[:, idx] *= OUTLIER_GAIN
    return x.to(torch.float16)
