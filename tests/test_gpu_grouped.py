"""Grouped decode product (w4a16_gemv_grouped): layers that read the same
activations in one launch, each output within the per-element bound of the
oracle."""

import numpy as np
import pytest
import torch

from oracle import w4a16_oracle as O
from weight_only_bit_04_b300 import synth
from weight_only_bit_04_b300 import w4a16 as W

pytestmark = pytest.mark.gpu


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_within(y, y_ref, B):
    y = y.astype(np.float64)
    assert np.all(np.isfinite(y)), "non-finite output"
    r = O.error_ratio(y, y_ref, B)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3f}"


def group_case(Ns, K, M, g, sym, bits, tag):
    x = synth.activations_np(M, K, 0.01, synth.seed_for(tag, "x", M, K))
    fmts, packs, refs = [], [], []
    for i, N in enumerate(Ns):
        W16 = synth.weights_np(N, K, synth.seed_for(tag, "w", i, N, K, g, sym, bits))
        y_ref, B, (q, s, z), _ = O.w4a16_linear(x, W16, g, sym, None, bits)
        fmt = W.make_format(N, K, g, sym, False, bits=bits)
        fmts.append(fmt)
        packs.append(W.pack(fmt, to_dev(q), to_dev(s), None if sym else to_dev(z)))
        refs.append((y_ref, B))
    return fmts, packs, to_dev(x), refs


@pytest.mark.parametrize("bits", [3, 4, 8])
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("M", [1, 5, 16])
@pytest.mark.parametrize("variant", ["default", "ring", "async"])
def test_qkv_like_group(cuda_ok, bits, sym, M, variant):
    fmts, packs, xd, refs = group_case((512, 200, 200), 1024, M, 128, sym, bits, "grp")
    kw = dict(register_ring=variant == "ring", async_copy=variant == "async")
    ys = W.gemv_grouped(fmts, packs, xd, **kw)
    for y, (y_ref, B) in zip(ys, refs):
        assert_within(y.cpu().numpy(), y_ref, B)


@pytest.mark.parametrize("g", [32, 64])
@pytest.mark.parametrize("n", [1, 2, 4])
def test_group_sizes_counts_and_ragged_k(cuda_ok, g, n):
    Ns = (384, 130, 1000, 17)[:n]
    fmts, packs, xd, refs = group_case(Ns, 1152, 3, g, False, 4, "grp-n")
    ys = W.gemv_grouped(fmts, packs, xd)
    for y, (y_ref, B) in zip(ys, refs):
        assert_within(y.cpu().numpy(), y_ref, B)


def test_exact_integer_case(cuda_ok):
    rng = np.random.default_rng(17)
    K, M = 2048, 16
    x = np.zeros((M, K), dtype=np.float16)
    for m in range(M):
        nz = rng.choice(K, 128, replace=False)
        x[m, nz] = rng.choice([-1.0, 1.0], 128)
    fmts, packs, refs = [], [], []
    for N in (384, 128, 256):
        q = rng.integers(0, 16, (N, K)).astype(np.uint8)
        s = np.ones((N, K // 128), dtype=np.float16)
        z = np.full((N, K // 128), 8, dtype=np.uint8)
        fmt = W.make_format(N, K, 128, False, False)
        fmts.append(fmt)
        packs.append(W.pack(fmt, to_dev(q), to_dev(s), to_dev(z)))
        refs.append(O.linear_ref(x, O.dequant(q, s, z, 128))[0])
    for kw in (dict(), dict(register_ring=True), dict(async_copy=True)):
        ys = W.gemv_grouped(fmts, packs, to_dev(x), **kw)
        for y, y_ref in zip(ys, refs):
            assert np.array_equal(y.cpu().numpy().astype(np.float64), y_ref)


def test_7b_qkv_and_gate_up_full_size(cuda_ok):
    """The two groups of a 7B decoder layer at full size, oracle on sampled rows."""
    K = 4096
    x = synth.activations_cuda(1, K, synth.LLAMA2_7B_OUTLIER_FRAC, synth.seed_for("grp7b", "x"))
    for Ns in ((4096, 4096, 4096), (11008, 11008)):
        fmts, packs, ws = [], [], []
        for i, N in enumerate(Ns):
            w = synth.weights_cuda(N, K, synth.seed_for("grp7b", "w", i, N))
            fmt = W.make_format(N, K, 128, False, False)
            q, s, z = W.quantize_rtn(fmt, w)
            fmts.append(fmt)
            packs.append(W.pack(fmt, q, s, z))
            ws.append((q, s, z))
        ys = W.gemv_grouped(fmts, packs, x, weights_ready=True)
        rng = np.random.default_rng(5)
        for (q, s, z), y, f in zip(ws, ys, fmts):
            rows = rng.choice(f.N, 48, replace=False)
            rt = torch.from_numpy(rows).cuda()
            y_ref, B = O.linear_ref(x.cpu().numpy(), O.dequant(q[rt].cpu().numpy(), s[rt].cpu().numpy(),
                                                               z[rt].cpu().numpy(), 128))
            assert_within(y.cpu().numpy()[:, rows], y_ref, B)
