"""Tensor-core GEMM (any M) parity against the CPU oracle, element by element.

Acceptance per element: |y_gpu - y_ref| <= 2e-3 * sum_k |x * w_hat| + 1e-3,
with y_ref the fp64 product of x and the oracle's dequantized weights; the
integer special case must match bit for bit.
"""

import numpy as np
import pytest
import torch

from oracle import w4a16_oracle as O
from weight_only_bit_04_b300 import synth
from weight_only_bit_04_b300 import w4a16 as W

pytestmark = pytest.mark.gpu

TILES = (1, 2, 3, 4, 5, 6)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_within(y, y_ref, B):
    y = y.astype(np.float64)
    assert np.all(np.isfinite(y)), "non-finite output"
    r = O.error_ratio(y, y_ref, B)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3f} at {np.unravel_index(r.argmax(), r.shape)}"


def no_timeouts():
    assert W.pipeline_timeouts() == 0


def run_case(N, K, M, g, sym, act, tile, frac=0.01, tag="gemm", ksplit=0):
    W16 = synth.weights_np(N, K, synth.seed_for(tag, "w", N, K, g, sym, act))
    x = synth.activations_np(M, K, frac, synth.seed_for(tag, "x", M, K))
    gidx = synth.act_order_g_idx(x, g) if act else None
    y_ref, B, (q, s, z), _ = O.w4a16_linear(x, W16, g, sym, gidx)
    fmt = W.make_format(N, K, g, sym, act)
    packed = W.pack(fmt, to_dev(q), to_dev(s), None if sym else to_dev(z), gidx)
    y = W.gemm(fmt, packed, to_dev(x), tile=tile, ksplit=ksplit)
    torch.cuda.synchronize()
    return y.cpu().numpy(), y_ref, B


@pytest.mark.parametrize("tile", TILES)
def test_single_linear(cuda_ok, tile):
    for M in (64, 256):
        y, y_ref, B = run_case(256, 512, M, 128, False, False, tile, tag="single")
        assert_within(y, y_ref, B)
    no_timeouts()


@pytest.mark.parametrize("tile", TILES)
def test_exact_integer_special_case(cuda_ok, tile):
    """s = 1, z = 8, x in {-1, 0, 1} with <= 128 nonzeros per row: y is exact."""
    rng = np.random.default_rng(6)
    N, K, M = 384, 2048, 300
    q = rng.integers(0, 16, (N, K)).astype(np.uint8)
    s = np.ones((N, K // 128), dtype=np.float16)
    z = np.full((N, K // 128), 8, dtype=np.uint8)
    x = np.zeros((M, K), dtype=np.float16)
    for m in range(M):
        nz = rng.choice(K, 128, replace=False)
        x[m, nz] = rng.choice([-1.0, 1.0], 128)
    y_ref, _ = O.linear_ref(x, O.dequant(q, s, z, 128))
    fmt = W.make_format(N, K, 128, False, False)
    packed = W.pack(fmt, to_dev(q), to_dev(s), to_dev(z))
    y = W.gemm(fmt, packed, to_dev(x), tile=tile).cpu().numpy().astype(np.float64)
    assert np.array_equal(y, y_ref)
    no_timeouts()


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("tile", TILES)
def test_group_sizes_and_schemes(cuda_ok, g, sym, tile):
    y, y_ref, B = run_case(512, 1024, 384, g, sym, False, tile)
    assert_within(y, y_ref, B)
    no_timeouts()


@pytest.mark.parametrize("N,K,g,M", [(200, 96, 32, 33), (130, 320, 64, 257), (1, 128, 128, 1),
                                     (17, 64, 32, 5), (1000, 1152, 128, 130), (384, 4096, 128, 16)])
@pytest.mark.parametrize("tile", TILES)
def test_ragged_shapes(cuda_ok, N, K, g, M, tile):
    y, y_ref, B = run_case(N, K, M, g, False, False, tile, tag="ragged")
    assert_within(y, y_ref, B)
    no_timeouts()


@pytest.mark.parametrize("tile", TILES)
def test_act_order(cuda_ok, tile):
    y, y_ref, B = run_case(512, 1024, 256, 128, False, True, tile, tag="act")
    assert_within(y, y_ref, B)
    y, y_ref, B = run_case(256, 512, 100, 32, True, True, tile, tag="act")
    assert_within(y, y_ref, B)
    no_timeouts()


def test_tiles_agree_and_deterministic(cuda_ok):
    """Every tile without a K split sums the same products in the same order:
    bit-identical; the default plan (which may split K) is deterministic and
    within the bound."""
    N, K, M = 1024, 2048, 512
    W16 = synth.weights_np(N, K, 55)
    x = synth.activations_np(M, K, 0.01, 56)
    y_ref, B, (q, s, z), _ = O.w4a16_linear(x, W16, 128, False)
    fmt = W.make_format(N, K, 128, False, False)
    packed = W.pack(fmt, to_dev(q), to_dev(s), to_dev(z))
    xd = to_dev(x)
    a = W.gemm(fmt, packed, xd, tile=1).cpu().numpy()
    for tile in TILES:
        b = W.gemm(fmt, packed, xd, tile=tile).cpu().numpy()
        assert np.array_equal(a.view(np.uint16), b.view(np.uint16)), tile
    d0 = W.gemm(fmt, packed, xd).cpu().numpy()
    for _ in range(2):
        assert np.array_equal(W.gemm(fmt, packed, xd).cpu().numpy().view(np.uint16), d0.view(np.uint16))
    assert_within(d0, y_ref, B)
    no_timeouts()


def test_gemm_matches_gemv_at_16_tokens(cuda_ok):
    """Both paths at M = 16 (the crossover): each within the bound of the oracle."""
    N, K, M = 2048, 4096, 16
    W16 = synth.weights_np(N, K, 61)
    x = synth.activations_np(M, K, 0.01, 62)
    y_ref, B, (q, s, z), _ = O.w4a16_linear(x, W16, 128, False)
    fmt = W.make_format(N, K, 128, False, False)
    packed = W.pack(fmt, to_dev(q), to_dev(s), to_dev(z))
    xd = to_dev(x)
    assert_within(W.gemm(fmt, packed, xd).cpu().numpy(), y_ref, B)
    assert_within(W.gemv(fmt, packed, xd).cpu().numpy(), y_ref, B)
    no_timeouts()


@pytest.mark.parametrize("N,K", synth.PREFILL_SHAPES)
@pytest.mark.parametrize("tile", TILES)
def test_prefill_act_order_full_size(cuda_ok, N, K, tile):
    """Prefill at full size (M = 2048, act order): oracle on sampled token rows."""
    M = synth.PREFILL_M
    xd = synth.activations_cuda(M, K, 0.01, synth.seed_for("prefill-test", "x", N, K))
    x = xd.cpu().numpy()
    gidx = synth.act_order_g_idx(x, 128)
    fmt = W.make_format(N, K, 128, False, True)
    Wd = synth.weights_cuda(N, K, synth.seed_for("prefill-test", "w", N, K))
    q, s, z = W.quantize_rtn(fmt, Wd, gidx)
    packed = W.pack(fmt, q, s, z, gidx)
    y = W.gemm(fmt, packed, xd, tile=tile).cpu().numpy()
    no_timeouts()
    # the oracle quantizes the same fp16 weights (GPU quantizer = oracle, bit for bit)
    qo, so, zo = O.rtn_quantize(Wd.cpu().numpy(), 128, False, gidx)
    assert np.array_equal(q.cpu().numpy(), qo)
    w_hat = O.dequant(qo, so, zo, 128, gidx)
    rng = np.random.default_rng(N + K)
    rows = np.unique(np.concatenate([[0, M - 1], rng.choice(M, 8, replace=False)]))
    y_ref, B = O.linear_ref(x[rows], w_hat)
    assert_within(y[rows], y_ref, B)


@pytest.mark.parametrize("tile", (3, 5, 6))
@pytest.mark.parametrize("ksplit", (2, 4, 8, 16))
def test_split_k(cuda_ok, tile, ksplit):
    """K split over a cluster: partial sums added through distributed shared memory."""
    for N, K, M, g in ((384, 2048, 100, 128), (200, 1152, 33, 64), (130, 1024, 257, 32)):
        y, y_ref, B = run_case(N, K, M, g, False, False, tile, tag="splitk", ksplit=ksplit)
        assert_within(y, y_ref, B)
    no_timeouts()


@pytest.mark.parametrize("ksplit", (1, 4, 16))
def test_split_k_exact_integer_case(cuda_ok, ksplit):
    rng = np.random.default_rng(8)
    N, K, M = 256, 4096, 64
    q = rng.integers(0, 16, (N, K)).astype(np.uint8)
    s = np.ones((N, K // 128), dtype=np.float16)
    z = np.full((N, K // 128), 8, dtype=np.uint8)
    x = np.zeros((M, K), dtype=np.float16)
    for m in range(M):
        nz = rng.choice(K, 128, replace=False)
        x[m, nz] = rng.choice([-1.0, 1.0], 128)
    y_ref, _ = O.linear_ref(x, O.dequant(q, s, z, 128))
    fmt = W.make_format(N, K, 128, False, False)
    packed = W.pack(fmt, to_dev(q), to_dev(s), to_dev(z))
    y = W.gemm(fmt, packed, to_dev(x), tile=6, ksplit=ksplit).cpu().numpy().astype(np.float64)
    assert np.array_equal(y, y_ref)
    no_timeouts()


@pytest.mark.parametrize("M", [16, 32, 64, 128])
def test_crossover_sweep_default_plan(cuda_ok, M):
    """8192 x 8192 batch sweep (GEMM side): default plan, oracle on sampled rows."""
    N = K = 8192
    seed = synth.seed_for("sweep-gemm", M)
    Wd = synth.weights_cuda(N, K, seed)
    xd = synth.activations_cuda(M, K, 0.01, seed + 1)
    fmt = W.make_format(N, K, 128, False, False)
    q, s, z = W.quantize_rtn(fmt, Wd)
    packed = W.pack(fmt, q, s, z)
    y = W.gemm(fmt, packed, xd).cpu().numpy()
    no_timeouts()
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 48, replace=False)]))
    rows_t = torch.from_numpy(rows).cuda()
    qo, so, zo = O.rtn_quantize(Wd[rows_t].cpu().numpy(), 128, False)
    y_ref, B = O.linear_ref(xd.cpu().numpy(), O.dequant(qo, so, zo, 128))
    assert_within(y[:, rows], y_ref, B)
