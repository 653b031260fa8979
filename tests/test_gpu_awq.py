"""Unfolded AWQ act scale ("AWQ + GPTQ Quantization, in depth", The two
algorithms, compactly) through the GPU path: the quantizer of fp16(W * s) and
the packer bit-exact against the oracle, and both products -- which divide
the activations by s as they load them -- within the per-element bound
|y_gpu - y_ref| <= 2e-3 * sum_k |fp16(x / s) * w_hat| + 1e-3.
"""

import numpy as np
import pytest
import torch

from oracle import w4a16_oracle as O
from weight_only_bit_04_b300 import synth
from weight_only_bit_04_b300 import w4a16 as W

pytestmark = pytest.mark.gpu

GEMV_VARIANTS = ("ring", "async")
TILES = (1, 2, 3, 4, 5, 6)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits16(a):
    return np.asarray(a).view(np.uint16)


def variant_kw(variant):
    return dict(register_ring=variant == "ring", async_copy=variant == "async")


def assert_within(y, y_ref, B):
    y = y.astype(np.float64)
    assert np.all(np.isfinite(y)), "non-finite output"
    r = O.error_ratio(y, y_ref, B)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3f} at {np.unravel_index(r.argmax(), r.shape)}"


def no_timeouts():
    assert W.pipeline_timeouts() == 0


def act_scale_np(K, seed):
    """Seeded act scale: most channels near 1, about 1 % in 2 .. 8 (the
    salient channels get the larger scales), all fp16 and positive."""
    rng = np.random.default_rng(seed)
    s = rng.uniform(0.6, 1.6, K)
    big = rng.choice(K, max(1, K // 100), replace=False)
    s[big] = rng.uniform(2.0, 8.0, big.size)
    return s.astype(np.float16)


def awq_case(N, K, M, g, sym, act, bits=4, tag="awq"):
    """Quantized by the GPU quantizer (checked bit-exact against the oracle)."""
    W16 = synth.weights_np(N, K, synth.seed_for(tag, "w", N, K, g, sym, act, bits))
    x = synth.activations_np(M, K, 0.01, synth.seed_for(tag, "x", M, K))
    s = act_scale_np(K, synth.seed_for(tag, "s", K))
    gidx = synth.act_order_g_idx(x, g) if act else None
    y_ref, B, (q, sc, z), _, _ = O.awq_linear(x, W16, s, g, sym, gidx, bits)
    fmt = W.make_format(N, K, g, sym, act, bits=bits, act_scale=True)
    sd = to_dev(s)
    qg, sg, zg = W.quantize_rtn(fmt, to_dev(W16), gidx, act_scale=sd)
    assert np.array_equal(qg.cpu().numpy(), q)
    assert np.array_equal(bits16(sg.cpu().numpy()), bits16(sc))
    if not sym:
        assert np.array_equal(zg.cpu().numpy(), z)
    packed = W.pack(fmt, qg, sg, zg, gidx, act_scale=sd)
    return fmt, packed, to_dev(x), y_ref, B


@pytest.mark.parametrize("bits", [3, 4, 8])
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("act", [False, True])
def test_quantize_pack_dequant_bit_exact(cuda_ok, bits, sym, act):
    N, K, g = 200, 384, 64
    W16 = synth.weights_np(N, K, synth.seed_for("awq-fmt", bits, sym, act))
    x = synth.activations_np(4, K, 0.01, 61)
    s = act_scale_np(K, 62)
    gidx = synth.act_order_g_idx(x, g) if act else None
    fmt = W.make_format(N, K, g, sym, act, bits=bits, act_scale=True)
    sd = to_dev(s)
    q, sc, z = W.quantize_rtn(fmt, to_dev(W16), gidx, act_scale=sd)
    qo, so, zo = O.rtn_quantize(O.awq_scale_weights(W16, s), g, sym, gidx, bits)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(bits16(sc.cpu().numpy()), bits16(so))
    got = W.dequant(fmt, W.pack(fmt, q, sc, z, gidx, act_scale=sd)).cpu().numpy()
    assert np.array_equal(bits16(got), bits16(O.dequant(qo, so, zo, g, gidx)))


@pytest.mark.parametrize("bits", [3, 4, 8])
@pytest.mark.parametrize("g", [32, 128])
@pytest.mark.parametrize("act", [False, True])
@pytest.mark.parametrize("M", [1, 5, 16])
@pytest.mark.parametrize("variant", GEMV_VARIANTS)
def test_gemv(cuda_ok, bits, g, act, M, variant):
    fmt, packed, xd, y_ref, B = awq_case(384, 1024, M, g, False, act, bits, "awq-gemv")
    assert_within(W.gemv(fmt, packed, xd, **variant_kw(variant)).cpu().numpy(), y_ref, B)
    no_timeouts()


@pytest.mark.parametrize("N,K,g", [(200, 96, 32), (130, 320, 64), (1000, 1152, 128)])
def test_gemv_ragged(cuda_ok, N, K, g):
    for M in (1, 7):
        fmt, packed, xd, y_ref, B = awq_case(N, K, M, g, True, False, 4, "awq-ragged")
        assert_within(W.gemv(fmt, packed, xd).cpu().numpy(), y_ref, B)


@pytest.mark.parametrize("bits", [3, 4, 8])
@pytest.mark.parametrize("act", [False, True])
@pytest.mark.parametrize("tile", TILES)
def test_gemm(cuda_ok, bits, act, tile):
    fmt, packed, xd, y_ref, B = awq_case(512, 1024, 300, 128, False, act, bits, "awq-gemm")
    assert_within(W.gemm(fmt, packed, xd, tile=tile).cpu().numpy(), y_ref, B)
    no_timeouts()


@pytest.mark.parametrize("ksplit", [2, 8])
def test_gemm_split_k_and_ragged(cuda_ok, ksplit):
    for N, K, M, g in ((384, 2048, 100, 128), (130, 1024, 257, 32)):
        fmt, packed, xd, y_ref, B = awq_case(N, K, M, g, False, True, 4, "awq-splitk")
        assert_within(W.gemm(fmt, packed, xd, tile=6, ksplit=ksplit).cpu().numpy(), y_ref, B)
    no_timeouts()


def exact_case(seed, N, K, M, act):
    """Codes with s = 1, z = 8, act scales 2^e (e in {0, -1, -2}), x in
    {-1, 0, 1} with 64 nonzeros per row: x / s and every partial sum are
    integers below 2048, exact in fp16, so y is bit-exact."""
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 16, (N, K)).astype(np.uint8)
    sc = np.ones((N, K // 128), dtype=np.float16)
    z = np.full((N, K // 128), 8, dtype=np.uint8)
    s = (2.0 ** rng.integers(-2, 1, K)).astype(np.float16)
    x = np.zeros((M, K), dtype=np.float16)
    for m in range(M):
        nz = rng.choice(K, 64, replace=False)
        x[m, nz] = rng.choice([-1.0, 1.0], 64)
    gidx = synth.act_order_g_idx(x, 128) if act else None
    y_ref, _ = O.linear_ref(O.awq_scale_activations(x, s), O.dequant(q, sc, z, 128, gidx))
    fmt = W.make_format(N, K, 128, False, act, act_scale=True)
    packed = W.pack(fmt, to_dev(q), to_dev(sc), to_dev(z), gidx, act_scale=to_dev(s))
    return fmt, packed, to_dev(x), y_ref


@pytest.mark.parametrize("act", [False, True])
def test_exact_integer_case(cuda_ok, act):
    fmt, packed, xd, y_ref = exact_case(71, 384, 2048, 16, act)
    for variant in GEMV_VARIANTS:
        y = W.gemv(fmt, packed, xd, **variant_kw(variant)).cpu().numpy().astype(np.float64)
        assert np.array_equal(y, y_ref)
    fmt, packed, xd, y_ref = exact_case(72, 384, 2048, 300, act)
    for tile in TILES:
        y = W.gemm(fmt, packed, xd, tile=tile).cpu().numpy().astype(np.float64)
        assert np.array_equal(y, y_ref), tile
    no_timeouts()


def test_searched_scale_lowers_the_layer_error_on_the_gpu(cuda_ok):
    """End to end: the oracle's scale search on synthetic calibration
    activations gives s; the GPU layer quantized with it has a smaller output
    error against the unquantized fp64 product than the plain round-to-nearest
    layer on held-out activations with the same salient channels."""
    N, K = 512, 1024
    W16 = synth.weights_np(N, K, 81)
    xall = synth.activations_np(144, K, 0.01, 82)  # one set of outlier channels
    x_cal, x = xall[:128], np.ascontiguousarray(xall[128:])
    s, alpha, losses = O.awq_search(W16, x_cal, 128, False, n_grid=10)
    assert alpha > 0
    y_true = x.astype(np.float64) @ W16.astype(np.float64).T
    fmt_awq = W.make_format(N, K, 128, act_scale=True)
    sd = to_dev(s)
    q, sc, z = W.quantize_rtn(fmt_awq, to_dev(W16), act_scale=sd)
    y_awq = W.gemv(fmt_awq, W.pack(fmt_awq, q, sc, z, act_scale=sd), to_dev(x)).cpu().numpy()
    fmt = W.make_format(N, K, 128)
    q0, s0, z0 = W.quantize_rtn(fmt, to_dev(W16))
    y_rtn = W.gemv(fmt, W.pack(fmt, q0, s0, z0), to_dev(x)).cpu().numpy()
    err_awq = np.linalg.norm(y_awq.astype(np.float64) - y_true)
    err_rtn = np.linalg.norm(y_rtn.astype(np.float64) - y_true)
    assert err_awq < 0.95 * err_rtn, (err_awq, err_rtn)
