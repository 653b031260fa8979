"""3- and 8-bit codes (W3A16, W8A16: the other widths named in "How do GPTQ
and AWQ differ ...", section "The shared setting") through the same entry
points: quantize / pack / dequant bit-exact against the CPU oracle, and both
products within the per-element bound |y_gpu - y_ref| <= 2e-3 * sum_k |x * w_hat| + 1e-3.
Every test runs once per width.
"""

import numpy as np
import pytest
import torch

from oracle import w4a16_oracle as O
from weight_only_bit_04_b300 import synth
from weight_only_bit_04_b300 import w4a16 as W

pytestmark = [pytest.mark.gpu, pytest.mark.parametrize("BITS", [3, 8])]
GEMV_VARIANTS = ("ring", "ring_sx", "async", "async_sx")
TILES = (1, 2, 3, 4, 5, 6)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits16(a):
    return np.asarray(a).view(np.uint16)


def variant_kw(variant):
    return dict(register_ring=variant.startswith("ring"), async_copy=variant.startswith("async"),
                stage_activations=variant.endswith("_sx"))


def fmtb(BITS, N, K, g, sym, act):
    return W.make_format(N, K, g, sym, act, bits=BITS)


def pack_oracle(fmt, q, s, z, gidx=None):
    return W.pack(fmt, to_dev(q), to_dev(s), None if fmt.symmetric else to_dev(z), gidx)


def assert_within(y, y_ref, B):
    y = y.astype(np.float64)
    assert np.all(np.isfinite(y)), "non-finite output"
    r = O.error_ratio(y, y_ref, B)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3f} at {np.unravel_index(r.argmax(), r.shape)}"


def no_timeouts():
    assert W.pipeline_timeouts() == 0


def oracle_case(BITS, N, K, M, g, sym, act, tag):
    W16 = synth.weights_np(N, K, synth.seed_for(tag, f"w{BITS}", N, K, g, sym, act))
    x = synth.activations_np(M, K, 0.01, synth.seed_for(tag, f"x{BITS}", M, K))
    gidx = synth.act_order_g_idx(x, g) if act else None
    y_ref, B, (q, s, z), _ = O.w4a16_linear(x, W16, g, sym, gidx, bits=BITS)
    fmt = fmtb(BITS, N, K, g, sym, act)
    return fmt, pack_oracle(fmt, q, s, z, gidx), to_dev(x), y_ref, B


# ---------------------------------------------------------------- format


@pytest.mark.parametrize("N,K,g,sym,act", [
    (256, 512, 128, False, False),
    (200, 96, 32, False, False),     # ragged rows and columns
    (136, 192, 64, True, False),
    (130, 256, 128, False, True),    # act order
    (64, 384, 64, True, True),
])
def test_pack_then_dequant_is_bit_exact(cuda_ok, BITS, N, K, g, sym, act):
    W16 = synth.weights_np(N, K, synth.seed_for(f"fmt{BITS}", N, K, g, sym, act))
    x = synth.activations_np(4, K, 0.01, synth.seed_for(f"fmt{BITS}-x", K))
    gidx = synth.act_order_g_idx(x, g) if act else None
    q, s, z = O.rtn_quantize(W16, g, sym, gidx, bits=BITS)
    fmt = fmtb(BITS, N, K, g, sym, act)
    got = W.dequant(fmt, pack_oracle(fmt, q, s, z, gidx)).cpu().numpy()
    assert np.array_equal(bits16(got), bits16(O.dequant(q, s, z, g, gidx)))


def test_pack_every_code_position(cuda_ok, BITS):
    """Random codes at every row/column position of a 128 x 64 tile (s = 1, z = 0),
    and each code value alone in each position of one lane's words."""
    N, K, g = 128, 64, 32
    rng = np.random.default_rng(0)
    fmt = fmtb(BITS, N, K, g, False, False)
    s = np.ones((N, K // g), dtype=np.float16)
    z = np.zeros((N, K // g), dtype=np.uint8)
    for r, c in [(0, 0), (8, 5), (17, 63), (127, 31), (64, 48)]:
        for v in (1, (1 << BITS) - 1):
            q = np.zeros((N, K), dtype=np.uint8)
            q[r, c] = v
            got = W.dequant(fmt, pack_oracle(fmt, q, s, z)).cpu().numpy()
            assert np.array_equal(got.astype(np.int64), q.astype(np.int64)), (r, c, v)
    for _ in range(4):
        q = rng.integers(0, 1 << BITS, (N, K)).astype(np.uint8)
        s = np.ones((N, K // g), dtype=np.float16)
        z = np.zeros((N, K // g), dtype=np.uint8)
        got = W.dequant(fmt, pack_oracle(fmt, q, s, z)).cpu().numpy()
        assert np.array_equal(got.astype(np.int64), q.astype(np.int64))


def test_dequant_every_scale_selected_zeros(cuda_ok, BITS):
    """Every finite fp16 scale, every code, zeros {0, middle, top} (8 bits) or
    every zero (3 bits)."""
    svals = np.arange(0x10000, dtype=np.uint32).astype(np.uint16).view(np.float16)
    svals = svals[np.isfinite(svals)]
    top = (1 << BITS) - 1
    zs = np.array([0, 128, 255] if BITS == 8 else list(range(top + 1)), dtype=np.uint8)
    g, K = (128, 256) if BITS == 8 else (32, 32)     # every code in every row
    N = svals.size * zs.size
    s = np.repeat(np.repeat(svals, zs.size)[:, None], K // g, axis=1)
    z = np.repeat(np.tile(zs, svals.size)[:, None], K // g, axis=1)
    q = np.tile(np.arange(K, dtype=np.int64) % (top + 1), (N, 1)).astype(np.uint8)
    fmt = fmtb(BITS, N, K, g, False, False)
    got = W.dequant(fmt, pack_oracle(fmt, q, s, z)).cpu().numpy()
    with np.errstate(over="ignore"):
        want = O.dequant(q, s, z, g)
    assert np.array_equal(bits16(got), bits16(want))


@pytest.mark.parametrize("N,K,g,sym,act", [
    (256, 512, 128, False, False),
    (96, 256, 32, False, False),
    (64, 384, 64, True, False),
    (128, 512, 128, False, True),
    (40, 256, 64, True, True),
])
def test_gpu_rtn_matches_oracle_bit_exactly(cuda_ok, BITS, N, K, g, sym, act):
    W16 = synth.weights_np(N, K, synth.seed_for(f"rtn{BITS}", N, K, g, sym, act))
    W16[0, :g] = np.float16(0.25)                    # constant group
    W16[1, :8] = np.array([-7.0, 8.0, 2.5, 3.5, -0.5, 0.5, -1.5, 1.5], dtype=np.float16)
    W16[1, 8:g] = np.float16(0.0)
    W16[2, :g] = np.abs(W16[2, :g]) + np.float16(0.01)  # one-signed group
    x = synth.activations_np(2, K, 0.01, synth.seed_for(f"rtn{BITS}-x", K))
    gidx = synth.act_order_g_idx(x, g) if act else None
    fmt = fmtb(BITS, N, K, g, sym, act)
    q, s, z = W.quantize_rtn(fmt, to_dev(W16), gidx)
    qo, so, zo = O.rtn_quantize(W16, g, sym, gidx, bits=BITS)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(bits16(s.cpu().numpy()), bits16(so))
    if not sym:
        assert np.array_equal(z.cpu().numpy(), zo)
    elif BITS == 8:
        qn = q.cpu().numpy()
        assert qn.min() >= 1 and qn.max() <= 255  # int8 absmax codes -127..127, offset by 128


# ---------------------------------------------------------------- GEMV


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("M", [1, 5, 16])
@pytest.mark.parametrize("variant", GEMV_VARIANTS)
def test_gemv_groups_and_schemes(cuda_ok, BITS, g, sym, M, variant):
    fmt, packed, xd, y_ref, B = oracle_case(BITS, 256, 1024, M, g, sym, False, "gemv8")
    assert_within(W.gemv(fmt, packed, xd, **variant_kw(variant)).cpu().numpy(), y_ref, B)
    no_timeouts()


@pytest.mark.parametrize("N,K,g", [(200, 96, 32), (130, 320, 64), (1, 128, 128), (17, 64, 32),
                                   (1000, 1152, 128)])
@pytest.mark.parametrize("variant", GEMV_VARIANTS)
def test_gemv_ragged_shapes(cuda_ok, BITS, N, K, g, variant):
    for M in (1, 7):
        fmt, packed, xd, y_ref, B = oracle_case(BITS, N, K, M, g, False, False, "gemv8-ragged")
        assert_within(W.gemv(fmt, packed, xd, **variant_kw(variant)).cpu().numpy(), y_ref, B)


@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("variant", GEMV_VARIANTS)
def test_gemv_act_order(cuda_ok, BITS, M, variant):
    for N, K, g, sym in ((512, 1024, 128, False), (256, 512, 32, True)):
        fmt, packed, xd, y_ref, B = oracle_case(BITS, N, K, M, g, sym, True, "gemv8-act")
        assert_within(W.gemv(fmt, packed, xd, **variant_kw(variant)).cpu().numpy(), y_ref, B)


@pytest.mark.parametrize("rows16", [2, 4, 8])
@pytest.mark.parametrize("ksplit", [1, 2, 4, 8, 16])
def test_gemv_every_launch_shape(cuda_ok, BITS, rows16, ksplit):
    fmt, packed, xd, y_ref, B = oracle_case(BITS, 256, 2048, 3, 64, False, False, "gemv8-plan")
    for variant in GEMV_VARIANTS:
        y = W.gemv(fmt, packed, xd, shape=rows16, ksplit=ksplit, **variant_kw(variant)).cpu().numpy()
        assert_within(y, y_ref, B)


def exact_integer_case(BITS, seed, N, K, M):
    """s = 1, z = 2^(b-1), every code, x in {-1, 0, 1} with 16 nonzeros per
    row: |y| <= 16 * 128, an integer fp16 holds exactly, so every summation
    order gives the same result."""
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 1 << BITS, (N, K)).astype(np.uint8)
    s = np.ones((N, K // 128), dtype=np.float16)
    z = np.full((N, K // 128), 1 << (BITS - 1), dtype=np.uint8)
    x = np.zeros((M, K), dtype=np.float16)
    for m in range(M):
        nz = rng.choice(K, 16, replace=False)
        x[m, nz] = rng.choice([-1.0, 1.0], 16)
    y_ref, _ = O.linear_ref(x, O.dequant(q, s, z, 128))
    fmt = fmtb(BITS, N, K, 128, False, False)
    return fmt, pack_oracle(fmt, q, s, z), to_dev(x), y_ref


@pytest.mark.parametrize("variant", GEMV_VARIANTS)
def test_gemv_exact_integer_case(cuda_ok, BITS, variant):
    for M in (1, 16):
        fmt, packed, xd, y_ref = exact_integer_case(BITS, 15, 384, 2048, M)
        y = W.gemv(fmt, packed, xd, **variant_kw(variant)).cpu().numpy().astype(np.float64)
        assert np.array_equal(y, y_ref)


def test_gemv_full_size_sampled_rows(cuda_ok, BITS):
    """11008 x 4096 (an MLP projection of a 7B decoder) at batch one, quantized
    on the GPU; the oracle checks sampled rows."""
    N, K = 11008, 4096
    seed = synth.seed_for("w8-full", N, K)
    Wd = synth.weights_cuda(N, K, seed)
    xd = synth.activations_cuda(1, K, synth.LLAMA2_7B_OUTLIER_FRAC, seed + 1)
    fmt = fmtb(BITS, N, K, 128, False, False)
    q, s, z = W.quantize_rtn(fmt, Wd)
    y = W.gemv(fmt, W.pack(fmt, q, s, z), xd).cpu().numpy()
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(seed).choice(N, 48, replace=False)]))
    qo, so, zo = O.rtn_quantize(Wd[torch.from_numpy(rows).cuda()].cpu().numpy(), 128, False, bits=BITS)
    y_ref, B = O.linear_ref(xd.cpu().numpy(), O.dequant(qo, so, zo, 128))
    assert_within(y[:, rows], y_ref, B)
    no_timeouts()


# ---------------------------------------------------------------- GEMM


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("tile", TILES)
def test_gemm_groups_and_schemes(cuda_ok, BITS, g, sym, tile):
    fmt, packed, xd, y_ref, B = oracle_case(BITS, 512, 1024, 300, g, sym, False, "gemm8")
    assert_within(W.gemm(fmt, packed, xd, tile=tile).cpu().numpy(), y_ref, B)
    no_timeouts()


@pytest.mark.parametrize("N,K,g,M", [(200, 96, 32, 33), (130, 320, 64, 257), (1, 128, 128, 1),
                                     (1000, 1152, 128, 130)])
@pytest.mark.parametrize("tile", TILES)
def test_gemm_ragged_shapes(cuda_ok, BITS, N, K, g, M, tile):
    fmt, packed, xd, y_ref, B = oracle_case(BITS, N, K, M, g, False, False, "gemm8-ragged")
    assert_within(W.gemm(fmt, packed, xd, tile=tile).cpu().numpy(), y_ref, B)
    no_timeouts()


@pytest.mark.parametrize("tile", TILES)
def test_gemm_act_order(cuda_ok, BITS, tile):
    for N, K, M, g, sym in ((512, 1024, 256, 128, False), (256, 512, 100, 32, True)):
        fmt, packed, xd, y_ref, B = oracle_case(BITS, N, K, M, g, sym, True, "gemm8-act")
        assert_within(W.gemm(fmt, packed, xd, tile=tile).cpu().numpy(), y_ref, B)
    no_timeouts()


@pytest.mark.parametrize("tile", (3, 5, 6))
@pytest.mark.parametrize("ksplit", (2, 4, 16))
def test_gemm_split_k(cuda_ok, BITS, tile, ksplit):
    for N, K, M, g in ((384, 2048, 100, 128), (130, 1024, 257, 32)):
        fmt, packed, xd, y_ref, B = oracle_case(BITS, N, K, M, g, False, False, "gemm8-splitk")
        assert_within(W.gemm(fmt, packed, xd, tile=tile, ksplit=ksplit).cpu().numpy(), y_ref, B)
    no_timeouts()


@pytest.mark.parametrize("tile", TILES)
def test_gemm_exact_integer_case(cuda_ok, BITS, tile):
    fmt, packed, xd, y_ref = exact_integer_case(BITS, 16, 384, 2048, 300)
    y = W.gemm(fmt, packed, xd, tile=tile).cpu().numpy().astype(np.float64)
    assert np.array_equal(y, y_ref)
    no_timeouts()


def test_gemm_tiles_agree(cuda_ok, BITS):
    """Without a K split every tile sums the same products in the same order."""
    fmt, packed, xd, y_ref, B = oracle_case(BITS, 1024, 2048, 512, 128, False, False, "gemm8-agree")
    a = W.gemm(fmt, packed, xd, tile=1).cpu().numpy()
    for tile in TILES:
        assert np.array_equal(bits16(W.gemm(fmt, packed, xd, tile=tile).cpu().numpy()), bits16(a)), tile
    assert_within(a, y_ref, B)
    no_timeouts()


def test_gemm_prefill_full_size_act_order(cuda_ok, BITS):
    """4096 x 4096 at 2048 tokens with act order; oracle on sampled token rows."""
    N = K = 4096
    M = synth.PREFILL_M
    xd = synth.activations_cuda(M, K, 0.01, synth.seed_for("w8-prefill", "x", N, K))
    x = xd.cpu().numpy()
    gidx = synth.act_order_g_idx(x, 128)
    fmt = fmtb(BITS, N, K, 128, False, True)
    Wd = synth.weights_cuda(N, K, synth.seed_for("w8-prefill", "w", N, K))
    q, s, z = W.quantize_rtn(fmt, Wd, gidx)
    y = W.gemm(fmt, W.pack(fmt, q, s, z, gidx), xd).cpu().numpy()
    no_timeouts()
    qo, so, zo = O.rtn_quantize(Wd.cpu().numpy(), 128, False, gidx, bits=BITS)
    assert np.array_equal(q.cpu().numpy(), qo)
    rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(7).choice(M, 8, replace=False)]))
    y_ref, B = O.linear_ref(x[rows], O.dequant(qo, so, zo, 128, gidx))
    assert_within(y[rows], y_ref, B)
