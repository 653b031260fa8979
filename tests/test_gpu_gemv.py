"""GEMV (1 <= M <= 16) parity against the CPU oracle, element by element.

Acceptance per element: |y_gpu - y_ref| <= 2e-3 * sum_k |x * w_hat| + 1e-3,
with y_ref the fp64 product of x and the oracle's dequantized weights.
"""

import numpy as np
import pytest
import torch

from oracle import w4a16_oracle as O
from weight_only_bit_04_b300 import synth
from weight_only_bit_04_b300 import w4a16 as W

pytestmark = pytest.mark.gpu


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# register ring / register ring with staged activations / asynchronous-copy ring
# / asynchronous-copy ring with staged activations
VARIANTS = ("ring", "ring_sx", "async", "async_sx")


def variant_kw(variant):
    return dict(register_ring=variant.startswith("ring"), async_copy=variant.startswith("async"),
                stage_activations=variant.endswith("_sx"))


def run_case(N, K, M, g, sym, act, frac=0.01, tag="gemv", shape=0, ksplit=0, variant="ring"):
    W16 = synth.weights_np(N, K, synth.seed_for(tag, "w", N, K, g, sym, act))
    x = synth.activations_np(M, K, frac, synth.seed_for(tag, "x", M, K))
    gidx = synth.act_order_g_idx(x, g) if act else None
    y_ref, B, (q, s, z), _ = O.w4a16_linear(x, W16, g, sym, gidx)
    fmt = W.make_format(N, K, g, sym, act)
    packed = W.pack(fmt, to_dev(q), to_dev(s), None if sym else to_dev(z), gidx)
    y = W.gemv(fmt, packed, to_dev(x), shape=shape, ksplit=ksplit, **variant_kw(variant))
    torch.cuda.synchronize()
    return y.cpu().numpy(), y_ref, B


def assert_within(y, y_ref, B):
    r = O.error_ratio(y.astype(np.float64), y_ref, B)
    assert np.all(np.isfinite(y)), "non-finite output"
    assert r.max() <= 1.0, f"max error ratio {r.max():.3f} at {np.unravel_index(r.argmax(), r.shape)}"


@pytest.mark.parametrize("variant", VARIANTS)
def test_single_linear_batch1(cuda_ok, variant):
    y, y_ref, B = run_case(256, 512, 1, 128, False, False, tag="single", variant=variant)
    assert_within(y, y_ref, B)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 7, 8, 9, 12, 16])
@pytest.mark.parametrize("variant", VARIANTS)
def test_token_counts(cuda_ok, M, variant):
    y, y_ref, B = run_case(384, 1024, M, 128, False, False, variant=variant)
    assert_within(y, y_ref, B)


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("variant", VARIANTS)
def test_group_sizes_and_schemes(cuda_ok, g, sym, M, variant):
    y, y_ref, B = run_case(256, 1024, M, g, sym, False, variant=variant)
    assert_within(y, y_ref, B)


@pytest.mark.parametrize("N,K,g", [(200, 96, 32), (130, 320, 64), (1, 128, 128), (17, 64, 32),
                                   (1000, 1152, 128)])
@pytest.mark.parametrize("variant", VARIANTS)
def test_ragged_shapes(cuda_ok, N, K, g, variant):
    for M in (1, 5):
        y, y_ref, B = run_case(N, K, M, g, False, False, tag="ragged", variant=variant)
        assert_within(y, y_ref, B)


@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("variant", VARIANTS)
def test_act_order(cuda_ok, M, variant):
    y, y_ref, B = run_case(512, 1024, M, 128, False, True, tag="act", variant=variant)
    assert_within(y, y_ref, B)
    y, y_ref, B = run_case(256, 512, M, 32, True, True, tag="act", variant=variant)
    assert_within(y, y_ref, B)


@pytest.mark.parametrize("rows16", [2, 4, 8])
@pytest.mark.parametrize("ksplit", [1, 2, 4, 8, 16])
def test_every_register_ring_launch_shape(cuda_ok, rows16, ksplit):
    for variant in VARIANTS:
        y, y_ref, B = run_case(256, 2048, 3, 64, False, False, tag="plan", shape=rows16, ksplit=ksplit,
                               variant=variant)
        assert_within(y, y_ref, B)


@pytest.mark.parametrize("variant", VARIANTS)
def test_exact_integer_special_case(cuda_ok, variant):
    """s = 1, z = 8, x in {-1, 0, 1} with <= 128 nonzeros per row: y is exact."""
    rng = np.random.default_rng(5)
    N, K = 384, 2048
    for M in (1, 8, 16):
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
        y = W.gemv(fmt, packed, to_dev(x), **variant_kw(variant)).cpu().numpy().astype(np.float64)
        assert np.array_equal(y, y_ref)


def test_deterministic(cuda_ok):
    N, K = 1024, 4096
    W16 = synth.weights_np(N, K, 77)
    x = synth.activations_np(4, K, 0.01, 78)
    fmt = W.make_format(N, K, 128, False, False)
    q, s, z = W.quantize_rtn(fmt, to_dev(W16))
    packed = W.pack(fmt, q, s, z)
    xd = to_dev(x)
    a = W.gemv(fmt, packed, xd).cpu().numpy()
    for _ in range(3):
        assert np.array_equal(W.gemv(fmt, packed, xd).cpu().numpy().view(np.uint16), a.view(np.uint16))


def _sampled_layer_parity(N, K, M, frac, tag, n_rows=64):
    """Full-size layer on the GPU; oracle on sampled rows (rows are independent)."""
    seed = synth.seed_for(tag, N, K)
    Wd = synth.weights_cuda(N, K, seed)
    xd = synth.activations_cuda(M, K, frac, seed + 1)
    fmt = W.make_format(N, K, 128, False, False)
    q, s, z = W.quantize_rtn(fmt, Wd)
    packed = W.pack(fmt, q, s, z)
    y = W.gemv(fmt, packed, xd).cpu().numpy()
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, N - 1], rng.choice(N, n_rows, replace=False)]))
    Wr = Wd[torch.from_numpy(rows).cuda()].cpu().numpy()
    qo, so, zo = O.rtn_quantize(Wr, 128, False)
    # the GPU quantizer agrees with the oracle on the sampled rows
    rows_t = torch.from_numpy(rows).cuda()
    assert np.array_equal(q[rows_t].cpu().numpy(), qo)
    assert np.array_equal(s[rows_t].cpu().numpy().view(np.uint16), so.view(np.uint16))
    assert np.array_equal(z[rows_t].cpu().numpy(), zo)
    y_ref, B = O.linear_ref(xd.cpu().numpy(), O.dequant(qo, so, zo, 128))
    assert_within(y[:, rows], y_ref, B)


@pytest.mark.parametrize("name,N,K", [(n, a, b) for n, a, b in synth.LLAMA2_7B_LINEARS[::3]] +
                         [("down", 4096, 11008)])
def test_llama2_7b_layer_shapes(cuda_ok, name, N, K):
    _sampled_layer_parity(N, K, 1, synth.LLAMA2_7B_OUTLIER_FRAC, "7b-" + name)


@pytest.mark.parametrize("name,N,K", [("k", 1024, 8192), ("gate", 28672, 8192), ("down", 8192, 28672)])
def test_llama_70b_layer_shapes(cuda_ok, name, N, K):
    _sampled_layer_parity(N, K, 1, synth.LLAMA_70B_OUTLIER_FRAC, "70b-" + name)


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_8192_square_sweep_gemv_part(cuda_ok, M):
    _sampled_layer_parity(8192, 8192, M, 0.01, "sweep", n_rows=32)


def test_weights_ready_flag_matches_default(cuda_ok):
    """Early weight streaming (weights packed and synchronised beforehand)."""
    N, K = 1024, 4096
    W16 = synth.weights_np(N, K, 91)
    x = synth.activations_np(8, K, 0.01, 92)
    y_ref, B, (q, s, z), _ = O.w4a16_linear(x, W16, 128, False)
    fmt = W.make_format(N, K, 128, False, False)
    packed = W.pack(fmt, to_dev(q), to_dev(s), to_dev(z))
    torch.cuda.synchronize()
    xd = to_dev(x)
    a = W.gemv(fmt, packed, xd).cpu().numpy()
    for _ in range(3):
        b = W.gemv(fmt, packed, xd, weights_ready=True)
    assert np.array_equal(b.cpu().numpy().view(np.uint16), a.view(np.uint16))
    assert_within(a, y_ref, B)


def test_inputs_ready_chain_matches(cuda_ok):
    """GEMVs that read the same activations, launched without waiting for one
    another (inputs ready), give the same outputs as when each waits."""
    N, K = 1024, 4096
    x = synth.activations_np(1, K, 0.01, 93)
    xd = to_dev(x)
    packs, fmt = [], W.make_format(N, K, 128, False, False)
    for i in range(3):
        q, s, z = W.quantize_rtn(fmt, to_dev(synth.weights_np(N, K, 94 + i)))
        packs.append(W.pack(fmt, q, s, z))
    torch.cuda.synchronize()
    ref = [W.gemv(fmt, p, xd).cpu().numpy() for p in packs]
    for variant in VARIANTS:
        outs = [torch.empty((1, N), dtype=torch.float16, device="cuda") for _ in packs]
        for i, p in enumerate(packs):
            W.gemv(fmt, p, xd, out=outs[i], inputs_ready=i > 0, weights_ready=True, **variant_kw(variant))
        torch.cuda.synchronize()
        for i, (o, r) in enumerate(zip(outs, ref)):
            got = o.cpu().numpy()
            if variant == "ring":  # the default kernel of this shape: same kernel, same order
                assert np.array_equal(got.view(np.uint16), r.view(np.uint16))
            else:
                q, s, z = O.rtn_quantize(synth.weights_np(N, K, 94 + i), 128, False)
                y_ref, B = O.linear_ref(x, O.dequant(q, s, z, 128))
                assert_within(got, y_ref, B)
    assert W.pipeline_timeouts() == 0


def test_default_picks_async_ring_for_large_layers(cuda_ok):
    """The default plan switches kernels at 64 row blocks; both sides match the oracle."""
    for N in (8064, 8192):
        K = 1024
        y, y_ref, B = run_case(N, K, 1, 128, False, False, tag="switch")
        assert_within(y, y_ref, B)
