"""Products at the size limits of the C ABI (N and K up to 2^20 each, the
GEMM up to 2^20 tokens) with extreme aspect ratios:
- one 128-row block over K = 2^20 columns (16384 steps of 64 columns);
- 8192 row blocks over K = 128 (two steps);
- 2^20 tokens, with and without act order.
Rows and tokens are independent, so the oracle checks sampled rows or
tokens. The GPU quantizer is checked bit for bit on the sampled rows; the
products must stay within the per-element bound
|y_gpu - y_ref| <= 2e-3 * sum_k |x * w_hat| + 1e-3."""

import numpy as np
import pytest
import torch

from oracle import w4a16_oracle as O
from weight_only_bit_04_b300 import synth
from weight_only_bit_04_b300 import w4a16 as W

pytestmark = pytest.mark.gpu

LIMIT = 1 << 20


def assert_within(y, y_ref, B):
    y = y.astype(np.float64)
    assert np.all(np.isfinite(y)), "non-finite output"
    r = O.error_ratio(y, y_ref, B)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3f} at {np.unravel_index(r.argmax(), r.shape)}"


def quantized_layer(N, K, g, seed, g_idx=None):
    Wd = synth.weights_cuda(N, K, seed)
    fmt = W.make_format(N, K, g, False, g_idx is not None)
    q, s, z = W.quantize_rtn(fmt, Wd, g_idx)
    return fmt, Wd, (q, s, z), W.pack(fmt, q, s, z, g_idx)


def oracle_rows(Wd, qsz, rows, g, g_idx=None):
    """The oracle's dequantized weights of the sampled rows, after checking
    the GPU quantizer's codes, scales and zeros on them."""
    rt = torch.from_numpy(rows).cuda()
    qo, so, zo = O.rtn_quantize(Wd[rt].cpu().numpy(), g, False, g_idx)
    q, s, z = qsz
    assert np.array_equal(q[rt].cpu().numpy(), qo)
    assert np.array_equal(s[rt].cpu().numpy().view(np.uint16), so.view(np.uint16))
    assert np.array_equal(z[rt].cpu().numpy(), zo)
    return O.dequant(qo, so, zo, g, g_idx)


def sample(n, k, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, n - 1], rng.choice(n, min(k, n), replace=False)]))


@pytest.mark.parametrize("M", [1, 16])
def test_gemv_one_row_block_longest_k(cuda_ok, M):
    N, K = 128, LIMIT
    fmt, Wd, qsz, packed = quantized_layer(N, K, 128, synth.seed_for("limit-k", M))
    xd = synth.activations_cuda(M, K, 0.01, synth.seed_for("limit-k-x", M))
    rows = sample(N, 22, 1)
    w_hat = oracle_rows(Wd, qsz, rows, 128)
    y_ref, B = O.linear_ref(xd.cpu().numpy(), w_hat)
    for kw in (dict(), dict(register_ring=True), dict(async_copy=True)):
        y = W.gemv(fmt, packed, xd, **kw).cpu().numpy()
        assert_within(y[:, rows], y_ref, B)
    assert W.pipeline_timeouts() == 0


def test_gemv_most_rows(cuda_ok):
    N, K, M = LIMIT, 128, 16
    fmt, Wd, qsz, packed = quantized_layer(N, K, 128, synth.seed_for("limit-n"))
    xd = synth.activations_cuda(M, K, 0.01, synth.seed_for("limit-n-x"))
    rows = sample(N, 256, 2)
    y_ref, B = O.linear_ref(xd.cpu().numpy(), oracle_rows(Wd, qsz, rows, 128))
    for kw in (dict(), dict(register_ring=True), dict(async_copy=True)):
        y = W.gemv(fmt, packed, xd, **kw).cpu().numpy()
        assert_within(y[:, rows], y_ref, B)
    assert W.pipeline_timeouts() == 0


@pytest.mark.parametrize("act", [False, True])
def test_gemm_most_tokens(cuda_ok, act):
    N, K, g, M = 136, 128, 32, LIMIT
    xd = synth.activations_cuda(M, K, 0.01, synth.seed_for("limit-m-x", act))
    gidx = synth.act_order_g_idx(xd.cpu().numpy(), g) if act else None
    fmt, Wd, qsz, packed = quantized_layer(N, K, g, synth.seed_for("limit-m", act), gidx)
    w_hat = oracle_rows(Wd, qsz, np.arange(N), g, gidx)
    y = W.gemm(fmt, packed, xd)
    toks = sample(M, 4096, 3)
    tt = torch.from_numpy(toks).cuda()
    y_ref, B = O.linear_ref(xd[tt].cpu().numpy(), w_hat)
    assert_within(y[tt].cpu().numpy(), y_ref, B)
    assert W.pipeline_timeouts() == 0


def test_gemm_longest_k(cuda_ok):
    N, K, M = 128, LIMIT, 32
    fmt, Wd, qsz, packed = quantized_layer(N, K, 128, synth.seed_for("limit-gemm-k"))
    xd = synth.activations_cuda(M, K, 0.01, synth.seed_for("limit-gemm-k-x"))
    rows = sample(N, 14, 4)
    y_ref, B = O.linear_ref(xd.cpu().numpy(), oracle_rows(Wd, qsz, rows, 128))
    for kw in (dict(), dict(tile=3), dict(tile=6, ksplit=16)):
        y = W.gemm(fmt, packed, xd, **kw).cpu().numpy()
        assert_within(y[:, rows], y_ref, B)
    assert W.pipeline_timeouts() == 0
