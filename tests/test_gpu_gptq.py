"""GPTQ on the GPU (w4a16_gptq) against the CPU oracle.

Both sides compute in fp64, so the codes, scales and zero points agree with
the oracle's; the column blocks of the GPU version add the same updates in
another order, which could only tip a value lying within ~1e-15 of a rounding
boundary (allowed: at most 0.01 % of the codes, each off by one). A layer
quantized on the GPU then runs through pack / GEMV / GEMM within the usual
bound.
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


def assert_codes_match(q, qo):
    diff = q != qo
    assert diff.sum() <= max(1, q.size // 10000), int(diff.sum())
    assert np.all(np.abs(q.astype(int) - qo.astype(int))[diff] == 1)


@pytest.mark.parametrize("bits", [3, 4, 8])
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("act", [False, True])
@pytest.mark.parametrize("g", [32, 128])
def test_matches_oracle(cuda_ok, bits, sym, act, g):
    N, K, T = 160, 512, 384
    W16 = synth.weights_np(N, K, synth.seed_for("gptq", bits, sym, act, g))
    x = synth.activations_np(T, K, 0.02, synth.seed_for("gptq-x", K))
    fmt = W.make_format(N, K, g, sym, act, bits=bits)
    q, s, z, gidx = W.gptq(fmt, to_dev(W16), to_dev(x))
    qo, so, zo, gidx_o = O.gptq_quantize(W16, x, g, sym, bits, act)
    assert_codes_match(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), so.view(np.uint16))
    if not sym:
        assert np.array_equal(z.cpu().numpy(), zo)
    if act:
        assert np.array_equal(gidx.astype(np.int64), gidx_o)
    else:
        assert gidx is None


def test_uncorrelated_inputs_give_the_rtn_quantizer(cuda_ok):
    """X = I: no error feedback; the GPU GPTQ equals the GPU round-to-nearest quantizer."""
    N, K = 200, 256
    W16 = to_dev(synth.weights_np(N, K, 91))
    x = to_dev(np.eye(K, dtype=np.float16))
    for sym in (False, True):
        fmt = W.make_format(N, K, 128, sym, False)
        q, s, z, _ = W.gptq(fmt, W16, x)
        qr, sr, zr = W.quantize_rtn(fmt, W16)
        assert torch.equal(q, qr) and torch.equal(s, sr)
        if not sym:
            assert torch.equal(z, zr)


def test_dead_channels_and_damping(cuda_ok):
    """Channels whose activations are all zero, and a larger damping factor."""
    N, K, T = 64, 256, 200
    W16 = synth.weights_np(N, K, 92)
    x = synth.activations_np(T, K, 0.02, 93)
    x[:, [0, 5, 77, 255]] = 0
    for damp in (0.01, 0.5):
        fmt = W.make_format(N, K, 64, False, True)
        q, s, z, gidx = W.gptq(fmt, to_dev(W16), to_dev(x), damp=damp)
        qo, so, zo, go = O.gptq_quantize(W16, x, 64, False, 4, True, damp=damp)
        assert_codes_match(q.cpu().numpy(), qo)
        assert np.array_equal(gidx.astype(np.int64), go)


def test_layer_4096_matches_oracle_and_beats_rtn(cuda_ok):
    """A 7B-width projection (K = 4096) with act order on 512 rows: oracle
    parity, then the layer error on the calibration set below RTN's."""
    N, K, T = 512, 4096, 1024
    W16 = synth.weights_np(N, K, 94)
    x = synth.activations_np(T, K, 0.01, 95)
    fmt = W.make_format(N, K, 128, False, True)
    q, s, z, gidx = W.gptq(fmt, to_dev(W16), to_dev(x))
    qo, so, zo, go = O.gptq_quantize(W16, x, 128, False, 4, True)
    qn = q.cpu().numpy()
    assert_codes_match(qn, qo)
    assert np.array_equal(gidx.astype(np.int64), go)
    e_gptq = O.layer_error(W16, O.dequant(qn, s.cpu().numpy(), z.cpu().numpy(), 128, gidx), x)
    fr = W.make_format(N, K, 128)
    qr, sr, zr = W.quantize_rtn(fr, to_dev(W16))
    e_rtn = O.layer_error(W16, O.dequant(qr.cpu().numpy(), sr.cpu().numpy(), zr.cpu().numpy(), 128), x)
    assert e_gptq < 0.9 * e_rtn, (e_gptq, e_rtn)


@pytest.mark.parametrize("bits", [3, 4, 8])
def test_gptq_layer_through_pack_gemv_and_gemm(cuda_ok, bits):
    N, K, T = 384, 1024, 512
    W16 = synth.weights_np(N, K, 96)
    x_cal = synth.activations_np(T, K, 0.02, 97)
    fmt = W.make_format(N, K, 128, False, True, bits=bits)
    q, s, z, gidx = W.gptq(fmt, to_dev(W16), to_dev(x_cal))
    packed = W.pack(fmt, q, s, z, gidx)
    w_hat = O.dequant(q.cpu().numpy(), s.cpu().numpy(), z.cpu().numpy(), 128, gidx)
    assert np.array_equal(W.dequant(fmt, packed).cpu().numpy().view(np.uint16), w_hat.view(np.uint16))
    for M in (1, 16, 300):
        x = synth.activations_np(M, K, 0.02, 98 + M)
        y_ref, B = O.linear_ref(x, w_hat)
        y = (W.gemv if M <= 16 else W.gemm)(fmt, packed, to_dev(x)).cpu().numpy().astype(np.float64)
        r = O.error_ratio(y, y_ref, B)
        assert r.max() <= 1.0, r.max()
    assert W.pipeline_timeouts() == 0
