"""Bit-exact GPU tests of quantize / pack / dequant against the CPU oracle."""

import numpy as np
import pytest
import torch

from oracle import w4a16_oracle as O
from weight_only_bit_04_b300 import synth
from weight_only_bit_04_b300 import w4a16 as W

pytestmark = pytest.mark.gpu


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def pack_from_oracle(fmt, q, s, z, g_idx=None):
    return W.pack(fmt, to_dev(q), to_dev(s), None if fmt.symmetric else to_dev(z), g_idx)


def bits16(a):
    return np.asarray(a).view(np.uint16)


@pytest.mark.parametrize("N,K,g,sym,act", [
    (256, 512, 128, False, False),   # single linear, batch 1 shape
    (200, 96, 32, False, False),     # ragged rows and columns
    (136, 192, 64, True, False),
    (130, 256, 128, False, True),    # act order
    (64, 384, 64, True, True),
])
def test_pack_then_dequant_is_bit_exact(cuda_ok, N, K, g, sym, act):
    W16 = synth.weights_np(N, K, synth.seed_for("fmt", N, K, g, sym, act))
    x = synth.activations_np(4, K, 0.01, synth.seed_for("fmt-x", K))
    gidx = synth.act_order_g_idx(x, g) if act else None
    q, s, z = O.rtn_quantize(W16, g, sym, gidx)
    fmt = W.make_format(N, K, g, sym, act)
    packed = pack_from_oracle(fmt, q, s, z, gidx)
    got = W.dequant(fmt, packed).cpu().numpy()
    want = O.dequant(q, s, z, g, gidx)
    assert np.array_equal(bits16(got), bits16(want))


def test_dequant_exhaustive_table(cuda_ok):
    """Every code q, every zero z and every finite fp16 scale s (bit patterns)."""
    allbits = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    svals = allbits.view(np.float16)
    svals = svals[np.isfinite(svals)]
    assert svals.size == 63488
    g, K = 32, 2048
    G = K // g
    pairs = svals.size * 16                      # (s, z) pairs, one group each
    N = -(-pairs // G)
    s_flat = np.zeros(N * G, dtype=np.float16)
    z_flat = np.zeros(N * G, dtype=np.uint8)
    s_flat[:pairs] = np.repeat(svals, 16)
    z_flat[:pairs] = np.tile(np.arange(16, dtype=np.uint8), svals.size)
    s = s_flat.reshape(N, G)
    z = z_flat.reshape(N, G)
    q = np.tile(np.arange(16, dtype=np.uint8), (N, K // 16))  # each group holds q = 0..15 twice
    fmt = W.make_format(N, K, g, False, False)
    packed = pack_from_oracle(fmt, q, s, z)
    got = W.dequant(fmt, packed).cpu().numpy()
    with np.errstate(over="ignore"):
        want = O.dequant(q, s, z, g)
    assert np.array_equal(bits16(got), bits16(want))


def test_pack_every_nibble_position(cuda_ok):
    """Each code value at each row/column position of a 128 x 64 tile, via dequant with s=1, z=0."""
    N, K, g = 128, 64, 32
    rng = np.random.default_rng(0)
    for _ in range(4):
        q = rng.integers(0, 16, (N, K)).astype(np.uint8)
        s = np.ones((N, K // g), dtype=np.float16)
        z = np.zeros((N, K // g), dtype=np.uint8)
        fmt = W.make_format(N, K, g, False, False)
        got = W.dequant(fmt, pack_from_oracle(fmt, q, s, z)).cpu().numpy()
        assert np.array_equal(got.astype(np.int64), q.astype(np.int64))


@pytest.mark.parametrize("N,K,g,sym,act", [
    (256, 512, 128, False, False),
    (96, 256, 32, False, False),
    (64, 384, 64, True, False),
    (128, 512, 128, False, True),
    (40, 256, 64, True, True),
])
def test_gpu_rtn_matches_oracle_bit_exactly(cuda_ok, N, K, g, sym, act):
    W16 = synth.weights_np(N, K, synth.seed_for("rtn", N, K, g, sym, act))
    # special groups: constant (s = 0 -> 1), exact rounding ties, one-signed
    W16[0, :g] = np.float16(0.25)
    W16[1, :8] = np.array([-7.0, 8.0, 2.5, 3.5, -0.5, 0.5, -1.5, 1.5], dtype=np.float16)
    W16[1, 8:g] = np.float16(0.0)
    W16[2, :g] = np.abs(W16[2, :g]) + np.float16(0.01)
    x = synth.activations_np(2, K, 0.01, synth.seed_for("rtn-x", K))
    gidx = synth.act_order_g_idx(x, g) if act else None
    fmt = W.make_format(N, K, g, sym, act)
    q, s, z = W.quantize_rtn(fmt, to_dev(W16), gidx)
    qo, so, zo = O.rtn_quantize(W16, g, sym, gidx)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(bits16(s.cpu().numpy()), bits16(so))
    if not sym:
        assert np.array_equal(z.cpu().numpy(), zo)
