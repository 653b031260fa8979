"""Pins of the oracle's unfolded-AWQ step (CPU only).

"The two algorithms, compactly" (AWQ + GPTQ Quantization, in depth): AWQ
enlarges the weights of the salient input channels by a factor s > 1 before
quantizing and shrinks those activation channels by s to compensate. These tests fix the
oracle's version of that step against exact rational arithmetic, against the
plain layer where the mathematics says the two must agree exactly, against a
pure-Python restatement, and check the scale search's invariants.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import brute
from oracle import w4a16_oracle as O
from weight_only_bit_04_b300 import synth

# every finite fp16 value, ascending, as exact fractions and bit patterns
_BITS = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
_VALS = _BITS.view(np.float16)
_FIN = np.isfinite(_VALS)
_ORDER = np.argsort(_VALS[_FIN].astype(np.float64), kind="stable")
F16_SORTED = _VALS[_FIN].astype(np.float64)[_ORDER]
F16_BITS = _BITS[_FIN][_ORDER]


def exact_round_fp16(v: Fraction) -> float:
    """Nearest finite fp16 to the exact rational v, ties to the even pattern."""
    i = int(np.searchsorted(F16_SORTED, float(v)))
    cands = sorted({j for j in (i - 2, i - 1, i, i + 1) if 0 <= j < F16_SORTED.size})
    dist = {j: abs(Fraction(F16_SORTED[j]) - v) for j in cands}
    d = min(dist.values())
    ties = [j for j in cands if dist[j] == d]
    if len(ties) > 1:
        ties = [j for j in ties if F16_BITS[j] % 2 == 0] or ties
    return float(F16_SORTED[ties[0]])


def sample_fp16(rng, n, lo_exp=-20, hi_exp=12):
    """Values spread over fp16 magnitudes (subnormal to large), random signs."""
    mags = 2.0 ** rng.uniform(lo_exp, hi_exp, n)
    return (rng.choice([-1.0, 1.0], n) * mags).astype(np.float16)


def test_activation_division_is_the_exactly_rounded_quotient():
    rng = np.random.default_rng(31)
    x = sample_fp16(rng, 3000)
    s = np.abs(sample_fp16(rng, 3000, -6, 6))
    s[s == 0] = np.float16(1.0)
    with np.errstate(over="ignore"):
        got = O.awq_scale_activations(x[None, :], s)[0].astype(np.float64)
    checked = 0
    for i in range(x.size):
        v = Fraction(float(x[i])) / Fraction(float(s[i]))
        if abs(v) >= 65520:  # rounds to infinity (IEEE overflow)
            assert np.isinf(got[i])
            continue
        want = exact_round_fp16(v)
        assert got[i] == want, (x[i], s[i], got[i], want)
        checked += 1
    assert checked > 2500


def test_weight_product_is_the_exactly_rounded_product():
    rng = np.random.default_rng(32)
    W = sample_fp16(rng, 3000, -20, 8)
    s = np.abs(sample_fp16(rng, 3000, -4, 4))
    s[s == 0] = np.float16(1.0)
    with np.errstate(over="ignore"):
        got = O.awq_scale_weights(W[None, :], s)[0].astype(np.float64)
    for i in range(W.size):
        v = Fraction(float(W[i])) * Fraction(float(s[i]))
        if abs(v) >= 65520:
            continue  # rounds to infinity
        assert got[i] == exact_round_fp16(v)


def test_unit_scale_is_the_plain_layer():
    N, K, M = 64, 512, 4
    W = synth.weights_np(N, K, 41)
    x = synth.activations_np(M, K, 0.01, 42)
    ones = np.ones(K, dtype=np.float16)
    for bits in (4, 8):
        y0, B0, qsz0, w0 = O.w4a16_linear(x, W, 128, False, bits=bits)
        y1, B1, qsz1, w1, xs = O.awq_linear(x, W, ones, 128, False, bits=bits)
        assert np.array_equal(y0, y1) and np.array_equal(B0, B1)
        assert all(np.array_equal(a, b) for a, b in zip(qsz0, qsz1))
        assert np.array_equal(xs, x)


def _normal_range(a, floor=2.0 ** -8):
    """Replace magnitudes below `floor` by +-floor so that scaling by 2^-5 .. 2^5
    stays in fp16's normal range (exact)."""
    a = a.copy()
    small = np.abs(a.astype(np.float64)) < floor
    a[small] = (np.where(a[small] < 0, -floor, floor)).astype(np.float16)
    return a


@pytest.mark.parametrize("exps", [(3,), (-2,), (5,), (0, 2, -1, 4)])
def test_power_of_two_scale_constant_per_group_leaves_y_unchanged(exps):
    """s[k] = 2^e with e constant on each group: the group's scale, zero point
    and codes are unchanged, w_hat is multiplied by 2^e and x divided by it,
    all exactly, so y is the plain layer's y bit for bit. A scale applied the
    wrong way (x * s or W / s) or along the wrong axis changes y."""
    N, K, M, g = 48, 512, 3, 128
    W = _normal_range(synth.weights_np(N, K, 43), 2.0 ** -6)
    x = _normal_range(synth.activations_np(M, K, 0.01, 44))
    e = np.array([exps[(k // g) % len(exps)] for k in range(K)], dtype=np.float64)
    s = (2.0 ** e).astype(np.float16)
    y0, _, (q0, s0, z0), _ = O.w4a16_linear(x, W, g, False)
    y1, _, (q1, s1, z1), _, _ = O.awq_linear(x, W, s, g, False)
    assert np.array_equal(q0, q1) and np.array_equal(z0, z1)
    assert np.array_equal(y0, y1)
    # the planted mistakes do not survive
    if any(v != 0 for v in exps):
        xs_wrong = O.fp16_rne(x.astype(np.float64) * s.astype(np.float64))
        w_hat1 = O.dequant(q1, s1, z1, g)
        assert not np.array_equal(O.linear_ref(xs_wrong, w_hat1)[0], y0)
        W_div = O.fp16_rne(W.astype(np.float64) / s.astype(np.float64))
        yq = O.w4a16_linear(O.awq_scale_activations(x, s), W_div, g, False)[0]
        assert not np.array_equal(yq, y0)


@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("act_order", [False, True])
def test_numpy_awq_matches_pure_python(sym, bits, act_order):
    N, K, M, g = 5, 96, 3, 32
    rng = np.random.default_rng(45)
    W = synth.weights_np(N, K, 46)
    x = synth.activations_np(M, K, 0.05, 47)
    s = rng.uniform(0.5, 4.0, K).astype(np.float16)
    gidx = synth.act_order_g_idx(x, g) if act_order else None
    y, B, (q, sc, z), w_hat, xs = O.awq_linear(x, W, s, g, sym, gidx, bits)
    yb, qb, sb, zb, xb = brute.awq_linear(x.astype(np.float64).tolist(), W.astype(np.float64).tolist(),
                                          s.astype(np.float64).tolist(), g, sym,
                                          None if gidx is None else gidx.tolist(), bits)
    assert q.tolist() == qb and sc.astype(np.float64).tolist() == sb and z.tolist() == zb
    assert xs.astype(np.float64).tolist() == xb
    assert np.allclose(y, np.array(yb), rtol=1e-12, atol=1e-12)


def test_mutant_unrounded_weight_product_is_caught():
    """Quantizing W * s without rounding it to fp16 first differs from the
    pure-Python restatement on some code."""
    N, K, g = 32, 512, 32
    rng = np.random.default_rng(48)
    W = synth.weights_np(N, K, 49)
    s = rng.uniform(0.5, 4.0, K).astype(np.float16)
    Ws_unrounded = W.astype(np.float64) * s.astype(np.float64)
    # the mutant: codes from the unrounded product (scale from the same values)
    qm = []
    for n in range(N):
        row = []
        for t in range(K // g):
            w = Ws_unrounded[n, t * g:(t + 1) * g]
            sc = float(O.fp16_rne((w.max() - w.min()) / 15))
            z = min(max(round(-w.min() / sc), 0), 15)
            row += [min(max(round(v / sc) + z, 0), 15) for v in w]
        qm.append(row)
    _, qb, _, _, _ = brute.awq_linear([[0.0] * K], W.astype(np.float64).tolist(),
                                      s.astype(np.float64).tolist(), g, False)
    q, _, _ = O.rtn_quantize(O.awq_scale_weights(W, s), g, False)
    assert q.tolist() == qb
    assert qm != qb


def test_search_alpha_zero_is_round_to_nearest():
    N, K, M = 32, 256, 64
    W = synth.weights_np(N, K, 50)
    x = synth.activations_np(M, K, 0.02, 51)
    s, alpha, losses = O.awq_search(W, x, 128, False, n_grid=10)
    assert losses.shape == (11,)
    _, _, _, w_hat = O.w4a16_linear(x, W, 128, False)
    xd = x.astype(np.float64)
    rtn_loss = np.linalg.norm(xd @ W.astype(np.float64).T - xd @ w_hat.astype(np.float64).T)
    assert losses[0] == rtn_loss
    assert losses.min() <= losses[0]
    assert np.isclose(losses[int(round(alpha * 10))], losses.min())
    assert s.dtype == np.float16 and np.all(s.astype(np.float64) > 0)


def test_search_protects_the_outlier_channels():
    """With a few large-activation channels (the salient 0.1-1 % of the
    section), the search picks alpha > 0, gives those channels the larger
    scales and lowers the output error below round-to-nearest."""
    N, K, M = 64, 512, 128
    W = synth.weights_np(N, K, 52)
    x = synth.activations_np(M, K, 0.01, 53)
    s, alpha, losses = O.awq_search(W, x, 128, False, n_grid=10)
    assert alpha > 0
    assert losses.min() < 0.95 * losses[0]
    s_x = np.mean(np.abs(x.astype(np.float64)), axis=0)
    top = np.argsort(s_x)[-max(1, K // 100):]
    assert s.astype(np.float64)[top].min() > np.median(s.astype(np.float64))


def test_dead_channel_keeps_unit_scale():
    N, K, M = 8, 128, 16
    W = synth.weights_np(N, K, 54)
    x = synth.activations_np(M, K, 0.05, 55)
    x[:, 7] = 0
    s, alpha, _ = O.awq_search(W, x, 128, False, n_grid=4)
    assert s[7] == np.float16(1.0)


def test_act_scale_validation():
    x = np.ones((1, 4), dtype=np.float16)
    with pytest.raises(ValueError):
        O.awq_scale_activations(x, np.array([1, 0, 1, 1], dtype=np.float16))
    with pytest.raises(ValueError):
        O.awq_scale_activations(x, np.array([1, -1, 1, 1], dtype=np.float16))
    with pytest.raises(TypeError):
        O.awq_scale_activations(x, np.ones(4, dtype=np.float32))
