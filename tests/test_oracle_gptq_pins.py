"""Pins of the oracle's GPTQ step (CPU only).

"The two algorithms, compactly" (AWQ + GPTQ Quantization, in depth): GPTQ
quantizes one column at a time and, with weights from the inverse of H = 2 X X^T,
pushes each column's rounding error onto the columns not yet quantized. The
oracle follows the page's Cholesky formulation; these tests tie it to an
independent restatement (after every column, the remaining weights are the
least-squares optimum of the damped quadratic error given the columns fixed
so far), to closed forms and limits, and to the method's purpose (a lower
layer-output error than round-to-nearest).
"""

import numpy as np
import pytest

from oracle import w4a16_oracle as O
from weight_only_bit_04_b300 import synth


def block_solve_gptq(W, x, g, sym, bits=4, act_order=False, damp=O.GPTQ_DAMP):
    """GPTQ restated without the Cholesky factor: after fixing columns f,
    the remaining columns r take w_r + delta_r with
    delta_r = -delta_f H_fr H_rr^-1 (the minimiser of the damped quadratic
    error (dw) H (dw)^T over the free columns)."""
    N, K = W.shape
    H = O.gptq_hessian(x)
    order = O.gptq_order(H, act_order)
    Hd = O.gptq_damped(H, damp)[np.ix_(order, order)]
    W0 = W.astype(np.float64)[:, order]
    cur = W0.copy()
    fixed_vals = np.zeros_like(W0)
    q = np.zeros((N, K), dtype=np.uint8)
    scales = np.zeros((N, K // g), dtype=np.float16)
    zeros = np.zeros((N, K // g), dtype=np.uint8)
    for j in range(K):
        t = j // g
        if j % g == 0:
            s, z = O.group_scale_zero(cur[:, j:j + g], sym, bits)
            scales[:, t], zeros[:, t] = s, z
        sd = scales[:, t].astype(np.float64)
        zd = zeros[:, t].astype(np.float64)
        if sym and bits == 8:
            qj = O.sym8_codes(cur[:, j:j + 1], sd[:, None])[:, 0]
        else:
            qj = O.quantize_codes(cur[:, j], sd, zd, bits)
        fixed_vals[:, j] = (qj.astype(np.float64) - zd) * sd
        q[:, order[j]] = qj
        f, r = np.arange(j + 1), np.arange(j + 1, K)
        if r.size:
            delta_f = fixed_vals[:, f] - W0[:, f]
            rhs = delta_f @ Hd[np.ix_(f, r)]                       # [N, |r|]
            delta_r = -np.linalg.solve(Hd[np.ix_(r, r)], rhs.T).T  # H_rr symmetric
            cur[:, r] = W0[:, r] + delta_r
    return q, scales, zeros


@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("act_order", [False, True])
@pytest.mark.parametrize("bits", [3, 4, 8])
def test_cholesky_form_equals_least_squares_restatement(sym, act_order, bits):
    N, K, T, g = 12, 32, 96, 8
    W = synth.weights_np(N, K, synth.seed_for("gptq-ls", sym, act_order, bits))
    x = synth.activations_np(T, K, 0.1, synth.seed_for("gptq-ls-x", K))
    q, s, z, gidx = O.gptq_quantize(W, x, g, sym, bits, act_order)
    qb, sb, zb = block_solve_gptq(W, x, g, sym, bits, act_order)
    assert np.array_equal(s.view(np.uint16), sb.view(np.uint16))
    assert np.array_equal(z, zb)
    assert np.array_equal(q, qb)


def test_uncorrelated_inputs_give_round_to_nearest():
    """X = I (every token one channel): H = 2I is diagonal, so is H^-1 and its
    Cholesky factor: no error feedback, GPTQ is round-to-nearest exactly."""
    N, K, g = 16, 64, 32
    W = synth.weights_np(N, K, 61)
    x = np.eye(K, dtype=np.float16)
    for sym in (False, True):
        q, s, z, gidx = O.gptq_quantize(W, x, g, sym, 4, act_order=True)
        qr, sr, zr = O.rtn_quantize(W, g, sym)
        assert gidx is not None and np.array_equal(gidx, np.arange(K) // g)  # equal diagonals: natural order
        assert np.array_equal(q, qr) and np.array_equal(s.view(np.uint16), sr.view(np.uint16))
        assert np.array_equal(z, zr)


def test_two_column_update_closed_form():
    """Two columns, one group each: after column 0 is rounded to w0_hat,
    column 1 moves by (w0 - w0_hat) * H01 / H11 (damped H), the optimal
    compensation for a fixed error in column 0."""
    x = np.array([[1.0, 0.5], [0.5, 2.0], [2.0, -1.0], [0.25, 0.75]], dtype=np.float16)
    W = np.array([[0.3, -0.7], [1.1, 0.2]], dtype=np.float16)
    H = O.gptq_damped(O.gptq_hessian(x))
    q, s, z, _ = O.gptq_quantize(W, x, 1, False, 4)
    for n in range(2):
        w0_hat = (float(q[n, 0]) - float(z[n, 0])) * float(s[n, 0])
        w1_cur = float(W[n, 1]) + (float(W[n, 0]) - w0_hat) * H[0, 1] / H[1, 1]
        # a one-member group reproduces its value: s = 0 -> 1, z = rint(-w), q = rint(w) + z
        s1, z1 = O.group_scale_zero(np.array([[w1_cur]]), False, 4)
        assert float(s[n, 1]) == float(s1[0]) and int(z[n, 1]) == int(z1[0])
        assert int(q[n, 1]) == int(O.quantize_codes(w1_cur, float(s1[0]), float(z1[0]), 4))


def test_large_damping_tends_to_round_to_nearest():
    N, K, T, g = 16, 128, 256, 32
    W = synth.weights_np(N, K, 62)
    x = synth.activations_np(T, K, 0.02, 63)
    q, s, z, _ = O.gptq_quantize(W, x, g, False, 4, damp=1e9)
    qr, sr, zr = O.rtn_quantize(W, g, False)
    assert np.array_equal(s.view(np.uint16), sr.view(np.uint16)) and np.array_equal(z, zr)
    # codes agree except where w / s sits exactly on a rounding tie, which the
    # 1e-9-relative feedback may tip either way (to a neighbouring code)
    ratio = W.astype(np.float64) / np.repeat(sr.astype(np.float64), g, axis=1)
    tie = np.abs(ratio - np.floor(ratio) - 0.5) == 0
    diff = q != qr
    assert np.all(tie[diff]) and np.all(np.abs(q.astype(int) - qr.astype(int))[diff] == 1)
    assert diff.sum() < 0.01 * q.size


def test_gptq_lowers_the_layer_error_and_act_order_lowers_it_more():
    """The method's purpose: on the calibration inputs the GPTQ layer's output
    error is below round-to-nearest's; act order, which quantizes the
    largest-activation columns early, when most columns are still free to take
    up their error, lowers it further (synthetic inputs with 2 %
    outlier channels, otherwise uncorrelated: about -11 % and -23 %)."""
    N, K, T, g = 64, 256, 512, 128
    W = synth.weights_np(N, K, 64)
    x = synth.activations_np(T, K, 0.02, 65)
    err = {}
    for act in (False, True):
        q, s, z, gidx = O.gptq_quantize(W, x, g, False, 4, act)
        err[act] = O.layer_error(W, O.dequant(q, s, z, g, gidx), x)
    qr, sr, zr = O.rtn_quantize(W, g, False)
    e_rtn = O.layer_error(W, O.dequant(qr, sr, zr, g), x)
    assert err[False] < 0.95 * e_rtn, (err, e_rtn)
    assert err[True] < 0.85 * e_rtn and err[True] < err[False], (err, e_rtn)


def test_act_order_map_is_a_group_map_in_descending_diag_order():
    N, K, T, g = 8, 256, 128, 64
    W = synth.weights_np(N, K, 66)
    x = synth.activations_np(T, K, 0.02, 67)
    q, s, z, gidx = O.gptq_quantize(W, x, g, True, 4, act_order=True)
    O.group_map(K, g, gidx)  # exactly g members per group
    d = np.diag(O.gptq_hessian(x))
    order = np.argsort(-d, kind="stable")
    assert np.array_equal(gidx[order], np.arange(K) // g)
    # the act-order map of the synthetic workloads is the same ranking (d_j = 2 sum_t x_tj^2)
    assert np.array_equal(gidx, synth.act_order_g_idx(x, g))


def test_mutants_are_caught():
    N, K, T, g = 12, 32, 96, 8
    W = synth.weights_np(N, K, 68)
    x = synth.activations_np(T, K, 0.1, 69)
    qb, sb, zb = block_solve_gptq(W, x, g, False)
    good = O.gptq_quantize(W, x, g, False)[0]
    assert np.array_equal(good, qb)
    # feedback with the wrong sign, or without the 1 / U[j, j] normalisation
    H = O.gptq_hessian(x)
    Hd = O.gptq_damped(H)
    U = O.gptq_factor(Hd)
    for variant in ("sign", "norm"):
        Wp = W.astype(np.float64).copy()
        qm = np.zeros((N, K), dtype=np.uint8)
        for j in range(K):
            t = j // g
            if j % g == 0:
                s, z = O.group_scale_zero(Wp[:, j:j + g], False, 4)
            qj = O.quantize_codes(Wp[:, j], s.astype(np.float64), z.astype(np.float64), 4)
            wq = (qj - z.astype(np.float64)) * s.astype(np.float64)
            err = (Wp[:, j] - wq) / (U[j, j] if variant == "sign" else 1.0)
            upd = np.outer(err, U[j, j + 1:])
            Wp[:, j + 1:] += upd if variant == "sign" else -upd
            qm[:, j] = qj
        assert not np.array_equal(qm, qb), variant


# --- damping ("The two algorithms, compactly": before the Cholesky factor, H
# gets damp * mean(diag H) added on its diagonal, damp = 0.01). The expected
# matrices below are worked out by hand from that line, not by the oracle.

H3 = np.array([[4.0, 1.0, 0.5],
               [1.0, 2.0, 0.25],
               [0.5, 0.25, 6.0]])
# mean(diag) = (4 + 2 + 6) / 3 = 4, so 0.01 * 4 = 0.04 is added on the diagonal
H3_DAMPED = np.array([[4.04, 1.0, 0.5],
                      [1.0, 2.04, 0.25],
                      [0.5, 0.25, 6.04]])
# a channel whose activations are all zero (row and column 0 of H are zero):
# its diagonal becomes 1 first, then mean(diag) = (1 + 3 + 5) / 3 = 3 -> + 0.03
H_DEAD = np.array([[0.0, 0.0, 0.0],
                   [0.0, 3.0, 1.0],
                   [0.0, 1.0, 5.0]])
H_DEAD_DAMPED = np.array([[1.03, 0.0, 0.0],
                          [0.0, 3.03, 1.0],
                          [0.0, 1.0, 5.03]])


def test_damping_constant_is_the_pages():
    assert O.GPTQ_DAMP == 0.01


def test_damping_hand_example():
    np.testing.assert_allclose(O.gptq_damped(H3), H3_DAMPED, rtol=0, atol=1e-15)
    np.testing.assert_allclose(O.gptq_damped(H3, 0.5), H3 + 2.0 * np.eye(3), rtol=0, atol=1e-15)
    before = H3.copy()
    np.testing.assert_array_equal(O.gptq_damped(H3, 0.0), H3)
    np.testing.assert_array_equal(H3, before)  # the input is left untouched


def test_damping_dead_channel_hand_example():
    np.testing.assert_allclose(O.gptq_damped(H_DEAD), H_DEAD_DAMPED, rtol=0, atol=1e-15)


def _mutant_max_diag(H, damp=O.GPTQ_DAMP):
    H = np.array(H, dtype=np.float64)
    dead = np.diag(H) == 0
    H[dead, dead] = 1.0
    return H + damp * np.max(np.diag(H)) * np.eye(H.shape[0])


def _mutant_per_element(H, damp=O.GPTQ_DAMP):
    H = np.array(H, dtype=np.float64)
    dead = np.diag(H) == 0
    H[dead, dead] = 1.0
    return H + damp * np.diag(np.diag(H))


@pytest.mark.parametrize("mutant", [_mutant_max_diag, _mutant_per_element])
def test_damping_pins_catch_mutants(mutant):
    assert not np.allclose(mutant(H3), H3_DAMPED, rtol=0, atol=1e-12)


def test_damping_dead_channel_pin_catches_late_fix():
    # damping computed from the raw diagonal (mean 8/3), the dead entry set to 1 afterwards
    late = H_DEAD + (0.01 * 8.0 / 3.0) * np.eye(3)
    late[0, 0] = 1.0
    assert not np.allclose(late, H_DEAD_DAMPED, rtol=0, atol=1e-12)
    assert not np.allclose(_mutant_max_diag(H_DEAD), H_DEAD_DAMPED, rtol=0, atol=1e-12)


def test_dead_channel_codes_are_round_to_nearest():
    """A channel that never fires gets no error feedback (its row and column of
    H are zero apart from the damped diagonal): in the first group, whose
    scale is set before any update, its codes are the round-to-nearest codes."""
    N, K, g = 16, 64, 32
    W = synth.weights_np(N, K, synth.seed_for("gptq-dead", "w"))
    x = synth.activations_np(96, K, 0.05, synth.seed_for("gptq-dead", "x"))
    dead = 5
    x[:, dead] = 0
    q, s, z, g_idx = O.gptq_quantize(W, x, g, False)
    q_rtn, s_rtn, z_rtn = O.rtn_quantize(W, g, False)
    np.testing.assert_array_equal(s[:, 0], s_rtn[:, 0])
    np.testing.assert_array_equal(z[:, 0], z_rtn[:, 0])
    np.testing.assert_array_equal(q[:, dead], q_rtn[:, dead])
    # the live columns after it do receive feedback: not all of them stay at RTN
    assert not np.array_equal(q[:, dead + 1:g], q_rtn[:, dead + 1:g])
