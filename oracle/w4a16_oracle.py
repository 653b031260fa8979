"""NumPy fp64 oracle for the W4A16 group-quantized linear layer.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing in the library
imports this module.

What it computes, step by step, and where each step comes from:

1. Group map. By default input column j belongs to group j // g: the usual
   group is 128 neighbouring input columns of one row under one scale
   ("AWQ + GPTQ Quantization, in depth", section "What W4A16 buys and why
   decoding gets faster"). With GPTQ act order a column->group map ``g_idx``
   is given instead ("The two algorithms, compactly": act order; the Q&A page
   "How do GPTQ and AWQ differ ...", option ``desc_act``). Every group must
   hold exactly g columns.
2. Scale and zero per (row, group), round to nearest ("LLM Quantization:
   INT8, GPTQ, and AWQ Explained", section "What quantization actually does":
   find the range, choose the scale that stretches the integer levels
   across it, and move every weight to its closest grid value). With b-bit codes, qmax = 2^b - 1:
   asymmetric: s = fp16((max - min) / qmax), z = clamp(rint(-min / s), 0, qmax);
   symmetric, 3 or 4 bits: s = fp16(2 * max|w| / qmax), z = 2^(b-1) (the
     linear formula over [-a, a], which reproduces the fixed zero point 8 of
     4 bits; 4 at 3 bits);
   symmetric, 8 bits: the page's own int8 absmax code, s = fp16(max|w| / 127),
     codes clamp(rint(w / s), -127, 127), stored with the offset z = 128.
   A scale that is zero (constant group, or a range that rounds to 0 in fp16)
   is replaced by 1.0: the pages do not treat this case.
3. Codes q = clamp(rint(w / s) + z, 0, qmax), the linear quantization formula
   q = round(x / S) + Z ("LLM Quantization: A Deep Dive into GPTQ, AWQ, and
   Post-Training Quantization", section "The Math of Quantization") with the
   clamp of the int8 example on the INT8/GPTQ/AWQ page. ``rint`` rounds half
   to even (the pages' own code rounds with torch.round, which does), and the
   division is fp64 with the *stored* fp16 scale.
4. Canonical packing: 32/b codes per uint32 along the packed axis, code j of
   word k // (32/b) in bits b*j .. b*j+b-1 for column k with k % (32/b) == j;
   zero points packed the same way along the group axis, padded with zeros.
   3-bit codes (32/3 is not whole) form one little-endian bit stream per
   row: column k in stream bits 3k .. 3k+2, 32 codes per 3 words.
5. Dequantization w_hat = fp16((q - z) * s) ("The Math of Quantization":
   x_approx = (q - Z) * S). The fp64 product is exact; one round to nearest
   even gives the fp16 weight (the INT8/GPTQ/AWQ page: the product itself is
   computed in fp16, on weights expanded back to fp16 block by block).
6. Output y = x . w_hat^T in fp64 (W is "out x in", "The two algorithms,
   compactly"), with the per-element bound B = |x| . |w_hat|^T used by the
   acceptance test |y_gpu - y| <= 2e-3 * B + 1e-3.

7. AWQ with the per-input-channel scale kept apart ("The two algorithms,
   compactly": AWQ enlarges the weights of salient input channels by a factor
   s > 1 before quantizing and shrinks those activation channels by s to
   compensate; folding 1/s into the preceding operation is the usual
   deployment).
   Unfolded, the layer stores s (fp16 [K]) and computes
   y = fp16(x / s) . dequant(quantize(fp16(W * s)))^T: both the product and
   the quotient are exact in fp64 and rounded once to fp16. The scale search
   of the same section (s = s_x ** alpha, s_x = mean |x| per channel, alpha
   from a grid over [0, 1], keep the alpha with the smallest output error)
   produces s from calibration activations.

8. GPTQ ("The two algorithms, compactly"): H = 2 X X^T over the calibration
   inputs, H += damp * mean(diag H) * I (damp 0.01), Hinv = the upper
   Cholesky factor U of H^-1 (H^-1 = U^T U); columns are taken in order (act
   order: by descending diag H); each column is quantized to its group's
   grid, err = (w_j - q_j) / U[j, j] and the columns not yet quantized get
   W[:, j+1:] -= err U[j, j+1:]. A group's scale and zero point are set when
   its first column is reached, from the current (already updated) weights
   of its columns; under act order the groups are runs of group_size
   columns in processing order.

No blocking, fusion or reordering beyond these definitions; library matmuls
(``@``) are used for the sums.
"""

from __future__ import annotations

import numpy as np

QMAX = 15  # 4-bit codes are 0..15
SYM_ZERO = 8  # symmetric 4-bit scheme: zero point fixed at 8
# code widths: 4 bits, and the other two the pages name ("How do GPTQ and AWQ
# differ ...", section "The shared setting": 3 and 8 bits)
BITS = (3, 4, 8)


def qmax(bits: int) -> int:
    if bits not in BITS:
        raise ValueError("bits must be 3, 4 or 8")
    return (1 << bits) - 1


def sym_zero(bits: int) -> int:
    """Fixed zero point of the symmetric scheme: 4 (3 bits), 8 (4 bits), 128 (8 bits)."""
    return 1 << (bits - 1)
TOL_REL = 2e-3  # |y_gpu - y_ref| <= TOL_REL * sum|x * w_hat| + TOL_ABS
TOL_ABS = 1e-3


# ---------------------------------------------------------------------------
# fp16 rounding
# ---------------------------------------------------------------------------
def fp16_rne(a) -> np.ndarray:
    """Round fp64 values to the nearest fp16 value, ties to even.

    NumPy converts float64 -> float16 directly (no detour through float32),
    rounding to nearest even. This is pinned in the tests against an
    exhaustive nearest-value search over all finite fp16 values and against
    ``struct``'s half-precision packing.
    """
    return np.asarray(a, dtype=np.float64).astype(np.float16)


# ---------------------------------------------------------------------------
# Step 1: group map
# ---------------------------------------------------------------------------
def group_map(K: int, group_size: int, g_idx=None) -> tuple[np.ndarray, int]:
    """Return (g_idx as int64 [K], number of groups G).

    Without ``g_idx`` column j is in group j // group_size. With ``g_idx``
    (act order) the map is validated: values in [0, G) and exactly
    ``group_size`` members per group, G = K / group_size.
    """
    if group_size <= 0:
        raise ValueError("group_size must be positive")
    if g_idx is None:
        G = -(-K // group_size)
        return np.arange(K, dtype=np.int64) // group_size, G
    g_idx = np.asarray(g_idx, dtype=np.int64)
    if g_idx.shape != (K,):
        raise ValueError("g_idx must have shape [K]")
    if K % group_size != 0:
        raise ValueError("act order needs K divisible by group_size")
    G = K // group_size
    if g_idx.min(initial=0) < 0 or g_idx.max(initial=0) >= G:
        raise ValueError("g_idx out of range")
    counts = np.bincount(g_idx, minlength=G)
    if not np.all(counts == group_size):
        raise ValueError("every group must have exactly group_size members")
    return g_idx, G


def group_members(g_idx: np.ndarray, G: int) -> list[np.ndarray]:
    """Columns of each group, in increasing column order."""
    return [np.flatnonzero(g_idx == t) for t in range(G)]


# ---------------------------------------------------------------------------
# Steps 2-3: round-to-nearest quantization
# ---------------------------------------------------------------------------
def quantize_codes(w: np.ndarray, s: np.ndarray, z: np.ndarray, bits: int = 4) -> np.ndarray:
    """q = clamp(rint(w / s) + z, 0, qmax); w, s, z broadcast, fp64 division."""
    w = np.asarray(w, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    q = np.rint(w / s) + np.asarray(z, dtype=np.float64)
    return np.clip(q, 0, qmax(bits)).astype(np.uint8)


def sym8_codes(w: np.ndarray, s: np.ndarray) -> np.ndarray:
    """8-bit symmetric codes: clamp(rint(w / s), -127, 127) + 128 (the int8
    absmax code of "What quantization actually does", offset to unsigned)."""
    w = np.asarray(w, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    return (np.clip(np.rint(w / s), -127, 127) + 128).astype(np.uint8)


def group_scale_zero(w: np.ndarray, sym: bool, bits: int = 4) -> tuple[np.ndarray, np.ndarray]:
    """Scale (fp16) and zero (uint8) of each row of ``w`` ([rows, members])."""
    w = np.asarray(w, dtype=np.float64)
    qm = qmax(bits)
    if sym:
        a = np.max(np.abs(w), axis=1)
        s = fp16_rne(a / 127.0) if bits == 8 else fp16_rne(2.0 * a / qm)
    else:
        mn = np.min(w, axis=1)
        mx = np.max(w, axis=1)
        s = fp16_rne((mx - mn) / qm)
    s = np.where(s == 0, np.float16(1.0), s).astype(np.float16)
    if sym:
        z = np.full(w.shape[0], sym_zero(bits), dtype=np.uint8)
    else:
        z = np.clip(np.rint(-mn / s.astype(np.float64)), 0, qm).astype(np.uint8)
    return s, z


def rtn_quantize(W, group_size: int, sym: bool, g_idx=None, bits: int = 4):
    """Round-to-nearest group quantization of fp16 ``W`` [N, K].

    Returns codes q uint8 [N, K] (original column order), scales fp16 [N, G]
    and zeros uint8 [N, G] (all 8, or 128 at 8 bits, when ``sym``).
    """
    W = np.asarray(W)
    if W.dtype != np.float16:
        raise TypeError("W must be float16")
    N, K = W.shape
    gi, G = group_map(K, group_size, g_idx)
    Wd = W.astype(np.float64)
    q = np.zeros((N, K), dtype=np.uint8)
    scales = np.zeros((N, G), dtype=np.float16)
    zeros = np.zeros((N, G), dtype=np.uint8)
    for t, cols in enumerate(group_members(gi, G)):
        w = Wd[:, cols]
        s, z = group_scale_zero(w, sym, bits)
        scales[:, t] = s
        zeros[:, t] = z
        sd = s.astype(np.float64)[:, None]
        q[:, cols] = sym8_codes(w, sd) if (sym and bits == 8) else quantize_codes(w, sd, z[:, None], bits)
    return q, scales, zeros


# ---------------------------------------------------------------------------
# Step 4: canonical packing (8 nibbles per uint32, along the packed axis)
# ---------------------------------------------------------------------------
def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """Pack uint8 codes [R, C] (0..15) into uint32 [R, ceil(C/8)].

    Nibble j (bits 4j..4j+3) of word c // 8 holds column c with c % 8 == j;
    missing columns of the last word are zero.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    if codes.max(initial=0) > QMAX:
        raise ValueError("codes must be 0..15")
    R, C = codes.shape
    W8 = -(-C // 8)
    padded = np.zeros((R, W8 * 8), dtype=np.uint32)
    padded[:, :C] = codes
    out = np.zeros((R, W8), dtype=np.uint32)
    for j in range(8):
        out |= padded[:, j::8] << np.uint32(4 * j)
    return out


def unpack_nibbles(words: np.ndarray, C: int) -> np.ndarray:
    """Inverse of ``pack_nibbles``: uint32 [R, ceil(C/8)] -> uint8 [R, C]."""
    words = np.asarray(words, dtype=np.uint32)
    R, W8 = words.shape
    out = np.zeros((R, W8 * 8), dtype=np.uint8)
    for j in range(8):
        out[:, j::8] = (words >> np.uint32(4 * j)) & np.uint32(0xF)
    return out[:, :C]


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Pack b-bit codes [R, C] into uint32 [R, ceil(C / (32/b))], code j of a
    word in bits b*j .. b*j+b-1; missing columns of the last word are zero.
    3 bits: a bit stream per row, column k in bits 3k .. 3k+2, ceil(3C/32) words."""
    if bits == 4:
        return pack_nibbles(codes)
    if bits == 3:
        codes = np.asarray(codes, dtype=np.uint8)
        if codes.max(initial=0) > 7:
            raise ValueError("codes must be 0..7")
        R, C = codes.shape
        nw = -(-3 * C // 32)
        stream = np.zeros((R, nw * 32), dtype=np.uint8)  # one bit per entry
        for b in range(3):
            stream[:, b:3 * C:3] = (codes >> b) & 1
        weights = (np.uint64(1) << np.arange(32, dtype=np.uint64))
        return (stream.reshape(R, nw, 32).astype(np.uint64) * weights).sum(axis=2).astype(np.uint32)
    codes = np.asarray(codes, dtype=np.uint8)
    per = 32 // bits
    R, C = codes.shape
    nw = -(-C // per)
    padded = np.zeros((R, nw * per), dtype=np.uint32)
    padded[:, :C] = codes
    out = np.zeros((R, nw), dtype=np.uint32)
    for j in range(per):
        out |= padded[:, j::per] << np.uint32(bits * j)
    return out


def unpack_codes(words: np.ndarray, C: int, bits: int) -> np.ndarray:
    """Inverse of ``pack_codes``."""
    if bits == 4:
        return unpack_nibbles(words, C)
    if bits == 3:
        words = np.asarray(words, dtype=np.uint32)
        R, nw = words.shape
        stream = ((words[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(R, nw * 32)
        out = np.zeros((R, C), dtype=np.uint8)
        for b in range(3):
            out |= (stream[:, b:3 * C:3].astype(np.uint8) << b)
        return out
    words = np.asarray(words, dtype=np.uint32)
    per = 32 // bits
    R, nw = words.shape
    out = np.zeros((R, nw * per), dtype=np.uint8)
    for j in range(per):
        out[:, j::per] = (words >> np.uint32(bits * j)) & np.uint32((1 << bits) - 1)
    return out[:, :C]


# ---------------------------------------------------------------------------
# Step 5: dequantization
# ---------------------------------------------------------------------------
def dequant(q, scales, zeros, group_size: int, g_idx=None) -> np.ndarray:
    """w_hat[n, k] = fp16((q[n,k] - z[n, g(k)]) * s[n, g(k)]), fp16 [N, K]."""
    q = np.asarray(q)
    N, K = q.shape
    gi, G = group_map(K, group_size, g_idx)
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)[:, gi]
    z = np.asarray(zeros, dtype=np.float64)[:, gi]
    return fp16_rne((q.astype(np.float64) - z) * s)


# ---------------------------------------------------------------------------
# Step 6: the linear layer and its acceptance bound
# ---------------------------------------------------------------------------
def linear_ref(x, w_hat) -> tuple[np.ndarray, np.ndarray]:
    """(y, B): y = x . w_hat^T and B = |x| . |w_hat|^T, both fp64 [M, N]."""
    xd = np.asarray(x, dtype=np.float64)
    wd = np.asarray(w_hat, dtype=np.float64)
    return xd @ wd.T, np.abs(xd) @ np.abs(wd).T


def tolerance(B) -> np.ndarray:
    """Per-element acceptance bound 2e-3 * B + 1e-3."""
    return TOL_REL * np.asarray(B, dtype=np.float64) + TOL_ABS


def error_ratio(y_test, y_ref, B) -> np.ndarray:
    """|y_test - y_ref| / (2e-3 * B + 1e-3): passes where <= 1."""
    return np.abs(np.asarray(y_test, dtype=np.float64) - y_ref) / tolerance(B)


def w4a16_linear(x, W, group_size: int, sym: bool, g_idx=None, bits: int = 4):
    """End to end: quantize fp16 W (b-bit codes), dequantize, multiply by fp16 x.

    Returns (y, B, (q, scales, zeros), w_hat).
    """
    q, s, z = rtn_quantize(W, group_size, sym, g_idx, bits)
    w_hat = dequant(q, s, z, group_size, g_idx)
    y, B = linear_ref(x, w_hat)
    return y, B, (q, s, z), w_hat


# ---------------------------------------------------------------------------
# Byte budget (closed form)
# ---------------------------------------------------------------------------
def packed_bytes_closed_form(N: int, K: int, group_size: int, sym: bool, bits: int = 4) -> float:
    """Bytes of one packed linear: codes N*K*b/8, fp16 scales N*G*2, b-bit
    zeros N*G*b/8 (none when symmetric), G = K / group_size ("What W4A16
    buys": one fp16 scale for a group of 128 = 0.125 bit/weight, 4-bit zero ~0.03)."""
    G = K / group_size
    return N * K * bits / 8 + N * G * 2 + (0 if sym else N * G * bits / 8)


def bits_per_weight(group_size: int, sym: bool, bits: int = 4) -> float:
    return bits + 16 / group_size + (0 if sym else bits / group_size)


# ---------------------------------------------------------------------------
# Step 7: AWQ, per-input-channel scale kept apart from the weights
# ---------------------------------------------------------------------------
def _check_act_scale(act_scale, K: int) -> np.ndarray:
    a = np.asarray(act_scale)
    if a.dtype != np.float16 or a.shape != (K,):
        raise TypeError("act_scale must be float16 [K]")
    if not np.all(np.isfinite(a)) or np.any(a.astype(np.float64) <= 0):
        raise ValueError("act_scale must be finite and positive")
    return a.astype(np.float64)


def awq_scale_weights(W, act_scale) -> np.ndarray:
    """fp16(W[n, k] * s[k]): the salient channels' weights scaled up before
    quantizing. The fp64 product of two fp16 values is exact."""
    W = np.asarray(W)
    if W.dtype != np.float16:
        raise TypeError("W must be float16")
    s = _check_act_scale(act_scale, W.shape[1])
    return fp16_rne(W.astype(np.float64) * s[None, :])


def awq_scale_activations(x, act_scale) -> np.ndarray:
    """fp16(x[m, k] / s[k]): the activations divided by the same scale. The
    fp64 quotient of two fp16 values is rounded once (fp64 carries more than
    2 * 11 + 2 bits, so rounding through it equals rounding the exact
    quotient)."""
    x = np.asarray(x)
    if x.dtype != np.float16:
        raise TypeError("x must be float16")
    s = _check_act_scale(act_scale, x.shape[1])
    return fp16_rne(x.astype(np.float64) / s[None, :])


def awq_linear(x, W, act_scale, group_size: int, sym: bool, g_idx=None, bits: int = 4):
    """Unfolded AWQ layer: quantize fp16(W * s), divide x by s, multiply.

    Returns (y, B, (q, scales, zeros), w_hat, x_scaled); B = |x_scaled| . |w_hat|^T.
    """
    Ws = awq_scale_weights(W, act_scale)
    q, s, z = rtn_quantize(Ws, group_size, sym, g_idx, bits)
    w_hat = dequant(q, s, z, group_size, g_idx)
    xs = awq_scale_activations(x, act_scale)
    y, B = linear_ref(xs, w_hat)
    return y, B, (q, s, z), w_hat, xs


def awq_grid(n_grid: int = 20) -> np.ndarray:
    """alpha = 0, 1/n, ..., 1 (the section's grid over [0, 1], ends included)."""
    return np.arange(n_grid + 1, dtype=np.float64) / n_grid


def awq_search(W, x, group_size: int, sym: bool, bits: int = 4, n_grid: int = 20):
    """AWQ's scale search for one linear layer, in the section's order.

    x: calibration activations [tokens, K] (fp16). Per input channel
    s_x = mean_t |x[t, k]|; for every alpha of the grid s = fp16(s_x ** alpha)
    (a channel with s_x = 0 carries no activation and keeps s = 1);
    Wq = dequant(quantize(fp16(W * s))) / s; loss = ||x W^T - x Wq^T||_F.
    Returns (s of the smallest loss, its alpha, all losses); ties keep the
    smaller alpha.
    """
    W = np.asarray(W)
    xd = np.asarray(x, dtype=np.float64)
    s_x = np.mean(np.abs(xd), axis=0)
    y_ref = xd @ W.astype(np.float64).T
    losses = []
    best = None
    for alpha in awq_grid(n_grid):
        sc = np.where(s_x > 0, s_x ** alpha if alpha > 0 else 1.0, 1.0)
        s16 = fp16_rne(sc)
        q, s, z = rtn_quantize(awq_scale_weights(W, s16), group_size, sym, bits=bits)
        Wq = dequant(q, s, z, group_size).astype(np.float64) / s16.astype(np.float64)[None, :]
        loss = float(np.linalg.norm(y_ref - xd @ Wq.T))
        losses.append(loss)
        if best is None or loss < best[0]:
            best = (loss, s16, float(alpha))
    return best[1], best[2], np.array(losses)


# ---------------------------------------------------------------------------
# Step 8: GPTQ -- quantize one column at a time, push the error onto the rest
# ---------------------------------------------------------------------------
GPTQ_DAMP = 0.01


def gptq_hessian(x) -> np.ndarray:
    """H = 2 X X^T with X = x^T (in x tokens): [K, K] fp64."""
    xd = np.asarray(x, dtype=np.float64)
    return 2.0 * (xd.T @ xd)


def gptq_order(H, act_order: bool) -> np.ndarray:
    """Processing order: natural, or by descending diag(H), ties to the lower column."""
    K = H.shape[0]
    if not act_order:
        return np.arange(K, dtype=np.int64)
    return np.argsort(-np.diag(H), kind="stable").astype(np.int64)


def gptq_damped(H, damp: float = GPTQ_DAMP) -> np.ndarray:
    """H + damp * mean(diag H) * I. A zero diagonal (a channel that never
    fires) is set to 1 first so that H stays invertible; its weights get no
    error feedback from other columns and none of theirs."""
    H = np.array(H, dtype=np.float64, copy=True)
    dead = np.diag(H) == 0
    H[dead, :] = 0.0
    H[:, dead] = 0.0
    H[dead, dead] = 1.0
    H += damp * np.mean(np.diag(H)) * np.eye(H.shape[0])
    return H


def gptq_factor(Hd) -> np.ndarray:
    """The upper Cholesky factor U of H^-1 (H^-1 = U^T U)."""
    Hinv = np.linalg.inv(Hd)
    return np.linalg.cholesky(Hinv).T  # cholesky gives lower L with Hinv = L L^T; U = L^T


def gptq_quantize(W, x, group_size: int, sym: bool, bits: int = 4, act_order: bool = False,
                  damp: float = GPTQ_DAMP):
    """GPTQ of fp16 W [N, K] with calibration activations x [tokens, K].

    Returns (q uint8 [N, K] in original column order, scales fp16 [N, G],
    zeros uint8 [N, G], g_idx int64 [K] or None). Group t of the returned
    format holds the columns processed in positions t*g .. t*g+g-1.
    """
    W = np.asarray(W)
    if W.dtype != np.float16:
        raise TypeError("W must be float16")
    N, K = W.shape
    if K % group_size:
        raise ValueError("K must be a multiple of group_size")
    H = gptq_hessian(x)
    order = gptq_order(H, act_order)
    Hd = gptq_damped(H, damp)[np.ix_(order, order)]
    U = gptq_factor(Hd)
    Wp = W.astype(np.float64)[:, order]  # working copy, processing order
    G = K // group_size
    q = np.zeros((N, K), dtype=np.uint8)
    scales = np.zeros((N, G), dtype=np.float16)
    zeros = np.zeros((N, G), dtype=np.uint8)
    for j in range(K):
        t = j // group_size
        if j % group_size == 0:
            s, z = group_scale_zero(Wp[:, j:j + group_size], sym, bits)
            scales[:, t], zeros[:, t] = s, z
        sd = scales[:, t].astype(np.float64)
        zd = zeros[:, t].astype(np.float64)
        w = Wp[:, j]
        qj = sym8_codes(w[:, None], sd[:, None])[:, 0] if (sym and bits == 8) else \
            quantize_codes(w, sd, zd, bits)
        wq = (qj.astype(np.float64) - zd) * sd  # the grid point (exact in fp64)
        err = (w - wq) / U[j, j]
        Wp[:, j + 1:] -= np.outer(err, U[j, j + 1:])
        Wp[:, j] = wq
        q[:, order[j]] = qj
    g_idx = None
    if act_order:
        g_idx = np.empty(K, dtype=np.int64)
        g_idx[order] = np.arange(K) // group_size
    return q, scales, zeros, g_idx


def layer_error(W, w_hat, x) -> float:
    """||x W^T - x w_hat^T||_F, the quantity both calibration methods reduce."""
    xd = np.asarray(x, dtype=np.float64)
    return float(np.linalg.norm(xd @ np.asarray(W, np.float64).T - xd @ np.asarray(w_hat, np.float64).T))
