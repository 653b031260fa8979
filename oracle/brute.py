"""Pure-Python scalar restatement of the oracle, for tiny shapes only.

TEST INFRASTRUCTURE ONLY. Shares no code with ``w4a16_oracle``: fp16 rounding
goes through ``struct``'s half-precision format (CPython rounds a double to
the nearest half, ties to even), rounding to integers through the built-in
``round`` (ties to even), sums are plain Python-float loops. It follows the
same steps as ``w4a16_oracle`` -- the linear quantization formula of "LLM
Quantization: A Deep Dive into GPTQ, AWQ, and Post-Training Quantization"
(section "The Math of Quantization") applied per group of input columns as in
"AWQ + GPTQ Quantization, in depth" (section "What W4A16 buys and why
decoding gets faster") -- written out element by element so that a slip in
the vectorised version (an index, a sign, a transposed operand) shows up as a
mismatch.
"""

from __future__ import annotations

import struct


def f16(v: float) -> float:
    """Nearest fp16 value of a double, ties to even (via struct 'e')."""
    return struct.unpack("<e", struct.pack("<e", v))[0]


def _clamp(v: int, lo: int, hi: int) -> int:
    return lo if v < lo else hi if v > hi else v


def quantize(W, group_size, sym, g_idx=None, bits=4):
    """W: list of rows of Python floats (fp16 values). Returns q, s, z lists.

    b-bit codes, top = 2^b - 1. Symmetric: 3 and 4 bits s = f16(2a/top),
    z = 2^(b-1); 8 bits (the int8 absmax code) s = f16(a/127),
    q = clamp(round(w/s), -127, 127) + 128.
    """
    top = (1 << bits) - 1
    N, K = len(W), len(W[0])
    if g_idx is None:
        g_idx = [k // group_size for k in range(K)]
    G = max(g_idx) + 1
    q = [[0] * K for _ in range(N)]
    s_out = [[0.0] * G for _ in range(N)]
    z_out = [[0] * G for _ in range(N)]
    for n in range(N):
        for t in range(G):
            cols = [k for k in range(K) if g_idx[k] == t]
            vals = [W[n][k] for k in cols]
            if sym:
                a = max(abs(v) for v in vals)
                s = f16(a / 127.0) if bits == 8 else f16(2.0 * a / top)
            else:
                lo, hi = min(vals), max(vals)
                s = f16((hi - lo) / top)
            if s == 0.0:
                s = 1.0
            if sym:
                z = 1 << (bits - 1)
            else:
                z = _clamp(round(-lo / s), 0, top)
            s_out[n][t] = s
            z_out[n][t] = z
            for k in cols:
                if sym and bits == 8:
                    q[n][k] = _clamp(round(W[n][k] / s), -127, 127) + 128
                else:
                    q[n][k] = _clamp(round(W[n][k] / s) + z, 0, top)
    return q, s_out, z_out


def dequant(q, s, z, g_idx):
    return [[f16((q[n][k] - z[n][g_idx[k]]) * s[n][g_idx[k]])
             for k in range(len(q[0]))] for n in range(len(q))]


def linear(x, w_hat):
    """y[m][n] = sum_k x[m][k] * w_hat[n][k] (W is out x in)."""
    M, N, K = len(x), len(w_hat), len(x[0])
    y = [[0.0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += x[m][k] * w_hat[n][k]
            y[m][n] = acc
    return y


def pack_word(codes, bits=4):
    """32/b codes -> one uint32, code i in bits b*i .. b*i+b-1."""
    w = 0
    for i, c in enumerate(codes):
        w |= (c & ((1 << bits) - 1)) << (bits * i)
    return w


def awq_linear(x, W, act_scale, group_size, sym, g_idx=None, bits=4):
    """Unfolded AWQ, element by element: W'[n][k] = f16(W[n][k] * s[k]) is
    quantized, x'[m][k] = f16(x[m][k] / s[k]); returns (y, q, s, z, x')."""
    K = len(W[0])
    Ws = [[f16(W[n][k] * act_scale[k]) for k in range(K)] for n in range(len(W))]
    xs = [[f16(x[m][k] / act_scale[k]) for k in range(K)] for m in range(len(x))]
    q, s, z = quantize(Ws, group_size, sym, g_idx, bits)
    gi = g_idx if g_idx is not None else [k // group_size for k in range(K)]
    return linear(xs, dequant(q, s, z, gi)), q, s, z, xs


def pack_stream3(codes):
    """3-bit codes of one row -> list of uint32 words of the bit stream, code
    k in stream bits 3k .. 3k+2 (bit i of the stream is bit i % 32 of word
    i // 32)."""
    total = 3 * len(codes)
    words = [0] * (-(-total // 32))
    for k, c in enumerate(codes):
        for b in range(3):
            if (c >> b) & 1:
                i = 3 * k + b
                words[i // 32] |= 1 << (i % 32)
    return words
