"""Host-side tests of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments before touching the GPU. No GPU needed."""

import ctypes
import os
import re

import pytest

from oracle import w4a16_oracle as O
from weight_only_bit_04_b300 import w4a16 as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, SMALL = 0, 1, 2, 3, 4
FAKE = 0x10000  # aligned, never dereferenced: every call below fails validation first


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"W4A16_API\s+[\w\s\*]+?\b(w4a16_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from weight_only_bit_04_b300 import build
    build.build()
    return W.lib()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("w4a16_pack", "w4a16_dequant", "w4a16_gemv", "w4a16_gemm"):
        assert required in names
    assert set(names) == set(W.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def fmt(N=256, K=512, g=128, sym=False, act=False, bits=4):
    return W.make_format(N, K, g, sym, act, bits)


def test_packed_bytes_layout(lib):
    f = fmt(4096, 4096)
    nr, kb, G = 32, 64, 32
    q = nr * kb * 4096
    s = nr * G * 256
    z = nr * G * 64
    assert W.packed_bytes(f) == q + s + z  # all multiples of 256
    # For N a multiple of 128 the blob is exactly the closed-form byte count.
    assert W.packed_bytes(f) == O.packed_bytes_closed_form(4096, 4096, 128, False)
    assert W.packed_bytes(fmt(4096, 4096, sym=True)) == O.packed_bytes_closed_form(4096, 4096, 128, True)
    fa = fmt(4096, 4096, act=True)
    assert W.packed_bytes(fa) == q + s + z + 4096 * 4
    # padding rows / columns are counted
    # (zeros: 2*3*64 = 384 bytes, the blob end is rounded up to 256)
    assert W.packed_bytes(fmt(200, 96, g=32)) == 2 * 2 * 4096 + 2 * 3 * 256 + 512


def test_packed_bytes_3bit(lib):
    """3-bit codes: 3 KiB tiles; zero points stay nibble pairs (64 B per group block)."""
    f3 = fmt(4096, 4096, bits=3)
    assert W.check_format(f3) == 0
    assert W.packed_bytes(f3) == 32 * 64 * 3072 + 32 * 32 * 256 + 32 * 32 * 64
    # the blob's zero points take 4 bits where the closed form counts 3
    assert W.packed_bytes(f3) == O.packed_bytes_closed_form(4096, 4096, 128, False, bits=3) + 4096 * 32 / 8
    assert W.packed_bytes(fmt(4096, 4096, sym=True, bits=3)) == O.packed_bytes_closed_form(4096, 4096, 128, True, 3)


def test_packed_bytes_8bit(lib):
    """8-bit codes: twice the code and zero-point bytes, the same scales."""
    for sym in (False, True):
        f8 = fmt(4096, 4096, sym=sym, bits=8)
        assert W.check_format(f8) == 0
        assert W.packed_bytes(f8) == O.packed_bytes_closed_form(4096, 4096, 128, sym, bits=8)
    # padding: 2 x 2 tiles of 8 KiB, scales 2*3*256, zeros 2*3*128 = 768 (a multiple of 256)
    assert W.packed_bytes(fmt(200, 96, g=32, bits=8)) == 2 * 2 * 8192 + 2 * 3 * 256 + 768


@pytest.mark.parametrize("kw,status", [
    (dict(bits=5), UNSUPPORTED),
    (dict(bits=2), UNSUPPORTED),
    (dict(bits=16), UNSUPPORTED),
    (dict(g=16), UNSUPPORTED),
    (dict(g=256), UNSUPPORTED),
    (dict(K=96, g=64), UNSUPPORTED),   # ragged last group
    (dict(N=0), INVALID),
    (dict(K=0), INVALID),
    (dict(N=(1 << 20) + 1), INVALID),
])
def test_bad_formats(lib, kw, status):
    f = fmt(**kw)
    assert W.check_format(f) == status
    assert W.packed_bytes(f) == 0


def test_status_strings(lib):
    for code, name in W.STATUS.items():
        assert lib.w4a16_status_string(code).decode() == name
    assert lib.w4a16_status_string(99).decode() == "W4A16_ERR_UNKNOWN"


def _call(lib, name, *args):
    return getattr(lib, name)(*args)


def test_pack_argument_checks(lib):
    f = fmt()
    nb = W.packed_bytes(f)
    r = lambda *a: _call(lib, "w4a16_pack", ctypes.byref(f), *a)
    assert r(None, FAKE, FAKE, None, FAKE, nb, None) == INVALID        # q NULL
    assert r(FAKE, FAKE, None, None, FAKE, nb, None) == INVALID        # zeros NULL (asym)
    assert r(FAKE, FAKE, FAKE, None, FAKE + 16, nb, None) == MISALIGNED
    assert r(FAKE, FAKE + 1, FAKE, None, FAKE, nb, None) == MISALIGNED
    assert r(FAKE, FAKE, FAKE, None, FAKE, nb - 1, None) == SMALL
    fs = fmt(sym=True)
    assert _call(lib, "w4a16_pack", ctypes.byref(fs), FAKE, FAKE, FAKE, None, FAKE,
                 W.packed_bytes(fs), None) == INVALID                  # zeros given (sym)
    fa = fmt(act=True)
    nba = W.packed_bytes(fa)
    assert _call(lib, "w4a16_pack", ctypes.byref(fa), FAKE, FAKE, FAKE, None, FAKE, nba,
                 None) == INVALID                                     # g_idx missing


def test_pack_rejects_bad_g_idx_on_host(lib):
    f = fmt(N=8, K=256, g=128, act=True)
    nb = W.packed_bytes(f)
    bad = (ctypes.c_int32 * 256)(*([0] * 129 + [1] * 127))            # group 0 has 129 members
    assert lib.w4a16_pack(ctypes.byref(f), FAKE, FAKE, FAKE, bad, FAKE, nb, None) == INVALID
    oob = (ctypes.c_int32 * 256)(*([0] * 128 + [2] * 128))
    assert lib.w4a16_pack(ctypes.byref(f), FAKE, FAKE, FAKE, oob, FAKE, nb, None) == INVALID


def test_gemv_argument_checks(lib):
    f = fmt()
    nb = W.packed_bytes(f)
    g = lambda packed, nbytes, x, y, M: lib.w4a16_gemv(ctypes.byref(f), packed, nbytes, x, y, M, None)
    X, Y = FAKE * 16, FAKE * 64
    assert g(None, nb, X, Y, 1) == INVALID
    assert g(FAKE, nb, X, Y, 0) == INVALID
    assert g(FAKE, nb, X, Y, 17) == INVALID
    assert g(FAKE, nb - 1, X, Y, 1) == SMALL
    assert g(FAKE + 128, nb, X, Y, 1) == MISALIGNED
    assert g(FAKE, nb, X + 2, Y, 1) == MISALIGNED
    assert g(FAKE, nb, X, Y + 8, 1) == MISALIGNED
    assert g(FAKE, nb, X, X, 1) == INVALID                              # y overlaps x
    bad = fmt(bits=2)
    assert lib.w4a16_gemv(ctypes.byref(bad), FAKE, nb, X, Y, 1, None) == UNSUPPORTED
    # explicit launch shapes are validated too
    ring, stage_x, async_copy = 2, 4, 8
    assert lib.w4a16_gemv_ex(ctypes.byref(f), FAKE, nb, X, Y, 1, 3, 1, 0, None) == INVALID      # rows16
    assert lib.w4a16_gemv_ex(ctypes.byref(f), FAKE, nb, X, Y, 1, 16, 1, ring, None) == INVALID
    assert lib.w4a16_gemv_ex(ctypes.byref(f), FAKE, nb, X, Y, 1, 8, 32, 0, None) == INVALID
    assert lib.w4a16_gemv_ex(ctypes.byref(f), FAKE, nb, X, Y, 1, 0, 0, 64, None) == INVALID    # unknown flag
    assert lib.w4a16_gemv_ex(ctypes.byref(f), FAKE, nb, X, Y, 1, 0, 0, ring | stage_x | 32, None) == INVALID
    assert lib.w4a16_gemv_ex(ctypes.byref(f), FAKE, nb, X, Y, 1, 0, 0, ring | async_copy, None) == INVALID


def test_gemm_and_workspace_checks(lib):
    f = fmt(act=True)
    nb = W.packed_bytes(f)
    assert lib.w4a16_gemm_workspace_bytes(ctypes.byref(f), 2048) == 2048 * 512 * 2
    assert lib.w4a16_gemm_workspace_bytes(ctypes.byref(fmt()), 2048) == 0
    X, Y = FAKE * 16, FAKE * 4096
    assert lib.w4a16_gemm(ctypes.byref(f), FAKE, nb, X, Y, 2048, None, 0, None) == SMALL
    assert lib.w4a16_gemm(ctypes.byref(f), FAKE, nb, X, Y, 0, None, 0, None) == INVALID
    assert lib.w4a16_gemm(ctypes.byref(f), FAKE, nb, X, Y, 2048, FAKE + 4, 2048 * 1024,
                          None) == MISALIGNED
    assert lib.w4a16_quantize_workspace_bytes(ctypes.byref(f)) == 512 * 4
    assert lib.w4a16_quantize_rtn(ctypes.byref(f), FAKE, None, FAKE, FAKE, FAKE, FAKE, 2048,
                                  None) == INVALID                    # g_idx missing


def test_dequant_checks(lib):
    f = fmt()
    nb = W.packed_bytes(f)
    assert lib.w4a16_dequant(ctypes.byref(f), FAKE, nb, None, None) == INVALID
    assert lib.w4a16_dequant(ctypes.byref(f), FAKE, nb, FAKE + 2, None) == MISALIGNED
    assert lib.w4a16_dequant(ctypes.byref(f), FAKE, 10, FAKE, None) == SMALL


def test_act_scale_format_and_entry_points(lib):
    """Unfolded AWQ: the blob grows by the fp16 act scale; the plain packer and
    quantizer refuse such a format, the AWQ ones require it and its scale."""
    f = W.make_format(256, 512, 128, False, False, act_scale=True)
    plain = fmt()
    assert W.check_format(f) == OK
    assert W.packed_bytes(f) == W.packed_bytes(plain) + 512 * 2          # K fp16 (a multiple of 256 here)
    assert W.packed_bytes(W.make_format(256, 96, 32, act_scale=True)) == \
        W.packed_bytes(W.make_format(256, 96, 32)) + 256                   # rounded up to 256 bytes
    bad = W.make_format(256, 512, act_scale=True)
    bad.has_act_scale = 2
    assert W.check_format(bad) == INVALID
    nb = W.packed_bytes(f)
    # plain packer: refuses (the scale would be lost); AWQ packer: needs the scale
    assert lib.w4a16_pack(ctypes.byref(f), FAKE, FAKE, FAKE, None, FAKE, nb, None) == INVALID
    assert lib.w4a16_pack_awq(ctypes.byref(f), FAKE, FAKE, FAKE, None, None, FAKE, nb, None) == INVALID
    assert lib.w4a16_pack_awq(ctypes.byref(f), FAKE, FAKE, FAKE, None, FAKE + 1, FAKE, nb, None) == MISALIGNED
    assert lib.w4a16_pack_awq(ctypes.byref(f), FAKE, FAKE, FAKE, None, FAKE, FAKE, nb - 1, None) == SMALL
    assert lib.w4a16_pack_awq(ctypes.byref(plain), FAKE, FAKE, FAKE, None, FAKE, FAKE,
                              W.packed_bytes(plain), None) == INVALID     # format without a scale
    # quantizers
    assert lib.w4a16_quantize_rtn(ctypes.byref(f), FAKE, None, FAKE, FAKE, FAKE, None, 0, None) == INVALID
    assert lib.w4a16_quantize_rtn_noalloc(ctypes.byref(f), FAKE, None, FAKE, FAKE, FAKE, None) == INVALID
    assert lib.w4a16_quantize_rtn_awq(ctypes.byref(f), FAKE, None, None, FAKE, FAKE, FAKE, None, 0,
                                      None) == INVALID                    # scale missing
    assert lib.w4a16_quantize_rtn_awq(ctypes.byref(f), FAKE, FAKE + 1, None, FAKE, FAKE, FAKE, None, 0,
                                      None) == MISALIGNED
    assert lib.w4a16_quantize_rtn_awq(ctypes.byref(plain), FAKE, FAKE, None, FAKE, FAKE, FAKE, None, 0,
                                      None) == INVALID
    # the GEMM stages x / s in the workspace even without act order
    assert lib.w4a16_gemm_workspace_bytes(ctypes.byref(f), 100) == 100 * 512 * 2
    X, Y = FAKE * 16, FAKE * 4096
    assert lib.w4a16_gemm(ctypes.byref(f), FAKE, nb, X, Y, 100, None, 0, None) == SMALL


def test_chain_argument_checks(lib):
    """The chain's host-side validation, before any device work."""
    n = 3
    fmts = (W.Format * n)(*[fmt(256, 512) for _ in range(n)])
    assert lib.w4a16_chain_workspace_bytes(fmts, 0, 1) == 0
    assert lib.w4a16_chain_workspace_bytes(fmts, n, 17) == 0
    nb = lib.w4a16_chain_workspace_bytes(fmts, n, 1)
    # counters (n + 2) x 128 B, then the layer table
    assert nb % 256 == 0 and nb >= (n + 2) * 128 + n * 64
    X, Y = FAKE * 16, FAKE * 64

    def layers(waits, x=X, y=Y, packed=FAKE):
        return (W.ChainLayer * n)(*[W.ChainLayer(packed, W.packed_bytes(fmts[0]), x, y + i * 4096, lo, hi)
                                    for i, (lo, hi) in enumerate(waits)])

    info = W.ChainInfo()
    ok_waits = [(0, -1), (0, 0), (0, 1)]
    prep = lambda f, l, M=1, ws=FAKE, wsb=nb: lib.w4a16_chain_prepare(f, l, n, M, ws, wsb, ctypes.byref(info))
    assert prep(fmts, layers([(0, -1), (1, 1), (0, 1)])) == INVALID    # waits on itself
    assert prep(fmts, layers([(0, 0), (0, 0), (0, 1)])) == INVALID     # first layer waits on itself
    assert prep(fmts, layers([(0, -1), (-1, 0), (0, 1)])) == INVALID   # negative index
    assert prep(fmts, layers(ok_waits), M=0) == INVALID
    assert prep(fmts, layers(ok_waits), M=17) == INVALID
    assert prep(fmts, layers(ok_waits), ws=FAKE + 16) == MISALIGNED
    assert prep(fmts, layers(ok_waits), wsb=nb - 1) == SMALL
    assert prep(fmts, layers(ok_waits, x=X + 2)) == MISALIGNED
    assert prep(fmts, layers(ok_waits, packed=FAKE + 128)) == MISALIGNED
    assert prep(fmts, layers(ok_waits, y=X)) == INVALID                 # y overlaps x
    mixed = (W.Format * n)(fmt(256, 512), fmt(256, 512, bits=8), fmt(256, 512))
    assert prep(mixed, layers(ok_waits)) == UNSUPPORTED
    act = (W.Format * n)(fmt(256, 512), fmt(256, 512, act=True), fmt(256, 512))
    assert prep(act, layers(ok_waits)) == UNSUPPORTED
    ragged = (W.Format * n)(fmt(256, 512), fmt(256, 96, g=32), fmt(256, 512))
    assert prep(ragged, layers(ok_waits)) == UNSUPPORTED               # K not a multiple of 64
    bad = W.ChainInfo(n, 4, 128, 0, 1, 0)
    assert lib.w4a16_chain_run(ctypes.byref(bad), FAKE, None) == INVALID  # no work items


def test_gemv_grouped_argument_checks(lib):
    n = 3
    fs = [fmt(256, 512), fmt(128, 512), fmt(384, 512)]
    fa = (W.Format * n)(*fs)
    pa = (ctypes.c_void_p * n)(FAKE, FAKE * 2, FAKE * 3)
    ba = (ctypes.c_size_t * n)(*[W.packed_bytes(f) for f in fs])
    X = FAKE * 64
    ya = (ctypes.c_void_p * n)(FAKE * 128, FAKE * 256, FAKE * 512)
    call = lambda f=fa, p=pa, b=ba, k=n, x=X, y=ya, M=1, flags=0: lib.w4a16_gemv_grouped(f, p, b, k, x, y, M, flags,
                                                                                         None)
    assert call(k=0) == INVALID
    assert call(k=5) == INVALID
    assert call(M=17) == INVALID
    assert call(x=X + 2) == MISALIGNED
    assert call(flags=2 | 8) == INVALID                        # both variants
    assert call(flags=4) == INVALID                            # staging is not offered here
    mixed = (W.Format * n)(fs[0], fmt(128, 1024), fs[2])       # another K
    assert call(f=mixed, b=(ctypes.c_size_t * n)(*[W.packed_bytes(f) for f in mixed])) == INVALID
    act = (W.Format * n)(fs[0], fmt(128, 512, act=True), fs[2])
    assert call(f=act, b=(ctypes.c_size_t * n)(*[W.packed_bytes(f) for f in act])) == UNSUPPORTED
    small = (ctypes.c_size_t * n)(ba[0], ba[1] - 1, ba[2])
    assert call(b=small) == SMALL
    assert call(y=(ctypes.c_void_p * n)(FAKE * 128, X, FAKE * 512)) == INVALID  # y overlaps x
