"""The no-allocation quantizer entry point, through the C ABI.

w4a16_quantize_rtn_noalloc serves callers that cannot allocate device memory
(code inside a framework or plugin that owns every device allocation, or a
path that must not allocate): its act-order scratch is a fixed array owned by
the library instead of caller workspace. It must give the same codes, scales
and zero points as the oracle's round-to-nearest quantizer and as
w4a16_quantize_rtn -- bit for bit, the tolerance every quantizer test here
uses -- on consecutive calls that reuse the shared array, at the largest K the
array admits, and when two host threads issue calls on one stream at once.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""

import ctypes
import threading

import numpy as np
import pytest
import torch

from oracle import w4a16_oracle as O
from weight_only_bit_04_b300 import synth
from weight_only_bit_04_b300 import w4a16 as W

pytestmark = pytest.mark.gpu

BUFFER_TOO_SMALL = 4


def _noalloc(fmt, w, g_idx, stream=None):
    lib = W.lib()
    N, K, G = fmt.N, fmt.K, fmt.G
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty((N, G), dtype=torch.float16, device=w.device)
    z = None if fmt.symmetric else torch.empty((N, G), dtype=torch.uint8, device=w.device)
    gi = None if g_idx is None else torch.as_tensor(g_idx, dtype=torch.int32).contiguous()
    st = lib.w4a16_quantize_rtn_noalloc(ctypes.byref(fmt), w.data_ptr(),
                                        None if gi is None else gi.data_ptr(), q.data_ptr(),
                                        s.data_ptr(), None if z is None else z.data_ptr(),
                                        (stream or torch.cuda.current_stream()).cuda_stream)
    assert st == 0, W.STATUS.get(st, st)
    return q, s, z


def _bits16(a):
    return np.ascontiguousarray(a).view(np.uint16)


def _assert_oracle(W16, g, sym, gidx, q, s, z):
    qo, so, zo = O.rtn_quantize(W16, g, sym, gidx)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(_bits16(s.cpu().numpy()), _bits16(so))
    if not sym:
        assert np.array_equal(z.cpu().numpy(), zo)


@pytest.mark.parametrize("N,K,g,sym,act", [(300, 4096, 128, False, True), (64, 2048, 32, True, True),
                                           (96, 1024, 64, False, False), (40, 65536, 128, False, True)])
def test_noalloc_quantizer_matches_oracle_twice(cuda_ok, N, K, g, sym, act):
    """Two calls in a row with new weights and a new act order each time
    (the second overwrites the shared column list), both bit-exact against
    the oracle; K = 65536 is the largest the fixed array holds."""
    fmt = W.make_format(N, K, g, sym, act)
    for call in range(2):
        W16 = synth.weights_np(N, K, synth.seed_for("noalloc-oracle", N, K, g, call))
        x = synth.activations_np(2, K, 0.01, synth.seed_for("noalloc-oracle-x", K, call))
        gidx = synth.act_order_g_idx(x, g) if act else None
        q, s, z = _noalloc(fmt, torch.from_numpy(W16).cuda(), gidx)
        torch.cuda.synchronize()
        _assert_oracle(W16, g, sym, gidx, q, s, z)


def test_noalloc_two_host_threads_share_one_stream(cuda_ok):
    """Two host threads issue act-order calls on one stream at the same time:
    each call's column list is copied and consumed by its own kernel before
    the other thread's copy lands, so every result matches the oracle."""
    N, K, g = 64, 4096, 128
    fmt = W.make_format(N, K, g, False, True)
    stream = torch.cuda.Stream()
    cases = []
    for t in range(2):
        for call in range(4):
            W16 = synth.weights_np(N, K, synth.seed_for("noalloc-thr", t, call))
            x = synth.activations_np(2, K, 0.01, synth.seed_for("noalloc-thr-x", t, call))
            cases.append((t, W16, torch.from_numpy(W16).cuda(), synth.act_order_g_idx(x, g)))
    torch.cuda.synchronize()
    outs = [None] * len(cases)
    errors = []
    start = threading.Barrier(2)

    def worker(t):
        try:
            start.wait()
            for i, (tt, _, wd, gidx) in enumerate(cases):
                if tt == t:
                    outs[i] = _noalloc(fmt, wd, gidx, stream)
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for (t, W16, _, gidx), (q, s, z) in zip(cases, outs):
        _assert_oracle(W16, g, False, gidx, q, s, z)


@pytest.mark.parametrize("N,K,g,sym,act", [(300, 4096, 128, False, True), (256, 1024, 32, True, True),
                                           (128, 512, 64, False, False)])
def test_noalloc_quantizer_matches_workspace_quantizer_twice(cuda_ok, N, K, g, sym, act):
    fmt = W.make_format(N, K, g, sym, act)
    for call in range(2):  # second call reuses the shared scratch with new inputs
        w = synth.weights_cuda(N, K, synth.seed_for("noalloc", N, K, g, call))
        x = synth.activations_np(4, K, 0.01, synth.seed_for("noalloc-x", K, call))
        gidx = synth.act_order_g_idx(x, g) if act else None
        q0, s0, z0 = W.quantize_rtn(fmt, w, gidx)
        q1, s1, z1 = _noalloc(fmt, w, gidx)
        torch.cuda.synchronize()
        assert torch.equal(q0, q1)
        assert torch.equal(s0.view(torch.int16), s1.view(torch.int16))
        if not sym:
            assert torch.equal(z0, z1)


def test_noalloc_rejects_k_beyond_its_scratch(cuda_ok):
    K = 65536 + 128
    fmt = W.make_format(8, K, 128, False, True)
    w = torch.zeros((8, K), dtype=torch.float16, device="cuda")
    q = torch.empty((8, K), dtype=torch.uint8, device="cuda")
    s = torch.empty((8, K // 128), dtype=torch.float16, device="cuda")
    z = torch.empty((8, K // 128), dtype=torch.uint8, device="cuda")
    gidx = (np.arange(K) // 128).astype(np.int32)
    st = W.lib().w4a16_quantize_rtn_noalloc(ctypes.byref(fmt), w.data_ptr(), gidx.ctypes.data, q.data_ptr(),
                                            s.data_ptr(), z.data_ptr(), None)
    assert st == BUFFER_TOO_SMALL
