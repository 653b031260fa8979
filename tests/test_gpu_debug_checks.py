"""The debug flavor of the library (libw4a16_debug.so, -DW4A16_DEBUG_CHECKS)
on the small shapes: chained decode products over every code width, group
size and scheme and over 1, 5 and 16 tokens, with ragged N and slices, must
record no failed index check and still match the oracle. It runs in a child
process that loads the debug library in place of the release one.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import os, sys
import numpy as np
import torch
sys.path.insert(0, os.environ["W4A16_ROOT"])
from oracle import w4a16_oracle as O
from weight_only_bit_04_b300 import synth
from weight_only_bit_04_b300 import w4a16 as W
W.LIB_PATH = os.path.join(os.environ["W4A16_ROOT"], "weight_only_bit_04_b300", "libw4a16_debug.so")
assert W.debug_check_word() == 0, "the debug library did not load"
cases = 0
for bits in (3, 4, 8):
    for g, sym in ((128, False), (64, True), (32, False)):
        for M in (1, 5, 16):
            # three layers each reading the previous one's output, then one
            # with a ragged N (200 rows) reading the first input, no wait
            dims = [1024, 1152, 640, 1920]
            x0 = synth.activations_np(M, dims[0], 0.01, synth.seed_for("dbg-x", bits, g, M))
            xs, layers, refs = [torch.from_numpy(x0).cuda()], [], []
            for i in range(len(dims) - 1):
                K, N = dims[i], dims[i + 1]
                W16 = synth.weights_np(N, K, synth.seed_for("dbg-w", bits, g, i))
                q, s, z = O.rtn_quantize(W16, g, sym, bits=bits)
                fmt = W.make_format(N, K, g, sym, False, bits=bits)
                packed = W.pack(fmt, torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(),
                                None if sym else torch.from_numpy(z).cuda())
                y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
                layers.append((fmt, packed, xs[-1], y, None if i == 0 else (i - 1, i - 1)))
                refs.append((q, s, z, g))
                xs.append(y)
            W16 = synth.weights_np(200, dims[0], synth.seed_for("dbg-w", bits, g, "ragged"))
            qr, sr, zr = O.rtn_quantize(W16, g, sym, bits=bits)
            fmt = W.make_format(200, dims[0], g, sym, False, bits=bits)
            packed = W.pack(fmt, torch.from_numpy(qr).cuda(), torch.from_numpy(sr).cuda(),
                            None if sym else torch.from_numpy(zr).cuda())
            yr = torch.full((M, 200), float("nan"), dtype=torch.float16, device="cuda")
            layers.append((fmt, packed, xs[0], yr, None))
            W.Chain(layers, M).run()
            torch.cuda.synchronize()
            xi = x0
            for (fmt, _, _, y, _), (q, s, z, gg) in zip(layers[:-1], refs):
                got = y.cpu().numpy().astype(np.float64)
                y_ref, B = O.linear_ref(xi, O.dequant(q, s, z, gg))
                assert np.all(np.isfinite(got)), (bits, g, sym, M)
                assert O.error_ratio(got, y_ref, B).max() <= 1.0, (bits, g, sym, M)
                xi = y.cpu().numpy()
            y_ref, B = O.linear_ref(x0, O.dequant(qr, sr, zr, g))
            assert O.error_ratio(yr.cpu().numpy().astype(np.float64), y_ref, B).max() <= 1.0
            cases += 1
word = W.debug_check_word()
assert word == 0, f"index check 0x{word:x} failed"
assert W.pipeline_timeouts() == 0
print(f"debug checks clean over {cases} chains")
"""


def test_debug_build_records_no_failed_check(cuda_ok):
    lib = os.path.join(ROOT, "weight_only_bit_04_b300", "libw4a16_debug.so")
    if not os.path.exists(lib):
        pytest.fail("libw4a16_debug.so is missing: build it with `python -m weight_only_bit_04_b300.build --all`")
    env = dict(os.environ, W4A16_ROOT=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "debug checks clean" in r.stdout


def test_release_build_reports_checks_unsupported(cuda_ok):
    from weight_only_bit_04_b300 import w4a16 as W
    assert W.debug_check_word() is None
