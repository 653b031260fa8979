"""The Python binding on a caller-given stream: every call made on a side
stream (a torch stream object or a raw handle) gives bit for bit the result
of the same call on the current stream, including the calls that allocate
their own output or act-order workspace."""

import numpy as np
import pytest
import torch

from weight_only_bit_04_b300 import synth
from weight_only_bit_04_b300 import w4a16 as W

pytestmark = pytest.mark.gpu


def bits16(t):
    return t.cpu().numpy().view(np.uint16)


def test_side_stream_results_match_the_current_stream(cuda_ok):
    N, K, g = 384, 1024, 128
    xs = synth.activations_np(300, K, 0.01, 91)
    gidx = synth.act_order_g_idx(xs, g)
    fmt = W.make_format(N, K, g, False, True)
    w = synth.weights_cuda(N, K, 92)
    q, s, z = W.quantize_rtn(fmt, w, gidx)
    packed = W.pack(fmt, q, s, z, gidx)
    xv = torch.from_numpy(np.ascontiguousarray(xs[:4])).cuda()
    xm = torch.from_numpy(xs).cuda()
    ref = [W.gemv(fmt, packed, xv), W.gemm(fmt, packed, xm), W.dequant(fmt, packed), packed]
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    for stream in (side, side.cuda_stream):
        q2, s2, z2 = W.quantize_rtn(fmt, w, gidx, stream=stream)
        got = [W.gemv(fmt, packed, xv, stream=stream), W.gemm(fmt, packed, xm, stream=stream),
               W.dequant(fmt, packed, stream=stream), W.pack(fmt, q2, s2, z2, gidx, stream=stream)]
        side.synchronize()
        for a, b in zip(ref, got):
            if a.dtype == torch.uint8:
                assert torch.equal(a, b)
            else:
                assert np.array_equal(bits16(a), bits16(b))
    assert W.pipeline_timeouts() == 0


def test_tensors_must_be_on_the_current_device(cuda_ok):
    fmt = W.make_format(256, 512, 128)
    x = torch.zeros((1, 512), dtype=torch.float16)  # host tensor
    packed = torch.zeros(W.packed_bytes(fmt), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        W.gemv(fmt, packed, x)
