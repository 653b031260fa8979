"""The failure paths of the library, exercised without a device fault.

"AWQ + GPTQ Quantization, in depth", section "Failure modes", names the
silent kernel fallback; the library's answer is that a failed launch is
reported (W4A16_ERR_CUDA and the cudaError_t) and that no in-kernel wait can
hang: every pipeline wait is bounded, and a wait that gives up stops its
launch, is counted, and leaves the outputs undefined. Here a launch failure
is injected on the host (w4a16_debug_fail_next_launch: nothing is launched),
and the waits of a chained launch are made to give up by a wait limit far
shorter than the work they cover (w4a16_set_wait_limit_ns). After each, a
normal call on the same context must still match the oracle.
"""

import numpy as np
import pytest
import torch

from oracle import w4a16_oracle as O
from weight_only_bit_04_b300 import synth
from weight_only_bit_04_b300 import w4a16 as W

pytestmark = pytest.mark.gpu

ERR_CUDA = 5
CUDA_ERROR_INVALID_CONFIGURATION = 9


def assert_within(y, y_ref, B):
    y = y.astype(np.float64)
    assert np.all(np.isfinite(y)), "non-finite output"
    assert O.error_ratio(y, y_ref, B).max() <= 1.0


def oracle_layer(N, K, M, seed):
    W16 = synth.weights_np(N, K, synth.seed_for("failure", N, K, seed))
    q, s, z = O.rtn_quantize(W16, 128, False)
    fmt = W.make_format(N, K, 128, False, False)
    packed = W.pack(fmt, torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), torch.from_numpy(z).cuda())
    x = synth.activations_np(M, K, 0.01, synth.seed_for("failure-x", K, M, seed))
    y_ref, B = O.linear_ref(x, O.dequant(q, s, z, 128))
    return fmt, packed, torch.from_numpy(x).cuda(), y_ref, B


@pytest.mark.parametrize("call", ["gemv", "gemm", "dequant", "chain"])
def test_injected_launch_error_is_reported_and_nothing_runs(cuda_ok, call):
    M = 32 if call == "gemm" else 1
    fmt, packed, x, y_ref, B = oracle_layer(256, 1024, M, 1)
    chain = None
    if call == "chain":
        y = torch.full((M, fmt.N), float("nan"), dtype=torch.float16, device="cuda")
        chain = W.Chain([(fmt, packed, x, y, None)], M)

    def run():
        if call == "gemv":
            return W.gemv(fmt, packed, x)
        if call == "gemm":
            return W.gemm(fmt, packed, x)
        if call == "dequant":
            return W.dequant(fmt, packed)
        chain.run()
        return y

    torch.cuda.synchronize()
    W.debug_fail_next_launch(CUDA_ERROR_INVALID_CONFIGURATION)
    with pytest.raises(W.W4A16Error) as info:
        run()
    assert info.value.status == ERR_CUDA
    assert info.value.cuda_error == CUDA_ERROR_INVALID_CONFIGURATION
    assert W.lib().w4a16_last_cuda_error() == CUDA_ERROR_INVALID_CONFIGURATION
    if chain is not None:
        torch.cuda.synchronize()
        assert torch.isnan(y.float()).all()  # the chained launch did not run
    # one-shot: the next call launches and is right
    out = run()
    torch.cuda.synchronize()
    if call == "dequant":
        assert torch.isfinite(out.float()).all()
    else:
        assert_within(out.cpu().numpy(), y_ref, B)
    assert W.pipeline_timeouts() == 0


def test_injected_error_can_be_cleared(cuda_ok):
    fmt, packed, x, y_ref, B = oracle_layer(128, 512, 1, 2)
    W.debug_fail_next_launch(CUDA_ERROR_INVALID_CONFIGURATION)
    W.debug_fail_next_launch(0)
    assert_within(W.gemv(fmt, packed, x).cpu().numpy(), y_ref, B)


def test_chain_waits_give_up_under_a_tiny_limit_and_the_context_recovers(cuda_ok):
    """A chain of four 28672x8192 layers (120 MB of codes each, tens of
    microseconds to stream), each reading the previous one's output: with a
    2-microsecond wait limit the wait for a previous layer gives up. The
    launch must return, count the timeouts, and leave the dependent layers'
    outputs unwritten (still NaN). With the default limit back, the same chain
    must run clean; sampled rows of every layer are checked against the oracle
    applied to the input that layer read."""
    N, K = 28672, 8192
    rows = np.arange(0, N, 97)  # 296 rows spread over every row block
    layers, ys, refs = [], [], []
    x = torch.from_numpy(synth.activations_np(1, K, 0.01, synth.seed_for("failure-chain-x"))).cuda()
    xin = x
    for i in range(4):
        fmt = W.make_format(N, K, 128, False, False)
        q, s, z = W.quantize_rtn(fmt, synth.weights_cuda(N, K, synth.seed_for("failure-chain", i)))
        packed = W.pack(fmt, q, s, z)
        y = torch.empty((1, N), dtype=torch.float16, device="cuda")
        layers.append((fmt, packed, xin, y, None if i == 0 else (i - 1, i - 1)))
        ys.append(y)
        refs.append((q[rows].cpu().numpy(), s[rows].cpu().numpy(), z[rows].cpu().numpy()))
        xin = y
        K = N  # the next layer reads this one's output
    chain = W.Chain(layers, 1)
    assert W.pipeline_timeouts() == 0

    for y in ys:
        y.fill_(float("nan"))
    prev = W.set_wait_limit_ns(2000)
    try:
        chain.run()
        torch.cuda.synchronize()  # the launch returns
    finally:
        W.set_wait_limit_ns(prev)
    assert W.pipeline_timeouts() > 0
    for y in ys[1:]:
        assert torch.isnan(y.float()).all(), "a layer ran although its dependency wait gave up"

    for y in ys:
        y.fill_(float("nan"))
    chain.run()
    torch.cuda.synchronize()
    assert W.pipeline_timeouts() == 0
    xi = x.cpu().numpy()
    for (q, s, z), y in zip(refs, ys):
        got = y.cpu().numpy()
        assert np.all(np.isfinite(got.astype(np.float64)))
        y_ref, B = O.linear_ref(xi, O.dequant(q, s, z, 128))
        assert_within(got[:, rows], y_ref, B)
        xi = got  # the next layer read what this one wrote


def test_wait_limit_setter_returns_the_previous_limit(cuda_ok):
    default = W.set_wait_limit_ns(0)
    assert default == 1_000_000_000
    assert W.set_wait_limit_ns(5000) == default
    assert W.set_wait_limit_ns(0) == 5000
    assert W.set_wait_limit_ns(0) == default
