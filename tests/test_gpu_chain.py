"""Chained decode products (w4a16_chain_*): one persistent launch over a list
of layers, each layer waiting on device counters for the layers it reads.

Each layer's output is checked against the oracle applied to the input that
layer actually read, and against the single-launch product within the same
bound; repeated runs must agree bit for bit (the K slices of a row group are
added in slice order). Outputs are poisoned with NaN before every run, so a
layer that read its input before the producer had written it shows up.
"""

import numpy as np
import pytest
import torch

from oracle import w4a16_oracle as O
from weight_only_bit_04_b300 import synth
from weight_only_bit_04_b300 import w4a16 as W

pytestmark = pytest.mark.gpu


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_within(y, y_ref, B):
    y = y.astype(np.float64)
    assert np.all(np.isfinite(y)), "non-finite output"
    r = O.error_ratio(y, y_ref, B)
    assert r.max() <= 1.0, f"max error ratio {r.max():.3f}"


def make_layer(N, K, g, sym, bits, seed):
    fmt = W.make_format(N, K, g, sym, False, bits=bits)
    w = synth.weights_cuda(N, K, seed)
    q, s, z = W.quantize_rtn(fmt, w)
    return fmt, W.pack(fmt, q, s, z), (q, s, z)


def single(fmt, packed, x):
    return W.gemv(fmt, packed, x)


@pytest.mark.parametrize("bits", [3, 4, 8])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_sequential_stack_with_real_data_flow(cuda_ok, bits, M):
    """y of layer i is the x of layer i+1: every layer waits for its predecessor."""
    dims = [1024, 2048, 1024, 512, 1536]
    layers, chain_layers = [], []
    x0 = synth.activations_cuda(M, dims[0], 0.01, 101)
    x = x0
    for i in range(len(dims) - 1):
        K, N = dims[i], dims[i + 1]
        fmt, packed, qsz = make_layer(N, K, 128, False, bits, synth.seed_for("chain", bits, i))
        y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        layers.append((fmt, packed, qsz, x, y))
        chain_layers.append((fmt, packed, x, y, None if i == 0 else (i - 1, i - 1)))
        x = y
    chain = W.Chain(chain_layers, M)
    first = None
    for _ in range(3):  # re-runs reset the counters
        for *_, y in layers:
            y.fill_(float("nan"))
        chain.run()
        torch.cuda.synchronize()
        assert W.pipeline_timeouts() == 0
        outs = [yi.cpu().numpy() for *_, yi in layers]
        if first is None:
            first = outs
        for a, b in zip(first, outs):  # deterministic
            assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
        for (fmt, packed, (q, s, z), xi, yi), got in zip(layers, outs):
            y_ref, B = O.linear_ref(xi.cpu().numpy(), O.dequant(q.cpu().numpy(), s.cpu().numpy(),
                                                                z.cpu().numpy(), 128))
            assert_within(got, y_ref, B)
            assert_within(single(fmt, packed, xi).cpu().numpy(), y_ref, B)


@pytest.mark.parametrize("g", [32, 64, 128])
@pytest.mark.parametrize("sym", [False, True])
def test_decoder_layer_dag(cuda_ok, g, sym):
    """q, k, v read one input; o waits for q..v; gate and up wait for o; down
    waits for gate and up; the next layer's q, k, v wait for down -- two
    layers of a small decoder, ragged N included."""
    M, H, F = 3, 512, 1408
    shapes = [("q", H, H), ("k", 200, H), ("v", 200, H), ("o", H, H), ("gate", F, H), ("up", F, H), ("down", H, F)]
    x_in = synth.activations_cuda(M, H, 0.01, 7)
    chain_layers, checks = [], []
    base = 0
    prev_down = None
    for layer in range(2):
        ys = {}
        for name, N, K in shapes:
            fmt, packed, qsz = make_layer(N, K, g, sym, 4, synth.seed_for("dag", layer, name, g, sym))
            y = torch.empty((M, N), dtype=torch.float16, device="cuda")
            if name in ("q", "k", "v"):
                x = x_in if prev_down is None else prev_down
                wait = None if prev_down is None else (base - 1, base - 1)
            elif name == "o":
                # attention is not modelled: o reads q's output (K = H), after q..v
                x, wait = ys["q"], (base + 0, base + 2)
            elif name in ("gate", "up"):
                x, wait = ys["o"], (base + 3, base + 3)
            else:  # down reads gate's output (K = F), after gate and up
                x, wait = ys["gate"], (base + 4, base + 5)
            ys[name] = y
            chain_layers.append((fmt, packed, x, y, wait))
            checks.append((fmt, packed, qsz, x, y))
        prev_down = ys["down"]
        base += len(shapes)
    chain = W.Chain(chain_layers, M)
    for _ in range(2):
        for *_, y in checks:
            y.fill_(float("nan"))
        chain.run()
        torch.cuda.synchronize()
        assert W.pipeline_timeouts() == 0
        for fmt, packed, (q, s, z), x, y in checks:
            got = y.cpu().numpy()
            zz = np.full(s.shape, 8, np.uint8) if sym else z.cpu().numpy()
            y_ref, B = O.linear_ref(x.cpu().numpy(), O.dequant(q.cpu().numpy(), s.cpu().numpy(), zz, g))
            assert_within(got, y_ref, B)


@pytest.mark.parametrize("bits", [4, 3, 8])
def test_llama2_7b_step_full_size(cuda_ok, bits):
    """One decode step of the 7B-shaped stack (32 x 7 linears; 3.37 GB at 4
    bits, 2.56 GB at 3, 6.63 GB at 8) as one chain with the decoder's
    dependencies; sampled layers within the bound of the oracle on sampled
    rows, and two runs bit for bit equal."""
    M = 1
    dev = torch.device("cuda")
    xs = {K: synth.activations_cuda(M, K, synth.LLAMA2_7B_OUTLIER_FRAC, synth.seed_for("c7b", K)) for K in (4096, 11008)}
    chain_layers, keep = [], []
    for layer in range(synth.LLAMA2_7B_LAYERS):
        base = len(chain_layers)
        for name, N, K in synth.LLAMA2_7B_LINEARS:
            fmt, packed, qsz = make_layer(N, K, 128, False, bits, synth.seed_for("c7b", bits, layer, name))
            y = torch.empty((M, N), dtype=torch.float16, device=dev)
            wait = {"q": (base - 1, base - 1), "k": (base - 1, base - 1), "v": (base - 1, base - 1),
                    "o": (base, base + 2), "gate": (base + 3, base + 3), "up": (base + 3, base + 3),
                    "down": (base + 4, base + 5)}[name]
            if layer == 0 and name in ("q", "k", "v"):
                wait = None
            chain_layers.append((fmt, packed, xs[K], y, wait))
            sample = layer in (0, 17, 31) or (layer == 9 and name == "down")
            keep.append((fmt, packed, xs[K], y, qsz if sample else None))
    chain = W.Chain(chain_layers, M)
    runs = []
    for _ in range(2):
        for _, _, _, y, _ in keep:
            y.fill_(float("nan"))
        chain.run()
        torch.cuda.synchronize()
        assert W.pipeline_timeouts() == 0
        runs.append([y.cpu().numpy() for _, _, _, y, _ in keep])
    for a, b in zip(*runs):
        assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    rng = np.random.default_rng(3)
    for (fmt, packed, x, y, qsz), got in zip(keep, runs[0]):
        if qsz is None:
            continue
        rows = rng.choice(fmt.N, 64, replace=False)
        rt = torch.from_numpy(rows).cuda()
        q, s, z = (t[rt].cpu().numpy() for t in qsz)
        y_ref, B = O.linear_ref(x.cpu().numpy(), O.dequant(q, s, z, 128))
        assert_within(got[:, rows], y_ref, B)
