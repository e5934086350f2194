"""The library's calls can be captured in a CUDA graph (after bwd.init has
uploaded the tables) and a replay computes exactly what the eager calls
compute.  A captured step freezes its kernel parameters, hyper-parameters and
step number included; the quantize / dequantize pair has none that change,
so its graph can be replayed on new data in the same buffers."""

import numpy as np
import pytest
import torch

from block_wise_dynamic_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bwd():
    from block_wise_dynamic_gb300 import build

    build.build()
    import block_wise_dynamic_gb300 as m

    m.init(0)
    return m


def test_graph_replay_matches_eager(bwd):
    dev = torch.device("cuda", 0)
    sizes = [3 * 2048 + 11, 2048, 777]
    ps = [W.gen_normal(n, 0.02, seed=70 + i, device=dev) for i, n in enumerate(sizes)]
    gs = [W.gen_normal(n, 1e-3, seed=80 + i, device=dev, dtype=torch.bfloat16) for i, n in enumerate(sizes)]
    sts = [bwd.state_init(n, dev) for n in sizes]
    # identical copies for the eager run
    pe = [p.clone() for p in ps]
    se = [tuple(x.clone() for x in s) for s in sts]
    x = W.quant_input(5 * 2048 + 3, seed=9, device=dev)
    codes = torch.empty(x.numel(), dtype=torch.uint8, device=dev)
    absmax = torch.empty(bwd.num_blocks(x.numel()), dtype=torch.float32, device=dev)
    y = torch.empty_like(x)

    mt = bwd.MultiTensorArgs(ps, gs, *[[s[k] for s in sts] for k in range(4)])
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):  # warm the argument caches off the capture
        bwd.quantize_blockwise(x, "signed", codes, absmax)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bwd.quantize_blockwise(x, "signed", codes, absmax)
        bwd.dequantize_blockwise(codes, absmax, "signed", out=y)
        mt.step(lr=1e-3, step=1)
    g.replay()
    torch.cuda.synchronize(dev)

    ce, ae = bwd.quantize_blockwise(x, "signed")
    ye = bwd.dequantize_blockwise(ce, ae, "signed")
    bwd.adam8bit_step_multi(pe, gs, *[[s[k] for s in se] for k in range(4)], lr=1e-3, step=1)
    torch.cuda.synchronize(dev)
    assert torch.equal(codes, ce) and torch.equal(absmax, ae) and torch.equal(y, ye)
    for a, b in zip(ps, pe):
        assert torch.equal(a, b)
    for a, b in zip(sts, se):
        for u, v in zip(a, b):
            assert torch.equal(u, v)

    # new data in the captured buffers, same graph
    x.copy_(W.quant_input(x.numel(), seed=10, device=dev))
    g.replay()
    torch.cuda.synchronize(dev)
    ce, ae = bwd.quantize_blockwise(x, "signed")
    assert torch.equal(codes, ce) and torch.equal(absmax, ae)
    assert np.array_equal(y.cpu().numpy(), bwd.dequantize_blockwise(ce, ae, "signed").cpu().numpy())
