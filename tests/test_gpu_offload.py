"""Host-buffer steps (block_wise_dynamic_gb300.offload): pipelining the
copies around the multi-tensor step changes nothing in the result."""

import pytest
import torch

from block_wise_dynamic_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_pipelined_host_step_equals_device_step():
    import block_wise_dynamic_gb300 as bwd
    from block_wise_dynamic_gb300.offload import PipelinedHostStep

    sizes = [5000, 2048 * 7, 123, 2048 * 3 + 1, 40_000]
    ps0 = [W.gen_normal(n, 0.02, 100 + i) for i, n in enumerate(sizes)]
    gsteps = [[W.gen_normal(n, 1e-3, 1000 * t + i, dtype=torch.bfloat16) for i, n in enumerate(sizes)]
              for t in range(3)]
    # reference: device-only steps
    rp = [p.to(DEV) for p in ps0]
    rg = [torch.empty(n, dtype=torch.bfloat16, device=DEV) for n in sizes]
    rs = [bwd.state_init(n, DEV) for n in sizes]
    ra = bwd.MultiTensorArgs(rp, rg, *[[s[k] for s in rs] for k in range(4)])
    # pipelined host-buffer steps, 2 tensors per chunk at most
    dp = [p.to(DEV) for p in ps0]
    dg = [torch.empty(n, dtype=torch.bfloat16, device=DEV) for n in sizes]
    ds = [bwd.state_init(n, DEV) for n in sizes]
    hg = [torch.empty(n, dtype=torch.bfloat16, pin_memory=True) for n in sizes]
    hp = [torch.empty(n, dtype=torch.float32, pin_memory=True) for n in sizes]
    pipe = PipelinedHostStep(dp, dg, *[[s[k] for s in ds] for k in range(4)], hg, hp, chunk_bytes=30_000)
    assert len(pipe.chunks) >= 3
    for t in range(3):
        for i in range(len(sizes)):
            rg[i].copy_(gsteps[t][i])
            hg[i].copy_(gsteps[t][i])
        ra.step(lr=1e-3, step=t + 1)
        pipe.step(lr=1e-3, step=t + 1)
        torch.cuda.synchronize()
        for i in range(len(sizes)):
            assert torch.equal(hp[i], rp[i].cpu())
            for a, b in zip(ds[i], rs[i]):
                assert torch.equal(a, b)
