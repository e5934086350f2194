"""The ZeRO-sharded 8-bit step on the GPU.

* Sharded equals unsharded: for P = 2, 3 and 8 the P ranks' local steps (one
  multi-tensor launch each over that rank's pieces, pointers offset into the
  full tensors, state for the pieces only) run one after another on one GPU;
  after several steps the parameters, and every rank's codes and absmax,
  equal the unsharded multi-tensor step's bit for bit.  Blocks are
  independent, so the split on block boundaries must change nothing.
* The driver class over a one-rank NCCL group (its collectives are then
  trivial, the kernel and the buffers real) matches the unsharded step.
The ranks never wait on one another: each local step is an ordinary launch.
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch

from block_wise_dynamic_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SIZES = [5000, 2048 * 3, 17, 70_001, 2048, 123_457, 1, 4096 + 2048]


@pytest.fixture(scope="module")
def bwd():
    from block_wise_dynamic_gb300 import build

    build.build()
    import block_wise_dynamic_gb300 as m

    m.init(0)
    return m


def _tensors(seed, gdt):
    ps = [W.gen_normal(n, 0.02, seed=seed + i, device=DEV) for i, n in enumerate(SIZES)]
    gs = [[W.gen_normal(n, 1e-3 * (i + 1), seed=seed + 100 * (s + 1) + i, device=DEV, dtype=gdt)
           for i, n in enumerate(SIZES)] for s in range(3)]
    return ps, gs


def _bits(t):
    if t.dtype == torch.float32:
        return t.cpu().view(torch.int32).numpy()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.cpu().view(torch.int16).numpy()
    return t.cpu().numpy()


@pytest.mark.parametrize("world", [2, 3, 8])
@pytest.mark.parametrize("gdt,pdt", [(torch.bfloat16, torch.float32), (torch.float32, torch.float32),
                                     (torch.float16, torch.float32), (torch.bfloat16, torch.bfloat16),
                                     (torch.float16, torch.float16)])
def test_sharded_steps_equal_the_unsharded_step(bwd, world, gdt, pdt):
    from block_wise_dynamic_gb300.zero import ShardLayout

    ps, gsteps = _tensors(11, gdt)
    ps = [p.to(pdt) for p in ps]
    ref = [p.clone() for p in ps]
    ref_st = [bwd.state_init(n, DEV) for n in SIZES]
    L = ShardLayout(SIZES, world)
    shard_st = [[bwd.state_init(c, DEV) for _, _, c in L.pieces[r]] for r in range(world)]
    for t, gs in enumerate(gsteps, start=1):
        bwd.MultiTensorArgs(ref, gs, *[[s[k] for s in ref_st] for k in range(4)]).step(lr=1e-3, step=t)
        for r in range(world):
            pcs = L.pieces[r]
            if not pcs:
                continue
            bwd.MultiTensorArgs([ps[i][o:o + c] for i, o, c in pcs], [gs[i][o:o + c] for i, o, c in pcs],
                                *[[s[k] for s in shard_st[r]] for k in range(4)]).step(lr=1e-3, step=t)
    torch.cuda.synchronize()
    for a, b in zip(ps, ref):
        assert np.array_equal(_bits(a), _bits(b))
    for r in range(world):
        for (i, o, c), st in zip(L.pieces[r], shard_st[r]):
            b0, b1 = o // 2048, -(-(o + c) // 2048)
            want = (ref_st[i][0][o:o + c], ref_st[i][1][b0:b1], ref_st[i][2][o:o + c], ref_st[i][3][b0:b1])
            for got, w in zip(st, want):
                assert np.array_equal(_bits(got), _bits(w))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _one_rank(index, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import block_wise_dynamic_gb300 as bwd
    from block_wise_dynamic_gb300.zero import ZeroAdam8bit

    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    ps, gsteps = _tensors(23, torch.bfloat16)
    ref = [p.clone() for p in ps]
    ref_st = [bwd.state_init(n, DEV) for n in SIZES]
    params = [torch.nn.Parameter(p.clone()) for p in ps]
    opt = ZeroAdam8bit(params, lr=1e-3, grad_dtype=torch.bfloat16)
    for t, gs in enumerate(gsteps, start=1):
        bwd.MultiTensorArgs(ref, gs, *[[s[k] for s in ref_st] for k in range(4)]).step(lr=1e-3, step=t)
        opt.zero_grad()
        for v, g in zip(opt.grad_views(), gs):
            v.copy_(g)
        work = opt.step(async_gather=(t == 2))
        if work is not None:
            work.wait()
    torch.cuda.synchronize()
    same = all(torch.equal(p.detach().view(-1), r) for p, r in zip(params, ref))
    pcs = opt.layout.pieces[0]
    st_same = all(torch.equal(st[0], ref_st[i][0][o:o + c]) and torch.equal(st[2], ref_st[i][2][o:o + c])
                  for (i, o, c), st in zip(pcs, opt.state))
    sd = opt.state_dict()
    opt.load_state_dict(sd)
    out["result"] = (same, st_same, len(pcs), sd["step"])
    dist.destroy_process_group()


def test_zero_driver_on_a_one_rank_nccl_group():
    import torch.multiprocessing as mp

    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_one_rank, args=(_free_port(), out), nprocs=1, join=True)
        same, st_same, npieces, step = out["result"]
    assert same and st_same and npieces == len([n for n in SIZES if n]) and step == 3
