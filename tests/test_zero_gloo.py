"""The ZeRO-sharded step's collective plumbing on CPU ranks (gloo, world
sizes 2 and 3): reduce-scatter of the flat gradient buffer, the rank's local
step on its pieces, all-gather of the parameters.  The local step here is the
oracle's 8-bit step (test only); after several steps every rank's parameters,
and the rank-owned states, equal the unsharded oracle run on the summed
gradients bit for bit.  Gradients are multiples of 2^-20 below 2^-8, so their
sums are exact in any order and every rank agrees on them."""

import os
import socket
import sys

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SIZES = [5000, 2048 * 3, 17, 0, 9000, 2048]
STEPS = 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _grad(i, n, rank, step):
    rng = np.random.default_rng(1000 * step + 37 * rank + i)
    return (rng.integers(-2 ** 12, 2 ** 12, n) * 2.0 ** -20).astype(np.float32)


def _param(i, n):
    return (np.random.default_rng(i).standard_normal(n) * 0.02).astype(np.float32)


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    from block_wise_dynamic_gb300.zero import ZeroAdam8bit

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    params = [torch.from_numpy(_param(i, n)) for i, n in enumerate(SIZES)]
    states = {}

    def oracle_local(pv, gv, t, hp):
        for j, (p, g) in enumerate(zip(pv, gv)):
            st = states.setdefault(j, oracle.state_init(p.numel()))
            res = oracle.adam8bit_step(p.numpy().copy(), g.numpy().copy(), *st,
                                       oracle.AdamHParams(lr=hp["lr"], step=t))
            p.copy_(torch.from_numpy(res[0]))
            states[j] = res[1:]

    opt = ZeroAdam8bit(params, lr=1e-3, reduce_op="sum", local_step=oracle_local)
    for step in range(1, STEPS + 1):
        opt.zero_grad()
        for i, (g, n) in enumerate(zip(opt.grad_views(), SIZES)):
            g.copy_(torch.from_numpy(_grad(i, n, rank, step)))
        opt.step()
    out[rank] = ([p.numpy().copy() for p in params], opt.layout.pieces[rank],
                 {j: tuple(np.asarray(x).copy() for x in s) for j, s in states.items()})
    dist.destroy_process_group()


def _unsharded(world):
    sys.path.insert(0, ROOT)
    import oracle

    ps = [_param(i, n) for i, n in enumerate(SIZES)]
    sts = [oracle.state_init(n) for n in SIZES]
    for step in range(1, STEPS + 1):
        for i, n in enumerate(SIZES):
            g = np.zeros(n, np.float32)
            for r in range(world):
                g = g + _grad(i, n, r, step)
            res = oracle.adam8bit_step(ps[i], g, *sts[i], oracle.AdamHParams(lr=1e-3, step=step))
            ps[i], sts[i] = res[0], res[1:]
    return ps, sts


def _check(world):
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        got = dict(out)
    ref_p, ref_st = _unsharded(world)
    for r in range(world):
        params, pieces, states = got[r]
        for a, b in zip(params, ref_p):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        for j, (ti, off, cnt) in enumerate(pieces):
            mc, ma, vc, va = states[j]
            rmc, rma, rvc, rva = ref_st[ti]
            b0, b1 = off // 2048, -(-(off + cnt) // 2048)
            assert np.array_equal(mc, rmc[off:off + cnt]) and np.array_equal(vc, rvc[off:off + cnt])
            assert np.array_equal(ma.view(np.uint32), rma[b0:b1].view(np.uint32))
            assert np.array_equal(va.view(np.uint32), rva[b0:b1].view(np.uint32))
    assert sum(len(got[r][1]) for r in range(world)) >= len([n for n in SIZES if n])


def test_zero_step_gloo_world2_matches_unsharded_oracle():
    _check(2)


def test_zero_step_gloo_world3_matches_unsharded_oracle():
    _check(3)


def _rank_autograd(rank, world, port, out):
    """A small model on each rank: autograd writes the gradients straight
    into the optimizer's flat buffer (p.grad are views of it)."""
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle
    from block_wise_dynamic_gb300.zero import ZeroAdam8bit

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.manual_seed(0)
    model = torch.nn.Sequential(torch.nn.Linear(48, 70), torch.nn.Tanh(), torch.nn.Linear(70, 5))
    params = list(model.parameters())
    states = {}

    def oracle_local(pv, gv, t, hp):
        for j, (p, g) in enumerate(zip(pv, gv)):
            st = states.setdefault(j, oracle.state_init(p.numel()))
            res = oracle.adam8bit_step(p.numpy().copy(), g.numpy().copy(), *st, oracle.AdamHParams(lr=hp["lr"], step=t))
            p.copy_(torch.from_numpy(res[0]))
            states[j] = res[1:]

    opt = ZeroAdam8bit(params, lr=1e-2, reduce_op="sum", local_step=oracle_local)
    flat = opt.flat_grad
    grads_seen = []
    for step in range(2):
        opt.zero_grad()
        x = torch.from_numpy(np.random.default_rng(10 * step + rank).standard_normal((16, 48)).astype(np.float32))
        model(x).square().mean().backward()
        assert all(p.grad.data_ptr() >= flat.data_ptr() for p in params)  # still views of the flat buffer
        grads_seen.append([p.grad.detach().clone().numpy() for p in params])
        opt.step()
    out[rank] = ([p.detach().numpy().copy() for p in params], grads_seen)
    dist.destroy_process_group()


def test_zero_step_takes_autograd_gradients_from_its_flat_buffer():
    """Two gloo ranks, a real backward pass each: every rank ends with the
    parameters of the unsharded oracle run on the sum of both ranks'
    gradients (the model and seeds are the same on both ranks)."""
    sys.path.insert(0, ROOT)
    import oracle

    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_autograd, args=(2, port, out), nprocs=2, join=True)
        got = dict(out)
    torch.manual_seed(0)
    model = torch.nn.Sequential(torch.nn.Linear(48, 70), torch.nn.Tanh(), torch.nn.Linear(70, 5))
    ps = [p.detach().numpy().reshape(-1).copy() for p in model.parameters()]
    sts = [oracle.state_init(p.size) for p in ps]
    for step in range(2):
        for i in range(len(ps)):
            g = (got[0][1][step][i].reshape(-1) + got[1][1][step][i].reshape(-1)).astype(np.float32)
            res = oracle.adam8bit_step(ps[i], g, *sts[i], oracle.AdamHParams(lr=1e-2, step=step + 1))
            ps[i], sts[i] = res[0], res[1:]
    for r in (0, 1):
        for a, b in zip(got[r][0], ps):
            assert np.array_equal(a.reshape(-1).view(np.uint32), b.view(np.uint32))


def _rank_checks(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    from block_wise_dynamic_gb300.zero import ZeroAdam8bit

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    a = torch.nn.Parameter(torch.zeros(10))
    b = torch.nn.Parameter(torch.zeros(3000))
    a.grad = torch.ones(10)
    res = []
    try:
        ZeroAdam8bit([a, b, a], reduce_op="sum", local_step=lambda *x: None)
        res.append("duplicate accepted")
    except ValueError:
        res.append("duplicate rejected")
    opt = ZeroAdam8bit([a, b], reduce_op="sum", grad_dtype=torch.float64, local_step=lambda *x: None)
    res.append(a.grad is None and b.grad is None)
    res.append(opt.grad_views()[1].dtype == torch.float64 and opt.grad_views()[1].shape == b.shape)
    out[rank] = res
    dist.destroy_process_group()


def test_zero_driver_argument_checks():
    """A parameter listed twice is refused; with a gradient dtype other than
    the parameters', stale gradients are cleared (the step reads only the
    flat buffer, through grad_views())."""
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_checks, args=(2, port, out), nprocs=2, join=True)
        got = dict(out)
    assert got[0] == got[1] == ["duplicate rejected", True, True]
