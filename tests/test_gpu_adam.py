"""GPU parity: the fused 8-bit Adam step through the C ABI against the
oracle's step (sections 一 and 二 of "8-BIT OPTIMIZERS VIA BLOCK-WISE
QUANTIZATION").

Tolerance of a step taken from identical input state: parameters rtol 1e-5,
atol 1e-7; at most 1e-4 of the codes may differ, each by at most one index;
absmax rtol 1e-6.  The kernel computes the moments with the same binary32
operations in the same order as the oracle, so the codes and absmax of the
new state are bit-identical, and the tests assert that as well; the
parameter update uses approximate sqrt and division and stays within a few
ulps of the update term, far inside the parameter tolerance."""

import numpy as np
import pytest
import torch

import oracle
from oracle.adam import widen_bf16
from block_wise_dynamic_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
B = 2048
U32 = np.uint32


@pytest.fixture(scope="module")
def bwd():
    from block_wise_dynamic_gb300 import build

    build.build()
    import block_wise_dynamic_gb300 as m

    m.init(0)
    return m


def g_to_np(g: torch.Tensor) -> np.ndarray:
    g = g.detach().cpu()
    if g.dtype == torch.bfloat16:
        return widen_bf16(g.view(torch.int16).numpy().view(np.uint16))
    return g.numpy()


def compare_step(gpu, ref, exact=True):
    """gpu, ref: (p, mc, ma, vc, va) numpy tuples of one tensor."""
    p, mc, ma, vc, va = gpu
    rp, rmc, rma, rvc, rva = ref
    np.testing.assert_allclose(p, rp, rtol=1e-5, atol=1e-7)
    for c, rc in ((mc, rmc), (vc, rvc)):
        d = np.abs(c.astype(np.int32) - rc.astype(np.int32))
        assert d.max(initial=0) <= 1
        assert np.count_nonzero(d) <= max(1e-4 * c.size, 0)
    np.testing.assert_allclose(ma, rma, rtol=1e-6, atol=0)
    np.testing.assert_allclose(va, rva, rtol=1e-6, atol=0)
    # the update term is at most ~lr; its few-ulp error bounds |p - rp|
    assert np.all(np.abs(p.astype(np.float64) - rp) <= 3e-8 + 4e-7 * np.abs(rp))
    if exact:
        assert np.array_equal(mc, rmc) and np.array_equal(vc, rvc)
        assert np.array_equal(ma.view(U32), rma.view(U32)) and np.array_equal(va.view(U32), rva.view(U32))


def random_state(n, seed, m_scale=1e-3, v_scale=1e-6):
    """A non-trivial 8-bit state: random moments quantized by the oracle."""
    rng = np.random.default_rng(seed)
    m = (rng.standard_normal(n) * m_scale * 10.0 ** rng.uniform(-2, 0, n)).astype(np.float32)
    v = (rng.standard_normal(n) ** 2 * v_scale * 10.0 ** rng.uniform(-3, 0, n)).astype(np.float32)
    mc, ma = oracle.quantize_blockwise(m, True)
    vc, va = oracle.quantize_blockwise(v, False)
    return mc, ma, vc, va


def to_dev(*arrs):
    return [torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in arrs]


def run_gpu(bwd, p, g, st, hp: oracle.AdamHParams):
    tp, tmc, tma, tvc, tva = to_dev(p, *st)
    tg = g.to(DEV)
    bwd.adam8bit_step(tp, tg, tmc, tma, tvc, tva, lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2,
                      eps=hp.eps, step=hp.step)
    torch.cuda.synchronize()
    return tuple(t.cpu().numpy() for t in (tp, tmc, tma, tvc, tva))


@pytest.mark.parametrize("gdt", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("n", [1, 2047, 2048, 2049, 5 * B + 77, 1 << 20])
def test_single_step_from_identical_state(bwd, n, gdt):
    p = W.gen_normal(n, 0.02, seed=n).numpy()
    g = W.gen_normal(n, 1e-2, seed=n + 1, dtype=gdt)
    st = random_state(n, n + 2)
    for t in (1, 7):
        hp = oracle.AdamHParams(lr=1e-3, step=t)
        got = run_gpu(bwd, p, g, st, hp)
        ref = oracle.adam8bit_step(p, g_to_np(g), *st, hp)
        compare_step(got, ref)


def test_first_step_from_state_init(bwd):
    n = 3 * B + 5
    mc, ma, vc, va = bwd.state_init(n, DEV)
    smc, sma, svc, sva = oracle.state_init(n)
    assert np.array_equal(mc.cpu().numpy(), smc) and np.array_equal(vc.cpu().numpy(), svc)
    assert np.all(ma.cpu().numpy() == 0) and np.all(va.cpu().numpy() == 0)
    p = W.gen_normal(n, 0.02, 1).numpy()
    g = W.gen_normal(n, 1e-2, 2)
    got = run_gpu(bwd, p, g, (smc, sma, svc, sva), oracle.AdamHParams(step=1))
    ref = oracle.adam8bit_step(p, g_to_np(g), smc, sma, svc, sva, oracle.AdamHParams(step=1))
    compare_step(got, ref)


def test_ten_step_trajectory_1m(bwd):
    """The 1,048,576-element workload for 10 steps with fresh gradients each
    step, GPU and oracle each carrying their own state."""
    wl = W.workload("adam_1m")
    n = wl.sizes[0]
    p0 = W.gen_normal(n, 0.02, seed=0)
    tp = p0.to(DEV)
    mc, ma, vc, va = bwd.state_init(n, DEV)
    rp = p0.numpy().copy()
    rst = oracle.state_init(n)
    for t in range(1, wl.steps + 1):
        g = W.gen_normal(n, wl.grad_std[0], seed=1000 + t)
        bwd.adam8bit_step(tp, g.to(DEV), mc, ma, vc, va, lr=wl.lr, step=t)
        hp = oracle.AdamHParams(lr=wl.lr, step=t)
        rp, *rst = oracle.adam8bit_step(rp, g.numpy(), *rst, hp)
    torch.cuda.synchronize()
    got = (tp.cpu().numpy(), mc.cpu().numpy(), ma.cpu().numpy(), vc.cpu().numpy(), va.cpu().numpy())
    compare_step(got, (rp, *rst))


def _multi_case(bwd, sizes, gdt, seed, offsets=None):
    """Run one multi-tensor step on the GPU and the oracle per tensor."""
    rng = np.random.default_rng(seed)
    host = []
    dev = []
    for i, n in enumerate(sizes):
        off = 0 if offsets is None else offsets[i]
        p = W.gen_normal(n, 0.02, seed * 7919 + i).numpy()
        g = W.gen_normal(n, float(10.0 ** rng.uniform(-5, -1)), seed * 7919 + 5000 + i, dtype=gdt)
        st = random_state(n, seed * 31 + i) if n else oracle.state_init(0)
        host.append((p, g_to_np(g), *st))
        # optional element offset makes the buffers unaligned
        tp = torch.empty(n + off, dtype=torch.float32, device=DEV)[off:]
        tp.copy_(torch.from_numpy(p))
        tg = torch.empty(n + off, dtype=gdt, device=DEV)[off:]
        tg.copy_(g)
        tmc = torch.empty(n + off, dtype=torch.uint8, device=DEV)[off:]
        tmc.copy_(torch.from_numpy(st[0]))
        tvc = torch.empty(n + off, dtype=torch.uint8, device=DEV)[off:]
        tvc.copy_(torch.from_numpy(st[2]))
        tma, tva = to_dev(st[1], st[3])
        dev.append((tp, tg, tmc, tma, tvc, tva))
    hp = oracle.AdamHParams(lr=2e-3, beta1=0.9, beta2=0.99, eps=1e-8, step=3)
    lists = list(zip(*dev))
    bwd.adam8bit_step_multi(*lists, lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, step=hp.step)
    torch.cuda.synchronize()
    for h, d in zip(host, dev):
        ref = oracle.adam8bit_step(*h, hp)
        got = tuple(x.cpu().numpy() for x in (d[0], d[2], d[3], d[4], d[5]))
        compare_step(got, ref)


@pytest.mark.parametrize("gdt", [torch.float32, torch.bfloat16, torch.float16])
def test_multi_ragged_list(bwd, gdt):
    rng = np.random.default_rng(5)
    sizes = [int(s) for s in rng.integers(1, 40_000, 60)] + [0, 2048, 4096, 1, 0, 2049]
    _multi_case(bwd, sizes, gdt, seed=11)


def test_multi_more_tensors_than_one_launch_holds(bwd):
    rng = np.random.default_rng(6)
    sizes = [int(s) for s in rng.integers(1, 3000, 1000)]
    _multi_case(bwd, sizes, torch.float32, seed=12)


def test_multi_with_unaligned_tensors(bwd):
    sizes = [2048 * 3, 5000, 2048, 7777]
    _multi_case(bwd, sizes, torch.bfloat16, seed=13, offsets=[1, 0, 3, 2])


def test_optimizer_drop_in_and_exact_resume(bwd):
    """Adam8bit replaces torch.optim.Adam; saving its state after k steps and
    resuming reproduces the uninterrupted run bit for bit."""
    torch.manual_seed(0)
    model = torch.nn.Sequential(torch.nn.Linear(64, 300), torch.nn.ReLU(), torch.nn.Linear(300, 10)).to(DEV)
    ref_model = [p.detach().cpu().numpy().ravel().copy() for p in model.parameters()]
    opt = bwd.Adam8bit(model.parameters(), lr=1e-3)
    ref_state = [oracle.state_init(p.size) for p in ref_model]
    x = torch.randn(128, 64, device=DEV)
    y = torch.randint(0, 10, (128,), device=DEV)
    saved = None
    for t in range(1, 7):
        opt.zero_grad()
        loss = torch.nn.functional.cross_entropy(model(x), y)
        loss.backward()
        grads = [p.grad.detach().cpu().numpy().ravel() for p in model.parameters()]
        opt.step()
        hp = oracle.AdamHParams(lr=1e-3, step=t)
        for i, g in enumerate(grads):
            ref_model[i], *ref_state[i] = oracle.adam8bit_step(ref_model[i], g, *ref_state[i], hp)
        for i, p in enumerate(model.parameters()):
            st = opt.state[p]
            got = (p.detach().cpu().numpy().ravel(), st["m_codes"].cpu().numpy(), st["m_absmax"].cpu().numpy(),
                   st["v_codes"].cpu().numpy(), st["v_absmax"].cpu().numpy())
            compare_step(got, (ref_model[i], *ref_state[i]))
        if t == 3:
            saved = ({k: v.clone() for k, v in model.state_dict().items()},
                     {"state": {k: {kk: (vv.clone() if torch.is_tensor(vv) else vv) for kk, vv in s.items()}
                                for k, s in opt.state_dict()["state"].items()},
                      "param_groups": opt.state_dict()["param_groups"]})
    final = [p.detach().clone() for p in model.parameters()]
    # resume from step 3
    model.load_state_dict(saved[0])
    opt2 = bwd.Adam8bit(model.parameters(), lr=1e-3)
    opt2.load_state_dict(saved[1])
    for p in model.parameters():
        assert opt2.state[p]["m_codes"].dtype == torch.uint8
    for t in range(4, 7):
        opt2.zero_grad()
        torch.nn.functional.cross_entropy(model(x), y).backward()
        opt2.step()
    for a, b in zip(final, model.parameters()):
        assert torch.equal(a, b.detach())


def _sampled_full_size(bwd, wl, blocks_per_tensor=2, max_tensors=80, steps=2, seed=0, pdt=torch.float32):
    """Run the whole workload through one multi-tensor call per step (the
    launch configuration the bench times) and check sampled blocks of the
    last step against the oracle, from the GPU's own input state.  With
    16-bit parameters (pdt) the oracle widens and rounds them back as the
    kernel does; their values may differ by one unit (compare_bf16_params),
    the codes and absmax not at all."""
    rng = np.random.default_rng(seed)
    T = len(wl.sizes)
    p16 = pdt != torch.float32
    ps, gs, sts = [], [], []
    for i, n in enumerate(wl.sizes):
        ps.append(W.gen_normal(n, 0.02, seed=i, device=DEV).to(pdt))
        gs.append(W.gen_normal(n, wl.grad_std[i], seed=100_000 + i, device=DEV, dtype=wl.grad_dtype))
        sts.append(bwd.state_init(n, DEV))
    args = bwd.MultiTensorArgs(ps, gs, *[[s[k] for s in sts] for k in range(4)])
    for t in range(1, steps):
        args.step(lr=wl.lr, step=t)
    pick = sorted(set([0, T - 1]) | set(rng.choice(T, min(T, max_tensors), replace=False).tolist()))
    samples = []
    for i in pick:
        n = wl.sizes[i]
        nb = (n + B - 1) // B
        for b in sorted(set([0, nb - 1]) | set(rng.choice(nb, min(nb, blocks_per_tensor), replace=False).tolist())):
            lo, hi = b * B, min(n, (b + 1) * B)
            pin = (ps[i][lo:hi].cpu().view(torch.int16).numpy().view(np.uint16) if p16
                   else ps[i][lo:hi].cpu().numpy())
            inp = (pin, g_to_np(gs[i][lo:hi]), sts[i][0][lo:hi].cpu().numpy(),
                   sts[i][1][b:b + 1].cpu().numpy(), sts[i][2][lo:hi].cpu().numpy(),
                   sts[i][3][b:b + 1].cpu().numpy())
            samples.append((i, b, lo, hi, inp))
    args.step(lr=wl.lr, step=steps)
    torch.cuda.synchronize()
    hp = oracle.AdamHParams(lr=wl.lr, step=steps)
    for i, b, lo, hi, inp in samples:
        if p16:
            ref = oracle.adam8bit_step(*inp, hp, p_bf16=pdt == torch.bfloat16, p_f16=pdt == torch.float16)
            compare_bf16_params(ps[i][lo:hi].cpu().view(torch.int16).numpy().view(np.uint16), ref[0],
                                f16=pdt == torch.float16)
            got = (sts[i][0][lo:hi], sts[i][1][b:b + 1], sts[i][2][lo:hi], sts[i][3][b:b + 1])
            for a, r in zip((x.cpu().numpy() for x in got), ref[1:]):
                assert np.array_equal(a.view(np.uint8), r.view(np.uint8))
            continue
        ref = oracle.adam8bit_step(*inp, hp)
        got = (ps[i][lo:hi].cpu().numpy(), sts[i][0][lo:hi].cpu().numpy(), sts[i][1][b:b + 1].cpu().numpy(),
               sts[i][2][lo:hi].cpu().numpy(), sts[i][3][b:b + 1].cpu().numpy())
        compare_step(got, ref)
    del ps, gs, sts, args
    torch.cuda.empty_cache()
    return len(samples)


def test_full_size_llama2_7b_sampled(bwd):
    assert _sampled_full_size(bwd, W.workload("llama2_7b")) > 100


def test_full_size_ragged_2000_sampled(bwd):
    assert _sampled_full_size(bwd, W.workload("ragged_2000")) > 100


def test_full_size_gpt_350m_flat_sampled(bwd):
    assert _sampled_full_size(bwd, W.workload("gpt_350m"), blocks_per_tensor=200) > 100


def test_full_size_llama2_7b_bf16_params_sampled(bwd):
    assert _sampled_full_size(bwd, W.workload("llama2_7b"), pdt=torch.bfloat16) > 100


def test_full_size_gpt_350m_f16_params_sampled(bwd):
    assert _sampled_full_size(bwd, W.workload("gpt_350m"), blocks_per_tensor=200, pdt=torch.float16) > 100


@pytest.mark.parametrize("gdt", [torch.float32, torch.bfloat16, torch.float16])
def test_adamw_single_step_from_identical_state(bwd, gdt):
    """Decoupled weight decay: p is scaled by 1 - lr*wd before the update."""
    n = 3 * B + 333
    p = W.gen_normal(n, 0.02, seed=77).numpy()
    g = W.gen_normal(n, 1e-2, seed=78, dtype=gdt)
    st = random_state(n, 79)
    for wd in (0.01, 0.2):
        hp = oracle.AdamHParams(lr=3e-3, weight_decay=wd, step=5)
        tp, tmc, tma, tvc, tva = to_dev(p, *st)
        bwd.adam8bit_step(tp, g.to(DEV), tmc, tma, tvc, tva, lr=hp.lr, weight_decay=wd, step=hp.step)
        torch.cuda.synchronize()
        got = tuple(t.cpu().numpy() for t in (tp, tmc, tma, tvc, tva))
        compare_step(got, oracle.adam8bit_step(p, g_to_np(g), *st, hp))


def test_adamw8bit_optimizer_matches_oracle(bwd):
    torch.manual_seed(1)
    ps = [torch.nn.Parameter(torch.randn(n, device=DEV) * 0.02) for n in (5000, 2048 * 3, 17)]
    ref = [(p.detach().cpu().numpy().copy(), *oracle.state_init(p.numel())) for p in ps]
    opt = bwd.AdamW8bit(ps, lr=2e-3, weight_decay=0.1)
    with pytest.raises(ValueError):
        bwd.Adam8bit(ps, weight_decay=0.1)
    for t in range(1, 5):
        grads = [torch.randn(p.numel(), device=DEV) * 1e-2 for p in ps]
        for p, g in zip(ps, grads):
            p.grad = g
        opt.step()
        hp = oracle.AdamHParams(lr=2e-3, weight_decay=0.1, step=t)
        ref = [oracle.adam8bit_step(r[0], g.cpu().numpy(), *r[1:], hp) for r, g in zip(ref, grads)]
    for p, r in zip(ps, ref):
        st = opt.state[p]
        got = (p.detach().cpu().numpy(), st["m_codes"].cpu().numpy(), st["m_absmax"].cpu().numpy(),
               st["v_codes"].cpu().numpy(), st["v_absmax"].cpu().numpy())
        compare_step(got, r)


def test_optimizer_skipped_gradients_and_failed_step(bwd):
    """The drop-in optimizer with fresh gradient tensors every step: a
    parameter without a gradient is skipped (its step count stays), the
    launch plan is rebuilt when that pattern changes, and a step whose launch
    is refused leaves every step count where it was."""
    torch.manual_seed(2)
    sizes = (5000, 2048 * 2, 17)
    ps = [torch.nn.Parameter(torch.randn(n, device=DEV) * 0.02) for n in sizes]
    ref = [[p.detach().cpu().numpy().copy(), *oracle.state_init(p.numel())] for p in ps]
    steps = [0, 0, 0]
    opt = bwd.Adam8bit(ps, lr=1e-3)
    pattern = [(0, 1, 2), (0, 2), (0, 2), (0, 1, 2), (0, 1, 2)]
    for k, live in enumerate(pattern):
        for i, p in enumerate(ps):
            p.grad = torch.randn(p.numel(), device=DEV) * 1e-2 if i in live else None
        if k == 3:  # a refused launch (non-finite lr): nothing moves
            opt.param_groups[0]["lr"] = float("nan")
            before = [p.detach().clone() for p in ps]
            with pytest.raises(bwd.BwdError):
                opt.step()
            assert [opt.state[p]["step"] for p in ps] == steps
            assert all(torch.equal(a, b.detach()) for a, b in zip(before, ps))
            opt.param_groups[0]["lr"] = 1e-3
        opt.step()
        for i in live:
            steps[i] += 1
            hp = oracle.AdamHParams(lr=1e-3, step=steps[i])
            ref[i] = list(oracle.adam8bit_step(ref[i][0], ps[i].grad.cpu().numpy(), *ref[i][1:], hp))
        assert [opt.state[p]["step"] for p in ps] == steps
    for p, r in zip(ps, ref):
        st = opt.state[p]
        got = (p.detach().cpu().numpy(), st["m_codes"].cpu().numpy(), st["m_absmax"].cpu().numpy(),
               st["v_codes"].cpu().numpy(), st["v_absmax"].cpu().numpy())
        compare_step(got, tuple(r))


def test_optimizer_parameter_groups_with_their_own_hyperparameters(bwd):
    """AdamW8bit over two parameter groups with different lr and weight
    decay (the second one bf16): each group's launches use its own
    hyperparameters, checked against the oracle per tensor."""
    torch.manual_seed(4)
    g1 = [torch.nn.Parameter(torch.randn(n, device=DEV) * 0.02) for n in (3000, 2048)]
    g2 = [torch.nn.Parameter((torch.randn(n, device=DEV) * 0.02).to(torch.bfloat16)) for n in (5000,)]
    opt = bwd.AdamW8bit([{"params": g1, "lr": 2e-3, "weight_decay": 0.1},
                         {"params": g2, "lr": 5e-4, "weight_decay": 0.0}])

    def bits16(t):
        return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)

    ref = {id(p): ((p.detach().cpu().numpy().copy() if p.dtype == torch.float32 else bits16(p)),
                   *oracle.state_init(p.numel())) for p in g1 + g2}
    for t in range(1, 4):
        for p in g1 + g2:
            p.grad = (torch.randn(p.numel(), device=DEV) * 1e-2).to(p.dtype)
        opt.step()
        for p, lr, wd in [(q, 2e-3, 0.1) for q in g1] + [(q, 5e-4, 0.0) for q in g2]:
            hp = oracle.AdamHParams(lr=lr, weight_decay=wd, step=t)
            ref[id(p)] = oracle.adam8bit_step(*ref[id(p)][:1], g_to_np(p.grad), *ref[id(p)][1:], hp,
                                              p_bf16=p.dtype == torch.bfloat16)
    for p in g1 + g2:
        st = opt.state[p]
        r = ref[id(p)]
        codes = (st["m_codes"].cpu().numpy(), st["m_absmax"].cpu().numpy(), st["v_codes"].cpu().numpy(),
                 st["v_absmax"].cpu().numpy())
        if p.dtype == torch.float32:
            compare_step((p.detach().cpu().numpy(), *codes), r)
        else:  # bf16 parameters: rounded fp32 updates; the states are exact
            compare_bf16_params(bits16(p), r[0])
            for c, rc in zip(codes, r[1:]):
                assert np.array_equal(c.view(np.uint8), rc.view(np.uint8))
        assert st["step"] == 3


def test_step_on_tensor_larger_than_2p31_elements(bwd):
    """64-bit indexing in the fused step: one tensor of 2^31 + 5 parameters;
    blocks at the 2^31 boundary and the ragged tail against the oracle."""
    n = (1 << 31) + 5
    p = torch.empty(n, dtype=torch.float32, device=DEV)
    p.normal_(0.0, 0.02, generator=torch.Generator(device=DEV).manual_seed(1))
    g = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    g.normal_(0.0, 1e-3, generator=torch.Generator(device=DEV).manual_seed(2))
    mc, ma, vc, va = bwd.state_init(n, DEV)
    bwd.adam8bit_step(p, g, mc, ma, vc, va, lr=1e-3, step=1)
    picks = [0, (1 << 31) // B - 1, (1 << 31) // B]
    saved = {}
    for b in picks:
        lo, hi = b * B, min(n, (b + 1) * B)
        saved[b] = (p[lo:hi].cpu().numpy(), g_to_np(g[lo:hi]), mc[lo:hi].cpu().numpy(), ma[b:b + 1].cpu().numpy(),
                    vc[lo:hi].cpu().numpy(), va[b:b + 1].cpu().numpy())
    bwd.adam8bit_step(p, g, mc, ma, vc, va, lr=1e-3, step=2)
    torch.cuda.synchronize()
    hp = oracle.AdamHParams(lr=1e-3, step=2)
    for b in picks:
        lo, hi = b * B, min(n, (b + 1) * B)
        ref = oracle.adam8bit_step(*saved[b], hp)
        got = (p[lo:hi].cpu().numpy(), mc[lo:hi].cpu().numpy(), ma[b:b + 1].cpu().numpy(),
               vc[lo:hi].cpu().numpy(), va[b:b + 1].cpu().numpy())
        compare_step(got, ref)
    del p, g, mc, ma, vc, va
    torch.cuda.empty_cache()


def compare_bf16_params(p_bits, ref_bits, f16=False):
    """bf16 (fp16 with f16) parameters: at most 1e-3 of them differ (the
    fp32 update is within a few ulps, so it can land on the other side of a
    rounding boundary), and those by one unit, unless their values agree
    within the bound compare_step puts on fp32 parameters, 3e-8 + 4e-7 |p|
    (inside the required atol 1e-7, rtol 1e-5): a result that cancels to
    near zero (p + update ~ 0) turns that absolute error into several units
    of its own small magnitude."""
    a = p_bits.astype(np.int32)
    b = ref_bits.astype(np.int32)
    d = np.abs(a - b)
    assert np.count_nonzero(d) <= max(1e-3 * d.size, 2)
    far = d > 1
    if far.any():
        def val(bits):
            bits = np.asarray(bits, dtype=np.uint16)
            if f16:
                return bits.view(np.float16).astype(np.float64)
            return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        xa, xb = val(p_bits[far]), val(ref_bits[far])
        assert np.all(np.abs(xa - xb) <= 3e-8 + 4e-7 * np.abs(xb)), (xa, xb)


@pytest.mark.parametrize("gdt", [torch.float32, torch.bfloat16, torch.float16])
def test_bf16_params_step_from_identical_state(bwd, gdt):
    from oracle.adam import round_to_bf16

    rng = np.random.default_rng(31)
    sizes = [3 * B + 7, 2048, 5000]
    ps = [torch.from_numpy(round_to_bf16((rng.standard_normal(n) * 0.02).astype(np.float32)).view(np.int16))
          .view(torch.bfloat16) for n in sizes]
    gs = [W.gen_normal(n, 1e-2, 40 + i, dtype=gdt) for i, n in enumerate(sizes)]
    sts = [random_state(n, 50 + i) for i, n in enumerate(sizes)]
    dp = [p.to(DEV) for p in ps]
    dst = [to_dev(*st) for st in sts]
    hp = oracle.AdamHParams(lr=1e-3, weight_decay=0.01, step=4)
    bwd.adam8bit_step_multi(dp, [g.to(DEV) for g in gs], *[[s[k] for s in dst] for k in range(4)],
                            lr=hp.lr, weight_decay=hp.weight_decay, step=hp.step)
    torch.cuda.synchronize()
    for i in range(len(sizes)):
        pb = ps[i].view(torch.int16).numpy().view(np.uint16)
        ref = oracle.adam8bit_step(pb, g_to_np(gs[i]), *sts[i], hp, p_bf16=True)
        got_p = dp[i].cpu().view(torch.int16).numpy().view(np.uint16)
        compare_bf16_params(got_p, ref[0])
        for a, b in zip((x.cpu().numpy() for x in dst[i]), ref[1:]):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_bf16_param_optimizer_and_single_tensor_call(bwd):
    from oracle.adam import widen_bf16

    torch.manual_seed(5)
    p = torch.nn.Parameter((torch.randn(6000, device=DEV) * 0.02).to(torch.bfloat16))
    opt = bwd.Adam8bit([p], lr=1e-3)
    ref = (p.detach().cpu().view(torch.int16).numpy().view(np.uint16).copy(), *oracle.state_init(6000))
    for t in range(1, 4):
        g = torch.randn(6000, device=DEV, dtype=torch.bfloat16) * 1e-2
        p.grad = g
        opt.step()
        ref = oracle.adam8bit_step(ref[0], widen_bf16(g.cpu().view(torch.int16).numpy().view(np.uint16)), *ref[1:],
                                   oracle.AdamHParams(lr=1e-3, step=t), p_bf16=True)
    st = opt.state[p]
    compare_bf16_params(p.detach().cpu().view(torch.int16).numpy().view(np.uint16), ref[0])
    assert np.array_equal(st["m_codes"].cpu().numpy(), ref[1]) and np.array_equal(st["v_codes"].cpu().numpy(), ref[3])
    # the single-tensor call routes bf16 parameters through the typed entry point
    q = p.detach().clone().view(-1)
    mc, ma, vc, va = bwd.state_init(q.numel(), DEV)
    bwd.adam8bit_step(q, p.grad.view(-1), mc, ma, vc, va, lr=1e-3, step=1)
    assert q.dtype == torch.bfloat16


@pytest.mark.parametrize("gdt", [torch.float32, torch.bfloat16, torch.float16])
def test_f16_params_step_from_identical_state(bwd, gdt):
    """IEEE binary16 parameters (the page's FP16 state): widened for the
    update, rounded back to nearest even; codes and absmax exact."""
    from oracle.adam import round_to_f16

    rng = np.random.default_rng(33)
    sizes = [3 * B + 7, 2048, 5000]
    ps = [torch.from_numpy(round_to_f16((rng.standard_normal(n) * 0.02).astype(np.float32)).view(np.int16))
          .view(torch.float16) for n in sizes]
    gs = [W.gen_normal(n, 1e-2, 60 + i, dtype=gdt) for i, n in enumerate(sizes)]
    sts = [random_state(n, 70 + i) for i, n in enumerate(sizes)]
    dp = [p.to(DEV) for p in ps]
    dst = [to_dev(*st) for st in sts]
    hp = oracle.AdamHParams(lr=1e-3, weight_decay=0.01, step=4)
    bwd.adam8bit_step_multi(dp, [g.to(DEV) for g in gs], *[[s[k] for s in dst] for k in range(4)],
                            lr=hp.lr, weight_decay=hp.weight_decay, step=hp.step)
    torch.cuda.synchronize()
    for i in range(len(sizes)):
        pb = ps[i].view(torch.int16).numpy().view(np.uint16)
        ref = oracle.adam8bit_step(pb, g_to_np(gs[i]), *sts[i], hp, p_f16=True)
        compare_bf16_params(dp[i].cpu().view(torch.int16).numpy().view(np.uint16), ref[0], f16=True)
        for a, b in zip((x.cpu().numpy() for x in dst[i]), ref[1:]):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_f16_param_optimizer(bwd):
    from oracle.adam import widen_f16

    torch.manual_seed(6)
    p = torch.nn.Parameter((torch.randn(7000, device=DEV) * 0.02).to(torch.float16))
    opt = bwd.Adam8bit([p], lr=1e-3)
    ref = (p.detach().cpu().view(torch.int16).numpy().view(np.uint16).copy(), *oracle.state_init(7000))
    for t in range(1, 4):
        g = (torch.randn(7000, device=DEV) * 1e-2).to(torch.float16)
        p.grad = g
        opt.step()
        ref = oracle.adam8bit_step(ref[0], widen_f16(g.cpu().view(torch.int16).numpy().view(np.uint16)), *ref[1:],
                                   oracle.AdamHParams(lr=1e-3, step=t), p_f16=True)
    st = opt.state[p]
    compare_bf16_params(p.detach().cpu().view(torch.int16).numpy().view(np.uint16), ref[0], f16=True)
    assert np.array_equal(st["m_codes"].cpu().numpy(), ref[1]) and np.array_equal(st["v_codes"].cpu().numpy(), ref[3])


@pytest.mark.parametrize("gdt", [torch.float32, torch.bfloat16, torch.float16])
def test_non_finite_gradients_do_not_fault(bwd, gdt):
    """NaN and infinite gradients (outside the method) in some blocks: the
    step completes and the other blocks are exactly the oracle's."""
    n = 5 * B
    rng = np.random.default_rng(41)
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    g[7] = np.nan
    g[B + 1000] = np.inf
    g[2 * B + 3] = -np.inf
    g[2 * B + 600] = np.nan
    st = random_state(n, 42)
    gt = torch.from_numpy(g).to(gdt)
    dp = torch.from_numpy(p).to(DEV)
    d = to_dev(*st)
    bwd.adam8bit_step(dp, gt.to(DEV), *d, lr=1e-3, step=3)
    torch.cuda.synchronize()
    hp = oracle.AdamHParams(lr=1e-3, step=3)
    lo = 3 * B
    ref = oracle.adam8bit_step(p[lo:], g_to_np(gt)[lo:], st[0][lo:], st[1][3:], st[2][lo:], st[3][3:], hp)
    got = (dp.cpu().numpy()[lo:], d[0].cpu().numpy()[lo:], d[1].cpu().numpy()[3:], d[2].cpu().numpy()[lo:],
           d[3].cpu().numpy()[3:])
    compare_step(got, ref)


def test_tiny_quotients_across_the_divisor_range(bwd):
    """Blocks whose new m or v absmax sits at either side of 2^-38 (where the
    kernel switches between the scaled and unscaled exact divisions) or far
    from it, each holding quotients down to 2^-80, signed zeros and
    subnormals: codes and absmax bit-identical to the oracle over two steps."""
    rng = np.random.default_rng(77)
    m_edge = 2.0 ** -38 * 10.0  # |g| giving m = 0.1 g at 2^-38 on the first step
    v_edge = np.sqrt(2.0 ** -38 * 1000.0)  # |g| giving v = 0.001 g^2 at 2^-38
    tops = [1.2 * m_edge, 0.6 * m_edge, 1.01 * m_edge, 0.99 * m_edge, 1.1 * v_edge, 0.8 * v_edge,
            1e-30, 1e-20, 1e-3, 1.0, 1e10]
    tops += list(2.0 ** rng.uniform(-60, 20, 21))
    blocks = []
    for top in tops:
        blk = rng.standard_normal(B)
        blk *= top / np.abs(blk).max()
        k = rng.integers(0, B, 300)
        blk[k] = rng.choice([-1.0, 1.0], 300) * 2.0 ** rng.uniform(-80, -40, 300) * top
        blk[rng.integers(0, B, 8)] = -0.0
        blk[rng.integers(0, B, 8)] = 0.0
        blocks.append(blk)
    g = np.concatenate(blocks).astype(np.float32)
    n = g.size
    p = np.zeros(n, np.float32)
    dp, dg = to_dev(p, g)
    st = [t for t in to_dev(*oracle.state_init(n))]
    ref = (p.copy(), *oracle.state_init(n))
    for t in (1, 2):
        gt = g if t == 1 else np.roll(g, 977)
        dg.copy_(torch.from_numpy(gt))
        bwd.adam8bit_step(dp, dg, *st, lr=1e-3, step=t)
        ref = oracle.adam8bit_step(ref[0], gt, *ref[1:], oracle.AdamHParams(lr=1e-3, step=t))
        torch.cuda.synchronize()
        if t == 1:  # both sides of the switch, for m and for v
            for a in (ref[2], ref[4]):
                assert {88, 89} <= set(((a.view(U32) >> 23) & 0xFF).tolist())
        for a, b in zip((x.cpu().numpy() for x in st), ref[1:]):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
