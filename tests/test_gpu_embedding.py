"""GPU parity of the stable embedding layer (csrc/embedding.cu, through the C
ABI) against the oracle (oracle/stable_embedding.py).

Tolerances, from the kernels' arithmetic (u = 2^-24, binary32):
  * init: one rounding on both sides -> bit-exact.
  * forward: each row sum is at most 32 sequential adds in a thread, 5
    shuffle levels and 2 adds over the group's warps (<= 39 roundings on
    sums of |x|), so mean and the centred sum of squares carry relative
    errors <= 40 u of the sums of magnitudes; y = (x - mean) rstd gamma +
    beta adds 4 roundings.  |y - y_ref| <= 640 u (1 + |xhat|) |gamma| +
    4 u |beta| covers it with a 16x margin.
  * backward: per token dx carries <= ~100 u of the sum of magnitudes of its
    terms (the saved statistics' error included); a dweight element sums k
    tokens' dx with atomic adds (k more roundings), dgamma and dbeta sum
    every token (per-thread sequence, then the CTAs' atomic adds).  The
    tests bound |err| by 2 (128 + k) u times the oracle's sum of the
    magnitudes of the terms (backward_abs_sums), k the number of adds into
    that element.
"""

import numpy as np
import pytest
import torch

from oracle import stable_embedding as se

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module")
def E():
    from block_wise_dynamic_gb300 import build as b

    b.build()
    from block_wise_dynamic_gb300 import embedding

    return embedding


def dev():
    return torch.device("cuda", 0)


def rand_weight(v, d, seed, scale=0.05):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((v, d)) * scale + rng.standard_normal((v, 1)) * 0.2 * scale).astype(np.float32)


def affine(d, seed):
    rng = np.random.default_rng(seed)
    return (1.0 + 0.3 * rng.standard_normal(d)).astype(np.float32), (0.1 * rng.standard_normal(d)).astype(np.float32)


def ids_for(t, v, seed):
    from block_wise_dynamic_gb300 import workloads as W

    return W.token_ids(t, v, seed).numpy()


def check_forward(E, w, gamma, beta, ids, offset=0):
    """Runs the kernel (the weight optionally placed `offset` floats into a
    larger buffer, which breaks 16-byte alignment) and compares with the oracle."""
    v, d = w.shape
    buf = torch.zeros(v * d + offset, dtype=torch.float32, device=dev())
    wd = buf[offset:].view(v, d)
    wd.copy_(torch.from_numpy(w))
    y, mean, rstd = E.forward(torch.from_numpy(ids).to(dev()), wd, torch.from_numpy(gamma).to(dev()),
                              torch.from_numpy(beta).to(dev()))
    torch.cuda.synchronize()
    ry, rmu, rr = se.forward(ids, w, gamma, beta)
    x = w[ids].astype(np.float64)
    xhat = (x - rmu[:, None]) * rr[:, None]
    tol = 640 * U * (1 + np.abs(xhat)) * np.abs(gamma.astype(np.float64)) + 4 * U * np.abs(beta) + 1e-30
    err = np.abs(y.cpu().numpy().astype(np.float64) - ry)
    assert np.all(err <= tol), float((err / tol).max())
    np.testing.assert_allclose(mean.cpu().numpy(), rmu, rtol=0, atol=float(64 * U * np.abs(x).mean(axis=1).max()))
    np.testing.assert_allclose(rstd.cpu().numpy(), rr, rtol=128 * U)
    return y, mean, rstd


def check_backward(E, w, gamma, ids, dy, offset=0, repeat=1):
    v, d = w.shape
    t = ids.size
    buf = torch.zeros(v * d + offset, dtype=torch.float32, device=dev())
    wd = buf[offset:].view(v, d)
    wd.copy_(torch.from_numpy(w))
    ids_d = torch.from_numpy(ids).to(dev())
    g_d = torch.from_numpy(gamma).to(dev())
    _, mean, rstd = E.forward(ids_d, wd, g_d, torch.zeros_like(g_d))
    dyb = torch.zeros(t * d + offset, dtype=torch.float32, device=dev())
    dy_d = dyb[offset:].view(t, d)
    dy_d.copy_(torch.from_numpy(dy.astype(np.float32)))
    dwb = torch.zeros(v * d + offset, dtype=torch.float32, device=dev())
    dw = dwb[offset:].view(v, d)
    dg = torch.zeros(d, dtype=torch.float32, device=dev())
    db = torch.zeros(d, dtype=torch.float32, device=dev())
    for _ in range(repeat):
        E.backward(ids_d, wd, g_d, mean, rstd, dy_d, dw, dg, db)
    torch.cuda.synchronize()
    dy32 = dy.astype(np.float32).astype(np.float64)
    rw, rg, rb = se.backward(ids, w, gamma, dy32)
    sw, sg, sb = se.backward_abs_sums(ids, w, gamma, dy32)
    k = np.bincount(ids, minlength=v)[:, None] * repeat
    tw = 2 * (128 + k) * U * sw * repeat + 1e-30
    err = np.abs(dw.cpu().numpy() - repeat * rw)
    assert np.all(err <= tw), float((err / tw).max())
    for got, ref, s in ((dg, rg, sg), (db, rb, sb)):
        tol = 2 * (128 + t * repeat) * U * s * repeat + 1e-30
        e = np.abs(got.cpu().numpy() - repeat * ref)
        assert np.all(e <= tol), float((e / tol).max())


def test_init_is_bit_exact(E):
    from block_wise_dynamic_gb300 import workloads as W

    for v, d in [(300, 77), (1000, 4096), (1, 1)]:
        words = W.random_words(v * d, seed=v + d).to(dev())
        w = torch.empty(v, d, dtype=torch.float32, device=dev())
        E.init_weight(w, words)
        ref = se.init_weight(words.cpu().numpy().view(np.uint32), v, d)
        assert np.array_equal(w.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("d", [4096, 1024, 256, 100, 4, 4092])  # fast path: D % 4 == 0, D <= 4096
def test_forward_fast_path(E, d):
    v = 700
    gamma, beta = affine(d, d)
    check_forward(E, rand_weight(v, d, d), gamma, beta, ids_for(3001, v, d))


@pytest.mark.parametrize("d", [1, 3, 4095, 4100, 5000, 130])  # element-wise path
def test_forward_other_shapes(E, d):
    v = 300
    gamma, beta = affine(d, d)
    check_forward(E, rand_weight(v, d, d), gamma, beta, ids_for(777, v, d))


def test_forward_unaligned_weight_takes_the_element_path(E):
    d, v = 256, 200
    gamma, beta = affine(d, 1)
    check_forward(E, rand_weight(v, d, 2), gamma, beta, ids_for(500, v, 3), offset=1)


def test_forward_extreme_rows(E):
    # constant rows (variance 0: y = beta), huge and tiny scales
    d, v = 512, 6
    w = rand_weight(v, d, 4)
    w[0] = 0.25
    w[1] *= 1e15  # squares stay finite in binary32
    w[2] *= 1e-30
    w[3] = 0.0
    gamma, beta = affine(d, 5)
    ids = np.array([0, 1, 2, 3, 4, 5, 0, 3], dtype=np.int64)
    y, _, _ = check_forward(E, w, gamma, beta, ids)
    assert np.array_equal(y.cpu().numpy()[0], beta)


def test_forward_invalid_ids_give_nan_rows(E):
    d, v = 128, 50
    w = rand_weight(v, d, 6)
    gamma, beta = affine(d, 7)
    ids = np.array([3, -1, 50, 7, 2 ** 40, 3], dtype=np.int64)
    ids_d = torch.from_numpy(ids).to(dev())
    y, mean, rstd = E.forward(ids_d, torch.from_numpy(w).to(dev()), torch.from_numpy(gamma).to(dev()),
                              torch.from_numpy(beta).to(dev()))
    y = y.cpu().numpy()
    bad = np.array([False, True, True, False, True, False])
    assert np.all(np.isnan(y[bad])) and np.all(np.isnan(mean.cpu().numpy()[bad]))
    ry, _, _ = se.forward(ids[~bad], w, gamma, beta)
    np.testing.assert_allclose(y[~bad], ry, rtol=1e-4, atol=1e-4)


def test_forward_without_statistics(E):
    d, v = 64, 10
    w = torch.from_numpy(rand_weight(v, d, 8)).to(dev())
    g, b = (torch.from_numpy(a).to(dev()) for a in affine(d, 9))
    ids = torch.arange(v, device=dev())
    y0, _, _ = E.forward(ids, w, g, b)
    y1, m, r = E.forward(ids, w, g, b, need_stats=False)
    assert m is None and r is None and torch.equal(y0, y1)


def test_forward_is_deterministic(E):
    d, v = 4096, 1000
    w = torch.from_numpy(rand_weight(v, d, 10)).to(dev())
    g, b = (torch.from_numpy(a).to(dev()) for a in affine(d, 11))
    ids = torch.from_numpy(ids_for(4000, v, 12)).to(dev())
    ya = E.forward(ids, w, g, b)[0]
    yb = E.forward(ids, w, g, b)[0]
    assert torch.equal(ya, yb)


@pytest.mark.parametrize("d", [4096, 1024, 100, 4, 4095, 3, 5000])
def test_backward(E, d):
    v = 400
    w = rand_weight(v, d, 20 + d)
    gamma, _ = affine(d, 21 + d)
    ids = ids_for(1500, v, 22 + d)
    dy = np.random.default_rng(23 + d).standard_normal((ids.size, d))
    check_backward(E, w, gamma, ids, dy)


def test_backward_unaligned_and_accumulating(E):
    d, v = 256, 300
    w = rand_weight(v, d, 30)
    gamma, _ = affine(d, 31)
    ids = ids_for(900, v, 32)
    dy = np.random.default_rng(33).standard_normal((ids.size, d))
    check_backward(E, w, gamma, ids, dy, offset=1)
    check_backward(E, w, gamma, ids, dy, repeat=2)


def test_backward_skips_invalid_ids(E):
    d, v = 128, 40
    w = rand_weight(v, d, 40)
    gamma, _ = affine(d, 41)
    ids = np.array([1, -3, 5, 40, 5, 2 ** 35], dtype=np.int64)
    ok = (ids >= 0) & (ids < v)
    dy = np.random.default_rng(42).standard_normal((ids.size, d)).astype(np.float32)
    ids_d = torch.from_numpy(ids).to(dev())
    wd = torch.from_numpy(w).to(dev())
    gd = torch.from_numpy(gamma).to(dev())
    _, mean, rstd = E.forward(ids_d, wd, gd, torch.zeros_like(gd))
    dw = torch.zeros_like(wd)
    dg = torch.zeros_like(gd)
    db = torch.zeros_like(gd)
    E.backward(ids_d, wd, gd, mean, rstd, torch.from_numpy(dy).to(dev()), dw, dg, db)
    rw, rg, rb = se.backward(ids[ok], w, gamma, dy[ok].astype(np.float64))
    np.testing.assert_allclose(dw.cpu().numpy(), rw, rtol=1e-4, atol=1e-5)
    np.testing.assert_allclose(db.cpu().numpy(), rb, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(dg.cpu().numpy(), rg, rtol=1e-4, atol=1e-5)


def test_module_autograd_and_8bit_adam_step(E):
    from block_wise_dynamic_gb300 import Adam8bit

    torch.manual_seed(0)
    v, d = 256, 128
    layer = E.StableEmbedding(v, d, device=dev())
    b = float(E.xavier_bound(v, d))
    assert float(layer.weight.detach().abs().max()) <= b
    ids = torch.from_numpy(ids_for(600, v, 50)).to(dev()).view(20, 30)
    c = torch.randn(20, 30, d, device=dev())
    loss = (layer(ids) * c).sum()
    loss.backward()
    w = layer.weight.detach().cpu().numpy()
    gamma = layer.norm_weight.detach().cpu().numpy()
    rw, rg, rb = se.backward(ids.cpu().numpy().reshape(-1), w, gamma, c.cpu().numpy().reshape(-1, d).astype(np.float64))
    np.testing.assert_allclose(layer.weight.grad.cpu().numpy(), rw, rtol=1e-4, atol=1e-5)
    np.testing.assert_allclose(layer.norm_weight.grad.cpu().numpy(), rg, rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(layer.norm_bias.grad.cpu().numpy(), rb, rtol=1e-4, atol=1e-4)
    opt = Adam8bit(layer.parameters(), lr=1e-3)
    before = layer.weight.detach().clone()
    opt.step()
    moved = (layer.weight.detach() - before).abs()
    touched = torch.zeros(v, dtype=torch.bool, device=dev())
    touched[ids.reshape(-1)] = True
    assert bool((moved[touched].amax(dim=1) > 0).all())       # rows with gradient moved
    assert float(moved[~touched].max()) == 0.0                  # the others did not


def test_full_size_embed_7b_sampled(E):
    """Llama-2-7B's embedding (32,000 x 4,096) with 16,384 Zipf-distributed
    tokens, in the launch configuration the bench times: y on sampled tokens,
    dweight on sampled rows (every token of those rows), dgamma and dbeta
    in full."""
    from block_wise_dynamic_gb300 import workloads as W

    v, d, t = W.EMBED_7B
    words = W.random_words(v * d, seed=1).to(dev())
    w = torch.empty(v, d, dtype=torch.float32, device=dev())
    E.init_weight(w, words)
    del words
    gamma, beta = affine(d, 60)
    ids = W.token_ids(t, v, seed=0)
    g_d, b_d = torch.from_numpy(gamma).to(dev()), torch.from_numpy(beta).to(dev())
    y, mean, rstd = E.forward(ids.to(dev()), w, g_d, b_d)
    dy = W.gen_normal(t * d, 1.0, seed=61, device=dev()).view(t, d)
    dw = torch.zeros_like(w)
    dg = torch.zeros_like(g_d)
    db = torch.zeros_like(g_d)
    E.backward(ids.to(dev()), w, g_d, mean, rstd, dy, dw, dg, db)
    torch.cuda.synchronize()
    wn = w.cpu().numpy()
    idn = ids.numpy()
    rng = np.random.default_rng(62)
    sample = rng.choice(t, 256, replace=False)
    ry, _, _ = se.forward(idn[sample], wn, gamma, beta)
    x = wn[idn[sample]].astype(np.float64)
    xhat = (x - x.mean(axis=1, keepdims=True)) / np.sqrt(x.var(axis=1, keepdims=True) + se.EPS)
    tol = 640 * U * (1 + np.abs(xhat)) * np.abs(gamma) + 4 * U * np.abs(beta)
    assert np.all(np.abs(y.cpu().numpy()[sample] - ry) <= tol)
    dyn = dy.cpu().numpy().astype(np.float64)
    counts = np.bincount(idn, minlength=v)
    rows = np.concatenate([np.argsort(-counts)[:3], rng.choice(np.flatnonzero(counts), 20, replace=False)])
    dwn = dw.cpu().numpy()
    for r in rows:
        sel = idn == r
        rw, _, _ = se.backward(np.zeros(int(sel.sum()), np.int64), wn[r:r + 1], gamma, dyn[sel])
        sw, _, _ = se.backward_abs_sums(np.zeros(int(sel.sum()), np.int64), wn[r:r + 1], gamma, dyn[sel])
        tolr = 2 * (128 + counts[r]) * U * sw[0] + 1e-30
        assert np.all(np.abs(dwn[r] - rw[0]) <= tolr), (int(r), int(counts[r]))
    untouched = np.flatnonzero(counts == 0)[:50]
    assert np.all(dwn[untouched] == 0.0)
    _, rg, rb = se.backward(idn, wn, gamma, dyn)
    _, sg, sb = se.backward_abs_sums(idn, wn, gamma, dyn)
    for got, ref, s in ((dg, rg, sg), (db, rb, sb)):
        tol = 2 * (128 + t) * U * s
        assert np.all(np.abs(got.cpu().numpy() - ref) <= tol)


def test_device_check_after_backward(E):
    """The backward's bounded waits complete in normal operation: the device
    fault flag stays clear."""
    import block_wise_dynamic_gb300 as bwd

    d, v = 4096, 500
    w = torch.from_numpy(rand_weight(v, d, 70)).to(dev())
    g, b = (torch.from_numpy(a).to(dev()) for a in affine(d, 71))
    ids = torch.from_numpy(ids_for(5000, v, 72)).to(dev())
    _, mean, rstd = E.forward(ids, w, g, b)
    dy = torch.randn(5000, d, device=dev())
    for _ in range(3):
        E.backward(ids, w, g, mean, rstd, dy, torch.zeros_like(w), torch.zeros_like(g), torch.zeros_like(g))
    bwd.check_device(0)


@pytest.mark.parametrize("case", ["many_chunks", "one_id", "all_distinct", "one_token", "two_tokens"])
def test_backward_runs_of_equal_ids(E, case):
    """The fast path sums the dL/dy rows of each run of equal ids within a
    chunk of tokens (at most 1,024 per chunk, chunks spread over the SMs):
    more tokens than one pass of chunks holds, every token on one id (one
    long run per chunk), every id distinct (runs of one), and one or two
    tokens."""
    rng = np.random.default_rng(80)
    if case == "many_chunks":
        v, d, ids = 3000, 64, ids_for(200_000, 3000, 81)
    elif case == "one_id":
        v, d, ids = 50, 512, np.full(20_000, 17, dtype=np.int64)
    elif case == "all_distinct":
        v, d = 6000, 1024
        ids = rng.permutation(v)[:5000].astype(np.int64)
    elif case == "one_token":
        v, d, ids = 10, 4096, np.array([7], dtype=np.int64)
    else:
        v, d, ids = 10, 4096, np.array([7, 7], dtype=np.int64)
    w = rand_weight(v, d, 82)
    gamma, _ = affine(d, 83)
    dy = rng.standard_normal((ids.size, d))
    check_backward(E, w, gamma, ids, dy)


def test_backward_with_unaligned_dgamma_dbeta(E):
    """The fast path with dgamma and dbeta placed one float into larger
    buffers (4-byte but not 16-byte aligned): the end-of-kernel adds take the
    scalar form."""
    d, v, t = 4096, 300, 2000
    w = rand_weight(v, d, 90)
    gamma, _ = affine(d, 91)
    ids = ids_for(t, v, 92)
    dy = np.random.default_rng(93).standard_normal((t, d)).astype(np.float32)
    wd, gd = torch.from_numpy(w).to(dev()), torch.from_numpy(gamma).to(dev())
    ids_d = torch.from_numpy(ids).to(dev())
    _, mean, rstd = E.forward(ids_d, wd, gd, torch.zeros_like(gd))
    gb = torch.zeros(2 * d + 2, device=dev())
    dg, db = gb[1:1 + d], gb[d + 2:]
    assert dg.data_ptr() % 16 == 4
    E.backward(ids_d, wd, gd, mean, rstd, torch.from_numpy(dy).to(dev()), torch.zeros_like(wd), dg, db)
    torch.cuda.synchronize()
    dy64 = dy.astype(np.float64)
    _, rg, rb = se.backward(ids, w, gamma, dy64)
    _, sg, sb = se.backward_abs_sums(ids, w, gamma, dy64)
    for got, ref, s_ in ((dg, rg, sg), (db, rb, sb)):
        assert np.all(np.abs(got.cpu().numpy() - ref) <= 2 * (128 + t) * U * s_ + 1e-30)


def test_backward_with_many_interleaved_invalid_ids(E):
    """About 30% of 5,000 token ids out of range, spread through the list:
    the staged backward issues no copy and takes no wait for them, so its
    per-buffer phase bookkeeping is exercised across skipped tokens."""
    d, v = 1024, 300
    w = rand_weight(v, d, 80)
    gamma, beta = affine(d, 81)
    rng = np.random.default_rng(82)
    ids = ids_for(5000, v, 83).copy()
    bad = rng.random(ids.size) < 0.3
    ids[bad] = np.where(rng.random(int(bad.sum())) < 0.5, -1 - rng.integers(0, 5, int(bad.sum())), v + rng.integers(0, 9, int(bad.sum())))
    dy = rng.standard_normal((ids.size, d)).astype(np.float32)
    ids_d = torch.from_numpy(ids).to(dev())
    wd = torch.from_numpy(w).to(dev())
    gd, bd = torch.from_numpy(gamma).to(dev()), torch.from_numpy(beta).to(dev())
    y, mean, rstd = E.forward(ids_d, wd, gd, bd)
    assert bool(torch.isnan(y[torch.from_numpy(bad).to(dev())]).all())
    dw, dg, db = torch.zeros_like(wd), torch.zeros_like(gd), torch.zeros_like(gd)
    E.backward(ids_d, wd, gd, mean, rstd, torch.from_numpy(dy).to(dev()), dw, dg, db)
    torch.cuda.synchronize()
    ok = ~bad
    dy64 = dy[ok].astype(np.float64)
    rw, rg, rb = se.backward(ids[ok], w, gamma, dy64)
    sw, sg, sb = se.backward_abs_sums(ids[ok], w, gamma, dy64)
    k = np.bincount(ids[ok], minlength=v)[:, None]
    assert np.all(np.abs(dw.cpu().numpy() - rw) <= 2 * (128 + k) * U * sw + 1e-30)
    t = int(ok.sum())
    for got, ref, s in ((dg, rg, sg), (db, rb, sb)):
        assert np.all(np.abs(got.cpu().numpy() - ref) <= 2 * (128 + t) * U * s + 1e-30)


def test_bounded_wait_gives_up_and_is_reported(E):
    """A wait that nothing completes (the self-test kernel) gives up after
    about a second, the fault word is reported once and cleared, and the
    device keeps working."""
    import time

    import block_wise_dynamic_gb300 as bwd
    from block_wise_dynamic_gb300 import _abi

    bwd.check_device(0)  # clean start
    t0 = time.perf_counter()
    _abi.check(bwd._lib.bwd_selftest_bounded_wait(None), "bwd_selftest_bounded_wait")
    with pytest.raises(_abi.BwdError) as err:
        bwd.check_device(0)
    assert "bounded wait" in str(err.value)
    assert 0.5 < time.perf_counter() - t0 < 30.0
    bwd.check_device(0)  # cleared
    d, v = 256, 50
    w = torch.from_numpy(rand_weight(v, d, 90)).to(dev())
    g, b = (torch.from_numpy(a).to(dev()) for a in affine(d, 91))
    ids = torch.arange(v, device=dev())
    y, mean, rstd = E.forward(ids, w, g, b)
    E.backward(ids, w, g, mean, rstd, torch.ones(v, d, device=dev()), torch.zeros_like(w), torch.zeros_like(g),
               torch.zeros_like(g))
    bwd.check_device(0)
    ry, _, _ = se.forward(np.arange(v), w.cpu().numpy(), g.cpu().numpy(), b.cpu().numpy())
    np.testing.assert_allclose(y.cpu().numpy(), ry, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("shape", [(0,), (3, 0)])
def test_zero_tokens_are_no_ops(E, shape):
    d, v = 256, 40
    w = torch.from_numpy(rand_weight(v, d, 12)).to(dev())
    g, b = (torch.from_numpy(a).to(dev()) for a in affine(d, 13))
    ids = torch.zeros(shape, dtype=torch.int64, device=dev())
    y, mean, rstd = E.forward(ids, w, g, b)
    assert tuple(y.shape) == shape + (d,) and mean.numel() == 0 and rstd.numel() == 0
    dw = torch.full_like(w, 0.5)
    dg = torch.full_like(g, 0.25)
    db = torch.full_like(g, -1.0)
    E.backward(ids.reshape(-1), w, g, mean, rstd, y.reshape(0, d), dw, dg, db)
    torch.cuda.synchronize()
    assert torch.all(dw == 0.5) and torch.all(dg == 0.25) and torch.all(db == -1.0)


def test_weight_larger_than_2p31_elements(E):
    """A 600,000 x 4,096 weight (2.46e9 elements, offsets past 2^31): tokens
    whose rows lie beyond element 2^31, and rows on both sides of it, against
    the oracle on those rows (forward, and backward into the weight's
    gradient)."""
    from block_wise_dynamic_gb300 import workloads as W

    v, d = 600_000, 4096
    w = torch.empty(v, d, dtype=torch.float32, device=dev())
    E.init_weight(w, None, generator=torch.Generator(device=dev()).manual_seed(5))
    edge = (1 << 31) // d  # first row starting at element 2^31
    rows = np.array([0, 1, v // 2 + 17, edge - 1, edge, edge + 1, v - 2, v - 1], dtype=np.int64)  # ascending
    assert np.all(np.diff(rows) > 0)
    rng = np.random.default_rng(63)
    idn = rows[rng.integers(0, rows.size, 600)]
    ids = torch.from_numpy(idn).to(dev())
    gamma, beta = affine(d, 64)
    g_d, b_d = torch.from_numpy(gamma).to(dev()), torch.from_numpy(beta).to(dev())
    y, mean, rstd = E.forward(ids, w, g_d, b_d)
    dy = W.gen_normal(idn.size * d, 1.0, seed=65, device=dev()).view(idn.size, d)
    dw = torch.zeros_like(w)
    dg = torch.zeros_like(g_d)
    db = torch.zeros_like(g_d)
    E.backward(ids, w, g_d, mean, rstd, dy, dw, dg, db)
    torch.cuda.synchronize()
    sub = w[torch.from_numpy(rows).to(dev())].cpu().numpy()
    local = np.searchsorted(rows, idn)  # index of each token's row in `rows`
    assert np.array_equal(rows[local], idn)
    ry, _, _ = se.forward(local, sub, gamma, beta)
    x = sub[local].astype(np.float64)
    xhat = (x - x.mean(axis=1, keepdims=True)) / np.sqrt(x.var(axis=1, keepdims=True) + se.EPS)
    tol = 640 * U * (1 + np.abs(xhat)) * np.abs(gamma) + 4 * U * np.abs(beta)
    assert np.all(np.abs(y.cpu().numpy() - ry) <= tol)
    dyn = dy.cpu().numpy().astype(np.float64)
    rw, _, _ = se.backward(local, sub, gamma, dyn)
    sw, _, _ = se.backward_abs_sums(local, sub, gamma, dyn)
    k = np.bincount(local, minlength=rows.size)[:, None]
    got = dw[torch.from_numpy(rows).to(dev())].cpu().numpy()
    assert np.all(np.abs(got - rw) <= 2 * (128 + k) * U * sw + 1e-30)
    assert float(dw[2].abs().max()) == 0.0 and float(dw[edge + 2].abs().max()) == 0.0
