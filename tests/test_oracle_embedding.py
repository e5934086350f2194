"""Pins of the stable-embedding oracle (oracle/stable_embedding.py) against
what fixes it independently: Glorot's variance condition and torch's
xavier_uniform_ range for the initialisation, torch's layer_norm / embedding
and their autograd in binary64, the invariants of a normalisation, and finite
differences."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import stable_embedding as se


def rand_weight(v, d, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((v, d)) * scale + rng.standard_normal((v, 1)) * 0.3 * scale).astype(np.float32)


@pytest.mark.parametrize("v,d", [(32000, 4096), (50304, 1024), (10, 3), (1, 1)])
def test_xavier_bound_gives_glorot_variance(v, d):
    b = float(se.xavier_bound(v, d))
    # U(-b, b) has variance b^2 / 3; Glorot's condition is 2 / (fan_in + fan_out)
    assert b * b / 3.0 == pytest.approx(2.0 / (v + d), rel=3 * 2.0 ** -24)


def test_xavier_range_matches_torch_initialiser_on_an_embedding_weight():
    v, d = 3000, 200
    w = torch.empty(v, d, dtype=torch.float64)
    torch.manual_seed(0)
    torch.nn.init.xavier_uniform_(w)
    b = float(se.xavier_bound(v, d))
    m = float(w.abs().max())
    assert m <= b * (1 + 1e-6)
    assert m >= b * 0.999  # 600k draws reach the end of the range


def test_init_weight_endpoints_and_moments():
    v, d = 7, 5
    b = se.xavier_bound(v, d)
    words = np.array([0, 0xFFFFFFFF, 0x80000000, 0x000000FF, 0x40000000] * 7, dtype=np.uint32)
    w = se.init_weight(words, v, d).reshape(-1)
    assert w.dtype == np.float32
    assert w[0] == -b                                          # u = 0
    assert w[1] == np.float32((1.0 - 2.0 ** -23) * float(b))   # largest u
    assert w[2] == 0.0                                         # u = 1/2
    assert w[3] == -b                                          # low 8 bits ignored
    assert w[4] == np.float32(-0.5) * b                        # u = 1/4
    rng = np.random.default_rng(3)
    big = se.init_weight(rng.integers(0, 2 ** 32, 200 * 300, dtype=np.uint64).astype(np.uint32), 200, 300)
    bb = float(se.xavier_bound(200, 300))
    assert abs(big.mean()) < 0.01 * bb
    assert big.var() == pytest.approx(bb * bb / 3, rel=0.02)
    assert np.abs(big).max() <= bb


def test_forward_matches_torch_layer_norm():
    v, d, t = 50, 37, 200
    w = rand_weight(v, d, 1)
    ids = np.random.default_rng(2).integers(0, v, t)
    gamma = np.random.default_rng(4).standard_normal(d).astype(np.float32)
    beta = np.random.default_rng(5).standard_normal(d).astype(np.float32)
    y, mu, rstd = se.forward(ids, w, gamma, beta)
    x = F.embedding(torch.from_numpy(ids), torch.from_numpy(w).double())
    ref = F.layer_norm(x, (d,), torch.from_numpy(gamma).double(), torch.from_numpy(beta).double(), eps=se.EPS)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(mu, x.mean(dim=1).numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(rstd, 1.0 / torch.sqrt(x.var(dim=1, unbiased=False) + se.EPS).numpy(), rtol=1e-12)


def test_forward_normalises_each_row():
    v, d = 20, 64
    w = rand_weight(v, d, 6, scale=3.0)
    ids = np.arange(v)
    y, _, _ = se.forward(ids, w, np.ones(d, np.float32), np.zeros(d, np.float32))
    x = w.astype(np.float64)
    var = x.var(axis=1)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-13)
    # var(xhat) = var / (var + eps) exactly (closed form)
    np.testing.assert_allclose(y.var(axis=1), var / (var + se.EPS), rtol=1e-12)


def test_forward_constant_row_gives_beta():
    d = 9
    w = np.full((3, d), 0.25, dtype=np.float32)
    beta = np.linspace(-1, 1, d).astype(np.float32)
    y, mu, rstd = se.forward([0, 2, 2], w, np.full(d, 7.0, np.float32), beta)
    np.testing.assert_array_equal(y, np.broadcast_to(beta.astype(np.float64), y.shape))
    assert np.all(mu == 0.25) and np.allclose(rstd, 1.0 / math.sqrt(se.EPS))


def test_backward_matches_torch_autograd():
    v, d, t = 40, 33, 300
    w = rand_weight(v, d, 7)
    ids = np.random.default_rng(8).integers(0, v, t)  # repeated ids accumulate
    gamma = np.random.default_rng(9).standard_normal(d).astype(np.float32)
    beta = np.random.default_rng(10).standard_normal(d).astype(np.float32)
    dy = np.random.default_rng(11).standard_normal((t, d))
    dw, dg, db = se.backward(ids, w, gamma, dy)
    W = torch.from_numpy(w).double().requires_grad_()
    G = torch.from_numpy(gamma).double().requires_grad_()
    B = torch.from_numpy(beta).double().requires_grad_()
    y = F.layer_norm(F.embedding(torch.from_numpy(ids), W), (d,), G, B, eps=se.EPS)
    y.backward(torch.from_numpy(dy))
    np.testing.assert_allclose(dw, W.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dg, G.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(db, B.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_backward_invariants():
    # one token per row, so dW rows are the per-token dx
    v, d = 30, 48
    w = rand_weight(v, d, 12)
    gamma = np.random.default_rng(13).standard_normal(d).astype(np.float32)
    dy = np.random.default_rng(14).standard_normal((v, d))
    dx, _, _ = se.backward(np.arange(v), w, gamma, dy)
    x = w.astype(np.float64)
    xhat = (x - x.mean(axis=1, keepdims=True)) / np.sqrt(x.var(axis=1, keepdims=True) + se.EPS)
    scale = np.abs(dx).sum(axis=1)
    # shifting a row does not change y: dx sums to zero
    assert np.all(np.abs(dx.sum(axis=1)) <= 1e-12 * scale)
    # scaling a row changes y only through eps: with g = dy gamma,
    # sum(dx xhat) = rstd * D * eps / (var + eps) * mean(g xhat)
    var = x.var(axis=1)
    g = dy * gamma.astype(np.float64)
    want = d * se.EPS / (var + se.EPS) / np.sqrt(var + se.EPS) * (g * xhat).mean(axis=1)
    np.testing.assert_allclose((dx * xhat).sum(axis=1), want, rtol=1e-6, atol=1e-12 * scale.max())


def test_backward_finite_differences():
    v, d, t = 5, 6, 9
    w = rand_weight(v, d, 15)
    ids = np.array([0, 1, 1, 4, 2, 2, 2, 0, 3])
    gamma = np.random.default_rng(16).standard_normal(d)
    beta = np.random.default_rng(17).standard_normal(d)
    c = np.random.default_rng(18).standard_normal((t, d))

    def loss(wq, gq, bq):
        x = wq[ids]
        xc = x - x.mean(axis=1, keepdims=True)
        xhat = xc / np.sqrt((xc * xc).mean(axis=1, keepdims=True) + se.EPS)
        return float(((xhat * gq + bq) * c).sum())

    dw, dg, db = se.backward(ids, w, gamma.astype(np.float32), c)
    # gradient of the loss with respect to gamma at the float32-rounded gamma
    g32 = gamma.astype(np.float32).astype(np.float64)
    w64 = w.astype(np.float64)
    h = 1e-6
    rng = np.random.default_rng(19)
    for _ in range(5):
        dW_dir, dG_dir, dB_dir = rng.standard_normal(w.shape), rng.standard_normal(d), rng.standard_normal(d)
        fd = (loss(w64 + h * dW_dir, g32 + h * dG_dir, beta + h * dB_dir)
              - loss(w64 - h * dW_dir, g32 - h * dG_dir, beta - h * dB_dir)) / (2 * h)
        an = (dw * dW_dir).sum() + (dg * dG_dir).sum() + (db * dB_dir).sum()
        assert fd == pytest.approx(an, rel=1e-6, abs=1e-7)


def test_rejects_out_of_range_ids():
    w = np.zeros((4, 3), np.float32)
    with pytest.raises(ValueError):
        se.forward([0, 4], w, np.ones(3, np.float32), np.zeros(3, np.float32))
    with pytest.raises(ValueError):
        se.backward([-1], w, np.ones(3, np.float32), np.zeros((1, 3)))
