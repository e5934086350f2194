"""Stable embedding layer (oracle).  TEST INFRASTRUCTURE ONLY.

Follows "8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION" (wiki.neutronadmin.com
/news/16836), section 二 / 稳定的词嵌入层 (stable embedding layer): the
embedding weight is initialised with Xavier uniform, and a layer
normalisation follows the embedding lookup so that its output has variance
close to 1; the uniform initialisation avoids the extreme values a normal one
can draw.

Readings where the page is silent:
  R13  Xavier (Glorot) uniform for a (V, D) weight, gain 1: U(-b, b) with
       b = sqrt(6 / (V + D)), so that Var(w) = b^2 / 3 = 2 / (V + D).  The
       bound is formed in binary64 and rounded once to binary32.  The random
       numbers are inputs: one 32-bit word r per weight, u = (r >> 8) * 2^-24
       in [0, 1), and w = binary32((2 u - 1) * b) (2 u - 1 is exact, so that
       is one rounding).
  R14  the normalisation is LayerNorm over the embedding dimension D with a
       learnable scale gamma (initially 1) and shift beta (initially 0),
       biased variance and eps = 1e-5:
           mu = mean(x),  var = mean((x - mu)^2),  rstd = 1 / sqrt(var + eps),
           xhat = (x - mu) * rstd,  y = xhat * gamma + beta,
       x the looked-up fp32 row.  The oracle computes in binary64.
  R15  the backward pass is the gradient of that map: with g = dy * gamma,
           dx = rstd * (g - mean(g) - xhat * mean(g * xhat)),
       dW[id] accumulates dx over every token with that id, dgamma = sum over
       tokens of dy * xhat, dbeta = sum over tokens of dy.
  Token ids outside [0, V) are outside the method (the GPU path writes NaN
  rows for them and skips them in the backward pass); the oracle rejects them.

Parity: ``xavier_bound`` and ``init_weight`` are pinned by Glorot's variance
condition and by torch.nn.init.xavier_uniform_'s range;
``forward`` and ``backward`` against torch's layer_norm / embedding with
autograd in binary64, against the invariants of the normalisation (zero mean
and unit variance of xhat; dx orthogonal to the constant vector and to xhat)
and against central finite differences on tiny inputs
(tests/test_oracle_embedding.py).
"""

from __future__ import annotations

import math
from typing import Tuple

import numpy as np

EPS = 1e-5


def xavier_bound(num_embeddings: int, dim: int) -> np.float32:
    """b = sqrt(6 / (V + D)) rounded once to binary32 (R13)."""
    return np.float32(math.sqrt(6.0 / (num_embeddings + dim)))


def init_weight(words: np.ndarray, num_embeddings: int, dim: int) -> np.ndarray:
    """Xavier-uniform (V, D) weight from one uint32 random word per element
    (R13): u = (r >> 8) 2^-24, w = f32((2u - 1) b)."""
    r = np.asarray(words, dtype=np.uint32).reshape(num_embeddings, dim)
    u = (r >> np.uint32(8)).astype(np.float64) * 2.0 ** -24
    two_u_minus_1 = (2.0 * u - 1.0).astype(np.float32)  # exact: multiples of 2^-23 in [-1, 1)
    return two_u_minus_1 * xavier_bound(num_embeddings, dim)  # one binary32 rounding


def _check_ids(ids: np.ndarray, num_embeddings: int) -> np.ndarray:
    ids = np.asarray(ids, dtype=np.int64).reshape(-1)
    if ids.size and (ids.min() < 0 or ids.max() >= num_embeddings):
        raise ValueError("token id outside [0, V)")
    return ids


def forward(ids: np.ndarray, weight: np.ndarray, gamma: np.ndarray, beta: np.ndarray,
            eps: float = EPS) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Lookup followed by LayerNorm (R14).  Returns y (T, D), mu (T,), rstd (T,)
    in binary64."""
    w = np.asarray(weight, dtype=np.float32)
    ids = _check_ids(ids, w.shape[0])
    x = w[ids].astype(np.float64)
    mu = x.mean(axis=1)
    xc = x - mu[:, None]
    var = (xc * xc).mean(axis=1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = xc * rstd[:, None]
    y = xhat * np.asarray(gamma, np.float64)[None, :] + np.asarray(beta, np.float64)[None, :]
    return y, mu, rstd


def backward(ids: np.ndarray, weight: np.ndarray, gamma: np.ndarray, dy: np.ndarray,
             eps: float = EPS) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Gradients of the loss with respect to the weight, gamma and beta given
    dL/dy (R15), binary64.  Normalisation statistics are recomputed from the
    weight."""
    w = np.asarray(weight, dtype=np.float32)
    ids = _check_ids(ids, w.shape[0])
    x = w[ids].astype(np.float64)
    mu = x.mean(axis=1)
    xc = x - mu[:, None]
    rstd = 1.0 / np.sqrt((xc * xc).mean(axis=1) + eps)
    xhat = xc * rstd[:, None]
    dy = np.asarray(dy, dtype=np.float64).reshape(x.shape)
    g = dy * np.asarray(gamma, np.float64)[None, :]
    dx = rstd[:, None] * (g - g.mean(axis=1, keepdims=True) - xhat * (g * xhat).mean(axis=1, keepdims=True))
    dweight = np.zeros(w.shape, dtype=np.float64)
    np.add.at(dweight, ids, dx)
    dgamma = (dy * xhat).sum(axis=0)
    dbeta = dy.sum(axis=0)
    return dweight, dgamma, dbeta


def backward_abs_sums(ids: np.ndarray, weight: np.ndarray, gamma: np.ndarray, dy: np.ndarray,
                      eps: float = EPS) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Sums of the magnitudes of the terms each gradient element adds up
    (dW: |dx| over the tokens of a row; dgamma: |dy xhat|; dbeta: |dy|): the
    scale of the rounding error of any summation order, for tolerances."""
    w = np.asarray(weight, dtype=np.float32)
    ids = _check_ids(ids, w.shape[0])
    x = w[ids].astype(np.float64)
    mu = x.mean(axis=1)
    xc = x - mu[:, None]
    rstd = 1.0 / np.sqrt((xc * xc).mean(axis=1) + eps)
    xhat = xc * rstd[:, None]
    dy = np.asarray(dy, dtype=np.float64).reshape(x.shape)
    g = dy * np.asarray(gamma, np.float64)[None, :]
    dx = rstd[:, None] * (g - g.mean(axis=1, keepdims=True) - xhat * (g * xhat).mean(axis=1, keepdims=True))
    sw = np.zeros(w.shape, dtype=np.float64)
    np.add.at(sw, ids, np.abs(dx) + rstd[:, None] * (np.abs(g) + np.abs(g).mean(axis=1, keepdims=True)
                                                    + np.abs(xhat) * np.abs(g * xhat).mean(axis=1, keepdims=True)))
    return sw, np.abs(dy * xhat).sum(axis=0), np.abs(dy).sum(axis=0)
