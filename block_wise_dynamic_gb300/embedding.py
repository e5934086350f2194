"""Stable embedding layer on the library's kernels.

"8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION" (summary on
wiki.neutronadmin.com/news/16836), section 二 / 稳定的词嵌入层: the embedding
weight is initialised Xavier-uniform and a layer normalisation follows the
lookup, which keeps the layer's output near unit variance.

Each function checks and marshals CUDA tensors and makes one call into
``libbwd.so`` (``bwd_embedding_*`` in ``include/bwd.h``); the lookup, the
normalisation and both passes run in the library's kernels.

  xavier_bound(V, D)           b = fp32(sqrt(6 / (V + D)))
  init_weight(weight, words)   weight = (2 u - 1) b from uint32 random words
  forward(ids, weight, gamma, beta, eps) -> (y, mean, rstd)
  backward(ids, weight, gamma, mean, rstd, dy, dweight, dgamma, dbeta)
  StableEmbedding              torch.nn.Module with autograd through them
"""

from __future__ import annotations

import torch

from . import _abi
from . import _lib, _need, _stream_handle

EPS = 1e-5

__all__ = ["EPS", "xavier_bound", "init_weight", "forward", "backward", "StableEmbedding"]


def xavier_bound(num_embeddings: int, dim: int) -> float:
    """Glorot's uniform bound for a (V, D) embedding weight."""
    b = _lib.bwd_embedding_xavier_bound(int(num_embeddings), int(dim))
    if b < 0:
        raise ValueError("num_embeddings and dim must be >= 1")
    return b


def _ids(ids: torch.Tensor, device: torch.device) -> torch.Tensor:
    _need(ids, "ids", torch.int64, None, device)
    return ids


def init_weight(weight: torch.Tensor, words: torch.Tensor | None = None, generator=None, stream=None) -> torch.Tensor:
    """Xavier-uniform fill of a (V, D) fp32 CUDA weight in place.  ``words``
    are uniform 32-bit random words (int32 or uint32 storage, one per
    element); drawn with torch's generator when not given."""
    if weight.dim() != 2:
        raise ValueError("weight must be (num_embeddings, dim)")
    _need(weight, "weight", torch.float32)
    n = weight.numel()
    if words is None:
        words = torch.randint(-(2 ** 31), 2 ** 31, (n,), dtype=torch.int64, device=weight.device,
                              generator=generator).to(torch.int32)
    if words.dtype not in (torch.int32, torch.uint32):
        raise TypeError("words must be int32 or uint32")
    _need(words, "words", words.dtype, n, weight.device)
    with torch.cuda.device(weight.device):
        st = _lib.bwd_embedding_init(words.data_ptr(), weight.shape[0], weight.shape[1], weight.data_ptr(),
                                     _stream_handle(weight.device, stream))
    _abi.check(st, "bwd_embedding_init")
    return weight


def forward(ids: torch.Tensor, weight: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor, eps: float = EPS,
            need_stats: bool = True, stream=None):
    """y (ids.shape + (D,)), and per-token mean and rstd (None when
    ``need_stats`` is false)."""
    if weight.dim() != 2:
        raise ValueError("weight must be (num_embeddings, dim)")
    v, d = weight.shape
    _need(weight, "weight", torch.float32)
    dev = weight.device
    _ids(ids, dev)
    _need(gamma, "gamma", torch.float32, d, dev)
    _need(beta, "beta", torch.float32, d, dev)
    t = ids.numel()
    y = torch.empty(*ids.shape, d, dtype=torch.float32, device=weight.device)
    mean = torch.empty(t, dtype=torch.float32, device=weight.device) if need_stats else None
    rstd = torch.empty(t, dtype=torch.float32, device=weight.device) if need_stats else None
    with torch.cuda.device(weight.device):
        st = _lib.bwd_embedding_forward(
            ids.data_ptr(), t, weight.data_ptr(), v, d, gamma.data_ptr(), beta.data_ptr(), float(eps), y.data_ptr(),
            mean.data_ptr() if mean is not None else None, rstd.data_ptr() if rstd is not None else None,
            _stream_handle(weight.device, stream))
    _abi.check(st, "bwd_embedding_forward")
    return y, mean, rstd


def backward(ids: torch.Tensor, weight: torch.Tensor, gamma: torch.Tensor, mean: torch.Tensor, rstd: torch.Tensor,
             dy: torch.Tensor, dweight: torch.Tensor, dgamma: torch.Tensor, dbeta: torch.Tensor, stream=None) -> None:
    """Accumulates the gradients into dweight (V, D), dgamma and dbeta (D)."""
    if weight.dim() != 2:
        raise ValueError("weight must be (num_embeddings, dim)")
    v, d = weight.shape
    t = ids.numel()
    _need(weight, "weight", torch.float32)
    dev = weight.device
    _ids(ids, dev)
    _need(gamma, "gamma", torch.float32, d, dev)
    _need(mean, "mean", torch.float32, t, dev)
    _need(rstd, "rstd", torch.float32, t, dev)
    _need(dy, "dy", torch.float32, t * d, dev)
    _need(dweight, "dweight", torch.float32, v * d, dev)
    _need(dgamma, "dgamma", torch.float32, d, dev)
    _need(dbeta, "dbeta", torch.float32, d, dev)
    with torch.cuda.device(weight.device):
        st = _lib.bwd_embedding_backward(
            ids.data_ptr(), t, weight.data_ptr(), v, d, gamma.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
            dy.data_ptr(), dweight.data_ptr(), dgamma.data_ptr(), dbeta.data_ptr(), _stream_handle(weight.device, stream))
    _abi.check(st, "bwd_embedding_backward")


class _StableEmbeddingFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, ids, weight, gamma, beta, eps):
        y, mean, rstd = forward(ids, weight, gamma, beta, eps)
        ctx.save_for_backward(ids, weight, gamma, mean, rstd)
        return y

    @staticmethod
    def backward(ctx, dy):
        ids, weight, gamma, mean, rstd = ctx.saved_tensors
        dweight = torch.zeros_like(weight)
        dgamma = torch.zeros_like(gamma)
        dbeta = torch.zeros_like(gamma)
        backward(ids, weight, gamma, mean, rstd, dy.contiguous(), dweight, dgamma, dbeta)
        return None, dweight, dgamma, dbeta, None


class StableEmbedding(torch.nn.Module):
    """Embedding lookup followed by LayerNorm, Xavier-uniform initialised
    (fp32 weight, CUDA only).  ``weight`` is (num_embeddings, dim); the
    normalisation's scale and shift are ``norm_weight`` (ones) and
    ``norm_bias`` (zeros)."""

    def __init__(self, num_embeddings: int, dim: int, eps: float = EPS, device=None, generator=None):
        super().__init__()
        device = torch.device(device if device is not None else "cuda")
        self.num_embeddings, self.dim, self.eps = int(num_embeddings), int(dim), float(eps)
        self.weight = torch.nn.Parameter(torch.empty(num_embeddings, dim, dtype=torch.float32, device=device))
        self.norm_weight = torch.nn.Parameter(torch.ones(dim, dtype=torch.float32, device=device))
        self.norm_bias = torch.nn.Parameter(torch.zeros(dim, dtype=torch.float32, device=device))
        with torch.no_grad():
            init_weight(self.weight, generator=generator)

    def forward(self, ids: torch.Tensor) -> torch.Tensor:
        return _StableEmbeddingFn.apply(ids.contiguous(), self.weight, self.norm_weight, self.norm_bias, self.eps)
