"""Seeded synthetic workloads: tensor shapes and value distributions.

These generators feed both the GPU path and the CPU oracle in the tests and
the bench.  They hold no part of the method's arithmetic: only shapes, seeds
and the distributions of parameters and gradients.

Workloads (the method's own page reports no kernel benchmark, so every input
is synthetic):
  adam_1m        one fp32 tensor of 1,048,576 elements; p ~ N(0, 0.02),
                 g fp32 ~ N(0, 1e-2) drawn fresh each step; 10 steps
  quant_2p28     2^28 fp32 elements ~ N(0, 1), 0.1% of positions (uniform,
                 seed 0) scaled x100; the signed map on x, the unsigned map
                 on x^2
  gpt_350m       GPT-style set: 24 layers, d 1024, ffn 4096, vocab 50,304
                 tied, 1024 learned positions -> 292 tensors, 354,871,296
                 params, run as ONE flattened fp32 buffer; g bf16 ~ N(0, 1e-3)
  llama2_7b      Llama-2-7B shapes: 32 x (q, k, v, o 4096^2; gate, up
                 11008 x 4096; down 4096 x 11008; two RMSNorm 4096) + embed
                 and untied lm_head 32000 x 4096 + final norm -> 291 tensors,
                 6,738,415,616 params; g bf16 ~ N(0, 1e-3)
  ragged_2000    2,000 fp32 tensors, sizes floor(exp(U(ln 1e3, ln 2^24)))
                 (NumPy default_rng(0)), per-tensor sigma exp(U(ln 1e-5,
                 ln 1e-1)); g fp32 ~ N(0, sigma)

Stable embedding layer (lookup + LayerNorm):
  embed_7b       Llama-2-7B's token embedding, V 32,000 x D 4,096, a batch of
                 4 sequences x 4,096 tokens = 16,384 token ids drawn with
                 Zipf frequencies p(rank k) ~ 1 / (k + 1) (natural
                 text's rank-frequency shape), ranks mapped to ids by a
                 seeded permutation; dL/dy ~ N(0, 1)
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Tuple

import numpy as np
import torch

P_STD = 0.02


def llama2_7b_shapes() -> List[Tuple[str, int]]:
    d, ffn, vocab, layers = 4096, 11008, 32000, 32
    out = [("embed_tokens", vocab * d)]
    for i in range(layers):
        for nm in ("q_proj", "k_proj", "v_proj", "o_proj"):
            out.append((f"layers.{i}.{nm}", d * d))
        for nm in ("gate_proj", "up_proj", "down_proj"):
            out.append((f"layers.{i}.{nm}", d * ffn))
        out.append((f"layers.{i}.input_layernorm", d))
        out.append((f"layers.{i}.post_attention_layernorm", d))
    out.append(("norm", d))
    out.append(("lm_head", vocab * d))
    return out


def gpt_350m_shapes() -> List[Tuple[str, int]]:
    d, ffn, vocab, layers, ctx = 1024, 4096, 50304, 24, 1024
    out = [("wte", vocab * d), ("wpe", ctx * d)]
    for i in range(layers):
        out += [
            (f"h.{i}.ln_1.weight", d), (f"h.{i}.ln_1.bias", d),
            (f"h.{i}.attn.c_attn.weight", d * 3 * d), (f"h.{i}.attn.c_attn.bias", 3 * d),
            (f"h.{i}.attn.c_proj.weight", d * d), (f"h.{i}.attn.c_proj.bias", d),
            (f"h.{i}.ln_2.weight", d), (f"h.{i}.ln_2.bias", d),
            (f"h.{i}.mlp.c_fc.weight", d * ffn), (f"h.{i}.mlp.c_fc.bias", ffn),
            (f"h.{i}.mlp.c_proj.weight", ffn * d), (f"h.{i}.mlp.c_proj.bias", d),
        ]
    out += [("ln_f.weight", d), ("ln_f.bias", d)]
    return out


def ragged_2000(count: int = 2000, seed: int = 0) -> Tuple[List[int], List[float]]:
    rng = np.random.default_rng(seed)
    sizes = np.floor(np.exp(rng.uniform(math.log(1e3), math.log(16_777_216), count))).astype(np.int64)
    sigmas = np.exp(rng.uniform(math.log(1e-5), math.log(1e-1), count))
    return [int(s) for s in sizes], [float(s) for s in sigmas]


@dataclass(frozen=True)
class Workload:
    name: str
    sizes: Tuple[int, ...]      # tensor sizes of the multi-tensor list
    grad_dtype: torch.dtype
    grad_std: Tuple[float, ...]  # per tensor
    steps: int
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8

    @property
    def numel(self) -> int:
        return int(sum(self.sizes))


def workload(name: str) -> Workload:
    if name == "adam_1m":
        return Workload(name, (1_048_576,), torch.float32, (1e-2,), 10)
    if name == "gpt_350m":
        n = sum(s for _, s in gpt_350m_shapes())
        return Workload(name, (n,), torch.bfloat16, (1e-3,), 100)
    if name == "llama2_7b":
        sizes = tuple(s for _, s in llama2_7b_shapes())
        return Workload(name, sizes, torch.bfloat16, (1e-3,) * len(sizes), 20)
    if name == "ragged_2000":
        sizes, sig = ragged_2000()
        return Workload(name, tuple(sizes), torch.float32, tuple(sig), 50)
    raise KeyError(name)


def gen_normal(n: int, std: float, seed: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    """N(0, std) of n elements from a seeded torch generator on ``device``.

    Drawn in fp32 and then cast, so a bf16 tensor holds the rounded fp32
    draws."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    x = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x if dtype == torch.float32 else x.to(dtype)


def quant_input(n: int = 1 << 28, seed: int = 0, device="cpu") -> torch.Tensor:
    """N(0, 1) with 0.1% of positions (uniform, seeded) scaled by 100."""
    x = gen_normal(n, 1.0, seed, device)
    rng = np.random.default_rng(seed)
    k = max(1, n // 1000)
    idx = torch.from_numpy(rng.choice(n, size=k, replace=False).astype(np.int64)).to(device)
    x[idx] *= 100.0
    return x


EMBED_7B = (32000, 4096, 4 * 4096)  # V, D, tokens per step


def token_ids(count: int, vocab: int, seed: int, zipf_s: float = 1.0, device="cpu") -> torch.Tensor:
    """int64 token ids with Zipf-like frequencies: rank k has probability
    proportional to 1 / (k + 1)^zipf_s, ranks permuted over the vocabulary."""
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, vocab + 1, dtype=np.float64) ** zipf_s
    p /= p.sum()
    ranks = rng.choice(vocab, size=count, p=p)
    ids = rng.permutation(vocab)[ranks]
    return torch.from_numpy(ids.astype(np.int64)).to(device)


def random_words(count: int, seed: int, device="cpu") -> torch.Tensor:
    """Uniform 32-bit random words (as int32 storage), e.g. for initialisers."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-(2 ** 31), 2 ** 31, (count,), dtype=torch.int64, generator=g).to(torch.int32).to(device)
