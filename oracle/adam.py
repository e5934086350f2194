"""8-bit Adam step (oracle).  TEST INFRASTRUCTURE ONLY.

Follows "8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION" (wiki.neutronadmin.com
/news/16836):
  * section 一: Adam keeps two states per parameter, the first moment (mean
    of the gradient) and the second moment (uncentred variance);
  * section 二, opening paragraph: the states live in GPU memory in low
    precision; for the parameter update they are dequantized to a high
    precision state, the update runs, and they are stored low precision again;
  * section 二 / 动态量化: the first moment takes the signed map, the second
    moment (always positive) the unsigned map.

Readings where the page is silent:
  R9   "high precision" is binary32 (the parameters are fp32 master weights);
  R10  the update is Adam with bias correction, with the corrections folded
       into two host scalars computed in binary64 and rounded once:
           bc1 = 1 - beta1**t,  bc2 = 1 - beta2**t,
           step_size = f32(lr / bc1),  bc2_sqrt = f32(sqrt(bc2)),
       and per element, every operation one binary32 rounding, in this order:
           m     = beta1 * m_old + (1 - beta1) * g
           v     = beta2 * v_old + ((1 - beta2) * g) * g
           denom = sqrt(v) / bc2_sqrt + eps
           p     = p - (step_size * m) / denom
  R11  the parameter update uses the fresh binary32 m and v; only afterwards
       are they requantized, block by block, each with a fresh absmax;
  t counts from 1; the state before step 1 is all codes of +0.0 with absmax 0
  (R6), which dequantizes to exact zeros.  bf16 gradients widen exactly.

bf16 or fp16 parameters (the page's low-precision weights with a
high-precision update; the page itself names FP16): p is widened to binary32,
updated as above, and rounded back to bf16 / IEEE binary16 (nearest, ties to
even).  fp16 gradients widen exactly, like bf16 ones.

Decoupled weight decay (AdamW; not on the page, the first extension of the
method): with weight_decay wd > 0 the parameters are first scaled,
p = p * f32(1 - lr * wd) (factor formed in binary64), then updated as above
with the same moments.  wd = 0 gives a factor of exactly 1.

Parity: ``adam_update_fp32`` is pinned against ``torch.optim.Adam`` and
``torch.optim.AdamW`` on the CPU (tests/test_oracle_adam.py) and against the
closed forms of Adam's first step and of a pure decay step;
the 8-bit step is pinned by its quantization invariants and by a trajectory
band around 32-bit Adam.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from .blockwise import dequantize_blockwise, num_blocks, quantize_blockwise
from .codebook import zero_code

F32 = np.float32


@dataclass(frozen=True)
class AdamHParams:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    step: int = 1

    def f32(self):
        """The hyper-parameters as the binary32 values a caller passes."""
        return (F32(self.lr), F32(self.beta1), F32(self.beta2), F32(self.eps))


def host_scalars(hp: AdamHParams):
    """R10 host scalars from the binary32 hyper-parameters, in binary64."""
    if hp.step < 1:
        raise ValueError("step counts from 1")
    lr, b1, b2, _ = (float(v) for v in hp.f32())
    wd = float(F32(hp.weight_decay))
    bc1 = 1.0 - b1 ** hp.step
    bc2 = 1.0 - b2 ** hp.step
    return {
        "step_size": F32(lr / bc1),
        "bc2_sqrt": F32(math.sqrt(bc2)),
        "one_minus_beta1": F32(1.0 - b1),
        "one_minus_beta2": F32(1.0 - b2),
        "decay": F32(1.0 - lr * wd),
    }


def widen_bf16(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) to binary32: the 16 bits are the high half."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def round_to_bf16(x) -> np.ndarray:
    """binary32 -> bf16 bit patterns, round to nearest, ties to even: keep
    the high 16 bits, add one unit when the dropped 16 bits exceed half a
    unit, or equal it and the kept part is odd.  NaNs stay NaN (quiet)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    hi = u >> 16
    lo = u & 0xFFFF
    up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & 1) == 1))
    r = (hi + up.astype(np.uint64)).astype(np.uint32)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r[nan] = (hi[nan] | 0x40).astype(np.uint32)
    return r.astype(np.uint16)


def widen_f16(bits) -> np.ndarray:
    """IEEE binary16 bit patterns (uint16) to binary32 (exact)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def round_to_f16(x) -> np.ndarray:
    """binary32 -> IEEE binary16 bit patterns, round to nearest, ties to
    even, with gradual underflow and overflow to infinity (NumPy's
    conversion, used here as a library step)."""
    with np.errstate(over="ignore"):  # overflow to infinity is the rounding rule
        return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def adam_update_fp32(p, g, m_old, v_old, hp: AdamHParams):
    """One binary32 Adam(W) update (R10).  Returns new (p, m, v); inputs unchanged."""
    if hp.weight_decay < 0.0:
        raise ValueError("weight decay must be >= 0")
    p = np.asarray(p, F32)
    g = np.asarray(g, F32)
    m_old = np.asarray(m_old, F32)
    v_old = np.asarray(v_old, F32)
    _, b1, b2, eps = hp.f32()
    s = host_scalars(hp)
    m = b1 * m_old + s["one_minus_beta1"] * g
    v = b2 * v_old + (s["one_minus_beta2"] * g) * g
    denom = np.sqrt(v) / s["bc2_sqrt"] + eps
    p_new = (p * s["decay"]) - (s["step_size"] * m) / denom
    return p_new.astype(F32), m.astype(F32), v.astype(F32)


def adam8bit_step(p, g, m_codes, m_absmax, v_codes, v_absmax, hp: AdamHParams, p_bf16: bool = False,
                  p_f16: bool = False):
    """One 8-bit Adam step on one flat tensor (R9-R11).

    Returns new ``(p, m_codes, m_absmax, v_codes, v_absmax)``.  With
    ``p_bf16`` (``p_f16``) the parameters are bf16 (IEEE binary16) bit
    patterns (uint16): they are widened to binary32 for the update and
    rounded back to nearest, ties to even.
    """
    m_old = dequantize_blockwise(m_codes, m_absmax, signed=True)
    v_old = dequantize_blockwise(v_codes, v_absmax, signed=False)
    if p_bf16 and p_f16:
        raise ValueError("p_bf16 and p_f16 exclude each other")
    if p_bf16:
        p32, m, v = adam_update_fp32(widen_bf16(p), g, m_old, v_old, hp)
        p_new = round_to_bf16(p32)
    elif p_f16:
        p32, m, v = adam_update_fp32(widen_f16(p), g, m_old, v_old, hp)
        p_new = round_to_f16(p32)
    else:
        p_new, m, v = adam_update_fp32(p, g, m_old, v_old, hp)
    mc, ma = quantize_blockwise(m, signed=True)
    vc, va = quantize_blockwise(v, signed=False)
    return p_new, mc, ma, vc, va


def adam8bit_step_multi(tensors, hp: AdamHParams):
    """The step over a list of tensors; blocks never span two tensors (R5).

    ``tensors`` is a list of ``(p, g, m_codes, m_absmax, v_codes, v_absmax)``.
    """
    return [adam8bit_step(*t, hp) for t in tensors]


def state_init(n: int):
    """State before step 1 (R6): codes of +0.0 and absmax 0."""
    nb = num_blocks(n)
    return (
        np.full(n, zero_code(True), np.uint8),
        np.zeros(nb, F32),
        np.full(n, zero_code(False), np.uint8),
        np.zeros(nb, F32),
    )
