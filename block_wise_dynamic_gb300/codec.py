"""Codec for Adam moments: fp32 first / second moments <-> the 8-bit
block-wise state of this library.

"8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION", section 二: the first moment
is stored with the signed dynamic-tree map, the always-positive second
moment with the unsigned map, each with one fp32 absmax per 2048-element
block.  These helpers run the library's quantize / dequantize kernels over
whole optimizer states, so a run can switch from ``torch.optim.Adam`` (or
``AdamW``) to the 8-bit optimizer mid-training and back, and states can be
stored compressed (2 bytes per parameter plus 8 bytes per block).
"""

from __future__ import annotations

from typing import Dict, Tuple

import torch

from . import dequantize_blockwise, num_blocks, quantize_blockwise


def compress_moments(m: torch.Tensor, v: torch.Tensor):
    """fp32 moments (CUDA, any shape, same numel) -> (m_codes, m_absmax,
    v_codes, v_absmax), flat."""
    if m.numel() != v.numel():
        raise ValueError("m and v must have the same number of elements")
    mc, ma = quantize_blockwise(m.detach().reshape(-1).float().contiguous(), "signed")
    vc, va = quantize_blockwise(v.detach().reshape(-1).float().contiguous(), "unsigned")
    return mc, ma, vc, va


def decompress_moments(m_codes, m_absmax, v_codes, v_absmax) -> Tuple[torch.Tensor, torch.Tensor]:
    """The 8-bit state back to flat fp32 moments."""
    return (dequantize_blockwise(m_codes, m_absmax, "signed"),
            dequantize_blockwise(v_codes, v_absmax, "unsigned"))


def load_from_fp32_adam(opt8, fp32_opt: torch.optim.Optimizer) -> None:
    """Fill an ``Adam8bit``/``AdamW8bit`` over the same parameters with the
    compressed state of an fp32 ``torch.optim.Adam``/``AdamW``.  Parameters
    without fp32 state are left untouched."""
    for p, st in fp32_opt.state.items():
        if "exp_avg" not in st:
            continue
        if p not in {q for g in opt8.param_groups for q in g["params"]}:
            raise ValueError("the two optimizers must hold the same parameters")
        mc, ma, vc, va = compress_moments(st["exp_avg"], st["exp_avg_sq"])
        step = st.get("step", 0)
        step = int(step.item()) if torch.is_tensor(step) else int(step)
        opt8.state[p] = {"step": step, "m_codes": mc, "m_absmax": ma, "v_codes": vc, "v_absmax": va}
    opt8._reset_plans()


def export_fp32_adam_state(opt8) -> Dict[torch.Tensor, dict]:
    """Per parameter: {"step", "exp_avg", "exp_avg_sq"} decompressed to fp32,
    shaped like the parameter (the keys ``torch.optim.Adam`` uses)."""
    out = {}
    for p, st in opt8.state.items():
        if "m_codes" not in st:
            continue
        m, v = decompress_moments(st["m_codes"], st["m_absmax"], st["v_codes"], st["v_absmax"])
        out[p] = {"step": torch.tensor(float(st["step"])), "exp_avg": m.view_as(p), "exp_avg_sq": v.view_as(p)}
    return out


def compressed_bytes(n: int) -> int:
    """Bytes of the 8-bit state of n parameters (codes + absmax of both moments)."""
    return 2 * n + 8 * num_blocks(n)
