"""Block-wise quantize / dequantize (oracle).  TEST INFRASTRUCTURE ONLY.

Follows "8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION" (wiki.neutronadmin.com
/news/16836):
  * section 二 / 逐块量化: the tensor is cut into blocks of 2048 elements and
    each block is normalised into [-1, 1] on its own, so an outlier only
    affects its own block;
  * section 一: quantization stands for values by a low-bit type (here: the
    nearest entry of the 256-entry dynamic map); dequantization maps back.

Readings where the page is silent:
  R5  blocks are [2048 b, min(2048 (b + 1), n)) of one flat tensor; the last
      block may be partial and is normalised over the elements it has;
  R6  the normaliser is the block's absolute maximum; an all-zero block keeps
      absmax 0 and every code is the code of +0.0;
  R7  the nearest code is the count of thresholds <= x / absmax (binary32
      IEEE division), i.e. a value exactly on a threshold takes the higher
      code; -0.0 and +0.0 both take the code of +0.0;
  R8  non-finite inputs are outside the method;
  dequantized value = binary32 product map[code] * absmax.

Parity: pinned by tests/test_oracle_blockwise.py (nearest code by brute force
in exact arithmetic, absmax and range invariants, outlier containment, the
round-trip error bound, the exact round trip of each block's absmax element).
"""

from __future__ import annotations

import numpy as np

from .codebook import BLOCK, dynamic_map, thresholds, zero_code


def num_blocks(n: int) -> int:
    return (int(n) + BLOCK - 1) // BLOCK


def quantize_blockwise(x, signed: bool):
    """Quantize a flat binary32 array block by block.

    Returns ``(codes uint8[n], absmax float32[ceil(n / 2048)])``.
    """
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32).ravel())
    n = x.size
    nb = num_blocks(n)
    if n == 0:
        return np.empty(0, np.uint8), np.empty(0, np.float32)
    # padding with zeros leaves every block's max |x| unchanged
    xp = np.zeros(nb * BLOCK, np.float32)
    xp[:n] = x
    xb = xp.reshape(nb, BLOCK)
    absmax = np.max(np.abs(xb), axis=1).astype(np.float32)
    nz = absmax != 0
    xn = np.zeros_like(xb)
    xn[nz] = xb[nz] / absmax[nz, None]           # binary32 IEEE division
    t = thresholds(signed)
    codes = np.searchsorted(t, xn.ravel(), side="right").astype(np.uint8)
    codes = codes.reshape(nb, BLOCK)
    codes[~nz] = zero_code(signed)
    return codes.ravel()[:n].copy(), absmax


def dequantize_blockwise(codes, absmax, signed: bool):
    """Map codes back: y = map[code] * absmax[block] (one binary32 multiply)."""
    codes = np.asarray(codes, dtype=np.uint8).ravel()
    absmax = np.asarray(absmax, dtype=np.float32).ravel()
    n = codes.size
    nb = num_blocks(n)
    if absmax.size != nb:
        raise ValueError("absmax must hold one value per 2048-element block")
    m = dynamic_map(signed)
    scale = np.repeat(absmax, BLOCK)[:n]
    return (m[codes] * scale).astype(np.float32)
