"""CPU oracle for 8-bit Adam with block-wise dynamic quantization.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously correct
statement of what the GPU path computes.  Only the test suite, the smoke check
in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it;
the product package never does, and the two share no code, tables or helpers.

Source of the method: the blog summary "8-BIT OPTIMIZERS VIA BLOCK-WISE
QUANTIZATION" (wiki.neutronadmin.com/news/16836), sections
  * 一、优化器遇到量化的故事      -- Adam's two moments, quantize / dequantize,
  * 二、三个方法构建无损FP8优化器 -- states stored low precision, dequantized
    for the update and stored low precision again (opening paragraph);
    逐块量化 (block-wise quantization, blocks of 2048 normalised into [-1, 1]);
    动态量化 (the dynamic tree type: sign, zero-run exponent, indicator bit,
    linear fraction; the unsigned variant reuses the sign bit as fraction).

Precision: the method stores fp32 parameters and runs the Adam update in fp32
(the page's "high-precision state"; the fp32 reading is the one the rest of
the description supports), and the absmax scales are fp32.  So every
element-wise operation here is a single IEEE-754 binary32 operation through
NumPy ``float32`` arrays (NumPy never contracts ``a*b+c`` into an FMA).
Host scalars (bias corrections) are derived in binary64 and rounded once.
Exact rational arithmetic (``fractions.Fraction``) builds the codebooks.

Modules
  codebook  -- the signed / unsigned dynamic-tree maps and their thresholds
  blockwise -- block-wise quantize / dequantize
  adam      -- the fp32 Adam update and the 8-bit Adam step (single, list)
  stable_embedding -- the stable embedding layer (section 二 / 稳定的词嵌入层):
               Xavier-uniform initialisation, lookup + LayerNorm forward and
               backward (binary64); imported as ``oracle.stable_embedding``

Parity status per function is listed in each module's header.
"""

from .codebook import (  # noqa: F401
    BLOCK,
    decode_signed,
    decode_unsigned,
    dynamic_map,
    thresholds,
    nearest_f32,
    zero_code,
)
from .blockwise import quantize_blockwise, dequantize_blockwise  # noqa: F401
from .adam import (  # noqa: F401
    AdamHParams,
    host_scalars,
    adam_update_fp32,
    adam8bit_step,
    adam8bit_step_multi,
    state_init,
)
