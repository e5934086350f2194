"""The synthetic workloads have the sizes their descriptions state."""

import numpy as np
import torch

from block_wise_dynamic_gb300 import workloads as W


def test_llama2_7b_set():
    shapes = W.llama2_7b_shapes()
    assert len(shapes) == 291
    n = sum(s for _, s in shapes)
    assert n == 6_738_415_616
    assert all(s % 2048 == 0 for _, s in shapes)
    assert (n + 2047) // 2048 == 3_290_242


def test_gpt_350m_set():
    shapes = W.gpt_350m_shapes()
    assert len(shapes) == 292
    n = sum(s for _, s in shapes)
    assert n == 354_871_296 == 173_277 * 2048
    wl = W.workload("gpt_350m")
    assert wl.sizes == (n,) and wl.grad_dtype == torch.bfloat16


def test_ragged_set():
    sizes, sig = W.ragged_2000()
    assert len(sizes) == 2000
    assert min(sizes) >= 1000 and max(sizes) < 16_777_216
    assert 3.0e9 < sum(sizes) < 4.0e9
    assert sum(1 for s in sizes if s % 2048 == 0) < 20
    assert 1e-5 <= min(sig) and max(sig) <= 1e-1


def test_generators_are_seeded():
    a = W.gen_normal(1000, 0.02, 3)
    b = W.gen_normal(1000, 0.02, 3)
    assert torch.equal(a, b)
    assert not torch.equal(a, W.gen_normal(1000, 0.02, 4))
    g = W.gen_normal(1000, 1e-3, 5, dtype=torch.bfloat16)
    assert g.dtype == torch.bfloat16
    x = W.quant_input(1 << 16, 0)
    big = (x.abs() > 20).sum().item()
    assert 30 <= big <= 66  # ~0.1% of 65536 scaled by 100
    assert np.isclose(float(x.std()), 3.3, rtol=0.5)
