"""The moment codec (block_wise_dynamic_gb300.codec): compression is the
block-wise quantizer (bit-exact against the oracle), and switching a run
from torch.optim.Adam/AdamW to the 8-bit optimizer continues with exactly
the oracle's 8-bit step from the compressed moments."""

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
U32 = np.uint32


def test_compress_decompress_bit_exact():
    from block_wise_dynamic_gb300 import codec

    rng = np.random.default_rng(0)
    n = 3 * 2048 + 100
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    v = (rng.standard_normal(n) ** 2 * 1e-6).astype(np.float32)
    mc, ma, vc, va = codec.compress_moments(torch.from_numpy(m).to(DEV), torch.from_numpy(v).to(DEV))
    omc, oma = oracle.quantize_blockwise(m, True)
    ovc, ova = oracle.quantize_blockwise(v, False)
    assert np.array_equal(mc.cpu().numpy(), omc) and np.array_equal(vc.cpu().numpy(), ovc)
    assert np.array_equal(ma.cpu().numpy().view(U32), oma.view(U32))
    assert np.array_equal(va.cpu().numpy().view(U32), ova.view(U32))
    dm, dv = codec.decompress_moments(mc, ma, vc, va)
    assert np.array_equal(dm.cpu().numpy().view(U32), oracle.dequantize_blockwise(omc, oma, True).view(U32))
    assert np.array_equal(dv.cpu().numpy().view(U32), oracle.dequantize_blockwise(ovc, ova, False).view(U32))
    assert codec.compressed_bytes(n) == 2 * n + 8 * 4


@pytest.mark.parametrize("decoupled", [False, True])
def test_switch_from_fp32_adam_mid_training(decoupled):
    import block_wise_dynamic_gb300 as bwd
    from block_wise_dynamic_gb300 import codec

    torch.manual_seed(3)
    wd = 0.05 if decoupled else 0.0
    params = [torch.nn.Parameter(torch.randn(n, device=DEV) * 0.02) for n in (4099, 2048 * 2)]
    fp32 = (torch.optim.AdamW if decoupled else torch.optim.Adam)(params, lr=1e-3, weight_decay=wd)
    for _ in range(3):
        for p in params:
            p.grad = torch.randn_like(p) * 1e-2
        fp32.step()
    opt8 = (bwd.AdamW8bit if decoupled else bwd.Adam8bit)(params, lr=1e-3, weight_decay=wd)
    codec.load_from_fp32_adam(opt8, fp32)
    # oracle: quantize torch's moments, then one 8-bit step at t = 4
    ref = []
    grads = [torch.randn_like(p) * 1e-2 for p in params]
    for p, g in zip(params, grads):
        st = fp32.state[p]
        mc, ma = oracle.quantize_blockwise(st["exp_avg"].cpu().numpy(), True)
        vc, va = oracle.quantize_blockwise(st["exp_avg_sq"].cpu().numpy(), False)
        hp = oracle.AdamHParams(lr=1e-3, weight_decay=wd, step=4)
        ref.append(oracle.adam8bit_step(p.detach().cpu().numpy(), g.cpu().numpy(), mc, ma, vc, va, hp))
        p.grad = g
    opt8.step()
    for p, r in zip(params, ref):
        st = opt8.state[p]
        assert st["step"] == 4
        np.testing.assert_allclose(p.detach().cpu().numpy(), r[0], rtol=1e-5, atol=1e-7)
        assert np.array_equal(st["m_codes"].cpu().numpy(), r[1]) and np.array_equal(st["v_codes"].cpu().numpy(), r[3])
        assert np.array_equal(st["m_absmax"].cpu().numpy(), r[2]) and np.array_equal(st["v_absmax"].cpu().numpy(), r[4])
    # export back: dequantized moments shaped like the parameters
    out = codec.export_fp32_adam_state(opt8)
    for p in params:
        assert out[p]["exp_avg"].shape == p.shape and out[p]["exp_avg_sq"].dtype == torch.float32
        assert float(out[p]["step"]) == 4.0
