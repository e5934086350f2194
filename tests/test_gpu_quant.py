"""GPU parity: block-wise quantize / dequantize through the C ABI, bit-exact
against the oracle (section 二 / 逐块量化 and 动态量化 of "8-BIT OPTIMIZERS VIA
BLOCK-WISE QUANTIZATION")."""

import numpy as np
import pytest
import torch

import oracle
from block_wise_dynamic_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
U32 = np.uint32


@pytest.fixture(scope="module")
def bwd():
    from block_wise_dynamic_gb300 import build

    build.build()
    import block_wise_dynamic_gb300 as m

    m.init(0)
    return m


def kind(signed):
    return "signed" if signed else "unsigned"


def gpu_quant(bwd, x_np, signed):
    x = torch.from_numpy(np.ascontiguousarray(x_np, np.float32)).to(DEV)
    c, a = bwd.quantize_blockwise(x, kind(signed))
    return c.cpu().numpy(), a.cpu().numpy()


def gpu_dequant(bwd, c_np, a_np, signed):
    c = torch.from_numpy(c_np).to(DEV)
    a = torch.from_numpy(a_np).to(DEV)
    return bwd.dequantize_blockwise(c, a, kind(signed)).cpu().numpy()


SIZES = [1, 2, 31, 2047, 2048, 2049, 4095, 4096, 3 * 2048 + 17, (1 << 20) + 123]


@pytest.mark.parametrize("signed", [True, False])
@pytest.mark.parametrize("n", SIZES)
def test_quantize_dequantize_bit_exact(bwd, n, signed):
    x = W.quant_input(n, seed=n).numpy()
    if not signed:
        x = x * x
    c, a = gpu_quant(bwd, x, signed)
    co, ao = oracle.quantize_blockwise(x, signed)
    assert np.array_equal(a.view(U32), ao.view(U32))
    assert np.array_equal(c, co)
    y = gpu_dequant(bwd, co, ao, signed)
    yo = oracle.dequantize_blockwise(co, ao, signed)
    assert np.array_equal(y.view(U32), yo.view(U32))


@pytest.mark.parametrize("signed", [True, False])
def test_unaligned_buffers_take_the_elementwise_path(bwd, signed):
    n = 5 * 2048 + 300
    x = W.quant_input(n + 1, seed=9).to(DEV)
    if not signed:
        x = x * x
    xv = x[1:]  # 4-byte offset: not 16-byte aligned
    codes = torch.empty(n + 3, dtype=torch.uint8, device=DEV)[3:]
    absmax = torch.empty((n + 2047) // 2048, dtype=torch.float32, device=DEV)
    bwd.quantize_blockwise(xv, kind(signed), codes=codes, absmax=absmax)
    co, ao = oracle.quantize_blockwise(xv.cpu().numpy(), signed)
    assert np.array_equal(codes.cpu().numpy(), co)
    assert np.array_equal(absmax.cpu().numpy().view(U32), ao.view(U32))
    out = torch.empty(n + 1, dtype=torch.float32, device=DEV)[1:]
    bwd.dequantize_blockwise(codes, absmax, kind(signed), out=out)
    yo = oracle.dequantize_blockwise(co, ao, signed)
    assert np.array_equal(out.cpu().numpy().view(U32), yo.view(U32))


@pytest.mark.parametrize("signed", [True, False])
def test_zero_blocks_and_signed_zeros(bwd, signed):
    B = 2048
    x = np.zeros(4 * B + 5, np.float32)
    x[B:2 * B] = -0.0
    x[2 * B:3 * B] = np.linspace(-1, 1, B, dtype=np.float32) if signed else np.linspace(0, 1, B, dtype=np.float32)
    x[2 * B + 7] = -0.0
    x[2 * B + 9] = 0.0
    x[3 * B + 1] = -1e-30 if signed else 1e-30
    c, a = gpu_quant(bwd, x, signed)
    co, ao = oracle.quantize_blockwise(x, signed)
    assert np.array_equal(c, co) and np.array_equal(a.view(U32), ao.view(U32))
    z = 128 if signed else 0
    assert np.all(c[:2 * B] == z) and a[0] == 0 and a[1] == 0
    y = gpu_dequant(bwd, c, a, signed)
    assert np.array_equal(y.view(U32), oracle.dequantize_blockwise(co, ao, signed).view(U32))


def _bits_range(lo_bits, hi_bits):
    return np.arange(lo_bits, hi_bits + 1, dtype=np.uint32).view(np.float32)


def _normalised_sweep(signed):
    """Normalised values that stress the code decision: every value of
    [0.5, 1]; +-64 ulps around every threshold; +-2 ulps around every 2^-16
    of the binary32 pattern range (the bucket edges of the lookup); a stride
    through all of (0, 1]; and tiny values."""
    t = oracle.thresholds(signed)
    parts = [_bits_range(0x3F000000, 0x3F800000)]
    tb = np.abs(t[t != 0]).view(U32).astype(np.int64)
    offs = np.arange(-64, 65)
    parts.append((tb[:, None] + offs[None, :]).ravel().astype(U32).view(np.float32))
    edges = (np.arange((127 - 27) << 7, (127 << 7) + 1, dtype=np.int64) << 16)
    parts.append((edges[:, None] + np.arange(-2, 3)[None, :]).ravel().astype(U32).view(np.float32))
    parts.append(_bits_range(1, 0x3F800000)[::97])
    parts.append(np.array([0.0, 1e-45, 1e-38, 1e-30, 4.9999997e-8, 5e-8, 5.0000004e-8], np.float32))
    v = np.unique(np.concatenate(parts))
    v = v[(v >= 0) & (v <= 1)]
    if signed:
        v = np.concatenate([v, -v])
    return v.astype(np.float32)


@pytest.mark.parametrize("signed", [True, False])
def test_code_decision_sweep(bwd, signed):
    """Blocks lead with 1.0, so absmax = 1 and x / absmax = x: the codes of
    the swept values must equal the oracle's."""
    v = _normalised_sweep(signed)
    per = 2047
    nb = (v.size + per - 1) // per
    pad = np.zeros(nb * per, np.float32)
    pad[: v.size] = v
    rows = np.concatenate([np.ones((nb, 1), np.float32), pad.reshape(nb, per)], axis=1).ravel()
    c, a = gpu_quant(bwd, rows, signed)
    co, ao = oracle.quantize_blockwise(rows, signed)
    assert np.all(a == 1.0)
    bad = np.nonzero(c != co)[0]
    assert bad.size == 0, f"{bad.size} codes differ, first at value {rows[bad[0]]!r}"


@pytest.mark.parametrize("offset", [0, 4])
@pytest.mark.parametrize("signed", [True, False])
def test_many_blocks_per_group_bit_exact(bwd, signed, offset):
    """Enough blocks that every quantizer group and dequantizer CTA walks
    several of them (the staged copies and the rotating output buffers are
    reused), a partial last block, and buffers 16 bytes past the allocation
    start (still the vector path): every code, absmax and value bit-exact."""
    n = (1 << 24) + 5 * 2048 + 77
    x = W.quant_input(n + offset, seed=21).to(DEV)
    if not signed:
        x = x * x
    xv = x[offset:]
    codes = torch.empty(n + offset, dtype=torch.uint8, device=DEV)[offset:]
    absmax = torch.empty((n + 2047) // 2048, dtype=torch.float32, device=DEV)
    bwd.quantize_blockwise(xv, kind(signed), codes=codes, absmax=absmax)
    co, ao = oracle.quantize_blockwise(xv.cpu().numpy(), signed)
    assert np.array_equal(absmax.cpu().numpy().view(U32), ao.view(U32))
    assert np.array_equal(codes.cpu().numpy(), co)
    out = torch.empty(n + offset, dtype=torch.float32, device=DEV)[offset:]
    bwd.dequantize_blockwise(codes, absmax, kind(signed), out=out)
    yo = oracle.dequantize_blockwise(co, ao, signed)
    assert np.array_equal(out.cpu().numpy().view(U32), yo.view(U32))


def test_full_size_2p28_sampled(bwd):
    """The 2^28-element workload: absmax of every block checked against a
    plain max, codes and dequantized values of sampled blocks bit-exact."""
    n = 1 << 28
    B = 2048
    x = W.quant_input(n, seed=0, device=DEV)
    rng = np.random.default_rng(0)
    nb = n // B
    out_blocks = np.unique((np.nonzero((x.abs() > 20).view(-1, B).any(1).cpu().numpy())[0]))
    sample = np.unique(np.concatenate([[0, nb - 1], rng.choice(nb, 96, replace=False), out_blocks[:32]]))
    for signed in (True, False):
        xs = x if signed else x * x
        c, a = bwd.quantize_blockwise(xs, kind(signed))
        torch.cuda.synchronize()
        ref_absmax = xs.view(-1, B).abs().amax(dim=1)
        assert torch.equal(a, ref_absmax)
        y = bwd.dequantize_blockwise(c, a, kind(signed))
        xc = xs.view(-1, B)[sample].cpu().numpy()
        cc = c.view(-1, B)[sample].cpu().numpy()
        yc = y.view(-1, B)[sample].cpu().numpy()
        for r in range(len(sample)):
            co, ao = oracle.quantize_blockwise(xc[r], signed)
            assert np.array_equal(cc[r], co)
            yo = oracle.dequantize_blockwise(co, ao, signed)
            assert np.array_equal(yc[r].view(U32), yo.view(U32))
        del c, a, y, xs
    del x
    torch.cuda.empty_cache()


@pytest.mark.parametrize("signed", [True, False])
def test_extreme_block_scales(bwd, signed):
    """Blocks whose absmax is subnormal, tiny, or close to FLT_MAX (the
    divisor takes IEEE division there) and blocks mixing a huge absmax with
    subnormal values, all bit-exact."""
    rng = np.random.default_rng(21)
    B = 2048
    scales = [1e-44, 1e-40, 3e-38, 1e-30, 1.0, 1e30, 1e37, 5e37]  # |x| stays finite
    rows = []
    for s in scales:
        r = (rng.standard_normal(B) * np.float32(s)).astype(np.float32)
        rows.append(r)
    mixed = (rng.standard_normal(B) * 1e-42).astype(np.float32)
    mixed[7] = np.float32(3.0e38)
    rows.append(mixed)
    neg_tiny = -np.abs(rng.standard_normal(B) * 1e-44).astype(np.float32)
    neg_tiny[3] = np.float32(2.5)  # -> tiny negative quotients, -0.0 vs negative subnormal
    rows.append(neg_tiny)
    x = np.concatenate(rows)
    if not signed:
        x = np.abs(x)
    c, a = gpu_quant(bwd, x, signed)
    co, ao = oracle.quantize_blockwise(x, signed)
    assert np.array_equal(a.view(U32), ao.view(U32))
    assert np.array_equal(c, co)


def test_non_finite_inputs_do_not_fault(bwd):
    """Outside the method, but they must not fault or touch other blocks."""
    B = 2048
    x = W.quant_input(4 * B, seed=5).numpy()
    x[10] = np.nan
    x[B + 3] = np.inf
    x[2 * B + 1] = -np.inf
    for signed in (True, False):
        c, a = gpu_quant(bwd, x, signed)
        co, ao = oracle.quantize_blockwise(x[3 * B:], signed)
        assert np.array_equal(c[3 * B:], co) and a[3] == ao[0]


def test_tensor_larger_than_2p31_elements(bwd):
    """64-bit indexing: one tensor of 2^31 + 2049 elements; the blocks at the
    2^31 boundary and the ragged tail are checked against the oracle."""
    B = 2048
    n = (1 << 31) + 2049
    x = torch.empty(n, dtype=torch.float32, device=DEV)
    x.normal_(0.0, 1.0, generator=torch.Generator(device=DEV).manual_seed(3))
    c, a = bwd.quantize_blockwise(x, "signed")
    y = bwd.dequantize_blockwise(c, a, "signed")
    torch.cuda.synchronize()
    nb = (n + B - 1) // B
    for b in (0, (1 << 31) // B - 1, (1 << 31) // B, nb - 1):
        lo, hi = b * B, min(n, (b + 1) * B)
        xb = x[lo:hi].cpu().numpy()
        co, ao = oracle.quantize_blockwise(xb, True)
        assert np.array_equal(c[lo:hi].cpu().numpy(), co)
        assert a[b].item() == ao[0]
        yo = oracle.dequantize_blockwise(co, ao, True)
        assert np.array_equal(y[lo:hi].cpu().numpy().view(U32), yo.view(U32))
    del x, c, a, y
    torch.cuda.empty_cache()


def test_nan_in_another_warp_than_the_block_maximum(bwd):
    """A NaN and the block's largest finite value in different warps, finite
    values up to 3e38, an all-NaN block, NaN beside infinity: the maxima
    ignore NaN, so the absmax is the largest finite magnitude and every
    finite element gets the oracle's code for the block with the NaN at 0;
    nothing faults."""
    B = 2048
    rng = np.random.default_rng(21)
    x = (rng.standard_normal(6 * B)).astype(np.float32)
    x[3] = np.nan                      # warp 0 of block 0 (quads 4 t + 512 k + j: thread 0)
    x[1500] = 3e38                     # a thread of another warp holds the maximum
    x[B + 700] = -np.nan
    x[B + 5] = -2.5e38
    x[2 * B:3 * B] = np.nan            # all NaN
    x[3 * B + 9] = np.nan
    x[3 * B + 10] = np.inf             # NaN beside infinity
    x[4 * B + 2047] = np.nan           # last element
    for signed in (True, False):
        with np.errstate(over="ignore"):
            xs = x if signed else np.where(np.isnan(x), x, x * x).astype(np.float32)
        c, a = gpu_quant(bwd, xs, signed)
        for b in (0, 1, 4):
            blk = xs[b * B:(b + 1) * B]
            fin = np.isfinite(blk)  # (squares of +-3e38 overflow to infinity on the unsigned side)
            with np.errstate(invalid="ignore"):  # inf / inf in a block holding an infinity
                co, ao = oracle.quantize_blockwise(np.where(np.isnan(blk), 0.0, blk).astype(np.float32), signed)
            assert a[b] == ao[0]
            assert np.array_equal(c[b * B:(b + 1) * B][fin], co[fin])
        co, ao = oracle.quantize_blockwise(xs[5 * B:], signed)
        assert np.array_equal(c[5 * B:], co) and a[5] == ao[0]


@pytest.mark.parametrize("signed", [True, False])
def test_tiny_quotients_on_both_sides_of_the_unscaled_switch(bwd, signed):
    """Block absmax just below and above 2^-38 and 2^126 (where the
    quantizers switch between the unscaled and scaled exact divisions) and
    elsewhere, each block holding quotients down to 2^-80 of both signs,
    signed zeros and subnormals (the unsigned map sees negative values too):
    codes and absmax bit-identical to the oracle."""
    B = 2048
    rng = np.random.default_rng(23)
    tops = [2.0 ** -38 * f for f in (0.6, 0.99, 1.0, 1.01, 1.5)]
    tops += [2.0 ** 126 * f for f in (0.9, 0.99, 1.0, 1.5)]
    tops += list(2.0 ** rng.uniform(-120, 120, 16))
    rows = []
    for top in tops:
        r = rng.standard_normal(B)
        r *= top / np.abs(r).max()
        k = rng.integers(0, B, 400)
        r[k] = rng.choice([-1.0, 1.0], 400) * 2.0 ** rng.uniform(-80, -30, 400) * top
        r[rng.integers(0, B, 8)] = -0.0
        r[rng.integers(0, B, 8)] = 0.0
        rows.append(r.astype(np.float32))
    x = np.concatenate(rows)
    fields = (np.abs(x).reshape(-1, B).max(axis=1).view(U32) >> 23) & 0xFF
    assert {88, 89, 252, 253} <= set(fields.tolist())
    c, a = gpu_quant(bwd, x, signed)
    co, ao = oracle.quantize_blockwise(x, signed)
    assert np.array_equal(a.view(U32), ao.view(U32))
    assert np.array_equal(c, co)
