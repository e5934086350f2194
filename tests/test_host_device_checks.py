"""The Python binding refuses tensors that live on a different GPU from the
one a call launches on, before anything reaches the library: a kernel given a
pointer into another device's memory would fault.  No GPU is needed: the
tensors are CPU tensors that report a CUDA device."""

import pytest
import torch

import block_wise_dynamic_gb300 as bwd
from block_wise_dynamic_gb300 import embedding as E


class OnDevice(torch.Tensor):
    """A CPU tensor that claims to live on cuda:<index> (host test stand-in)."""

    @staticmethod
    def make(t: torch.Tensor, index: int) -> "OnDevice":
        o = torch.Tensor._make_subclass(OnDevice, t)
        o._fake_index = index
        return o

    @property
    def is_cuda(self):
        return True

    @property
    def device(self):
        return torch.device("cuda", self._fake_index)


def fake(shape, dtype, index):
    return OnDevice.make(torch.zeros(shape, dtype=dtype), index)


def test_need_rejects_another_device():
    x = fake(8, torch.float32, 1)
    with pytest.raises(ValueError, match="cuda:1"):
        bwd._need(x, "x", torch.float32, 8, torch.device("cuda", 0))
    bwd._need(x, "x", torch.float32, 8, torch.device("cuda", 1))  # same device: accepted


def test_quantize_and_dequantize_reject_mixed_devices():
    n = 3000
    x = fake(n, torch.float32, 0)
    with pytest.raises(ValueError, match="codes"):
        bwd.quantize_blockwise(x, "signed", fake(n, torch.uint8, 1), fake(2, torch.float32, 0))
    with pytest.raises(ValueError, match="absmax"):
        bwd.quantize_blockwise(x, "signed", fake(n, torch.uint8, 0), fake(2, torch.float32, 1))
    with pytest.raises(ValueError, match="absmax"):
        bwd.dequantize_blockwise(fake(n, torch.uint8, 0), fake(2, torch.float32, 1), "signed")
    with pytest.raises(ValueError, match="out"):
        bwd.dequantize_blockwise(fake(n, torch.uint8, 0), fake(2, torch.float32, 0), "signed",
                                 out=fake(n, torch.float32, 1))


@pytest.mark.parametrize("which", range(5))
def test_adam_step_rejects_mixed_devices(which):
    n = 5000
    args = [fake(n, torch.bfloat16, 0), fake(n, torch.uint8, 0), fake(3, torch.float32, 0),
            fake(n, torch.uint8, 0), fake(3, torch.float32, 0)]
    args[which] = OnDevice.make(args[which].as_subclass(torch.Tensor), 1)
    with pytest.raises(ValueError, match="cuda:1"):
        bwd.adam8bit_step(fake(n, torch.float32, 0), *args, step=1)


def test_multi_tensor_args_reject_mixed_devices():
    sizes = [3000, 5000]
    ps = [fake(n, torch.float32, 0) for n in sizes]
    gs = [fake(n, torch.float32, 0) for n in sizes]
    st = [[fake(n, torch.uint8, 0), fake(bwd.num_blocks(n), torch.float32, 0),
           fake(n, torch.uint8, 0), fake(bwd.num_blocks(n), torch.float32, 0)] for n in sizes]
    bad_p = [ps[0], fake(5000, torch.float32, 1)]
    with pytest.raises(ValueError, match=r"params\[1\]"):
        bwd.MultiTensorArgs(bad_p, gs, *[[s[k] for s in st] for k in range(4)])
    st[1][3] = fake(bwd.num_blocks(5000), torch.float32, 1)
    with pytest.raises(ValueError, match=r"v_absmax\[1\]"):
        bwd.MultiTensorArgs(ps, gs, *[[s[k] for s in st] for k in range(4)])


def test_embedding_calls_reject_mixed_devices():
    v, d, t = 10, 8, 4
    w = fake((v, d), torch.float32, 0)
    with pytest.raises(ValueError, match="ids"):
        E.forward(fake(t, torch.int64, 1), w, fake(d, torch.float32, 0), fake(d, torch.float32, 0))
    with pytest.raises(ValueError, match="beta"):
        E.forward(fake(t, torch.int64, 0), w, fake(d, torch.float32, 0), fake(d, torch.float32, 1))
    good = dict(ids=fake(t, torch.int64, 0), weight=w, gamma=fake(d, torch.float32, 0),
                mean=fake(t, torch.float32, 0), rstd=fake(t, torch.float32, 0), dy=fake((t, d), torch.float32, 0),
                dweight=fake((v, d), torch.float32, 0), dgamma=fake(d, torch.float32, 0),
                dbeta=fake(d, torch.float32, 0))
    for name in ("dy", "dweight", "dgamma"):
        kw = dict(good)
        kw[name] = OnDevice.make(kw[name].as_subclass(torch.Tensor), 1)
        with pytest.raises(ValueError, match=name):
            E.backward(**kw)
