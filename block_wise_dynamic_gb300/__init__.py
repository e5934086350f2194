"""GB300-native 8-bit Adam with block-wise dynamic quantization.

Python binding of the C ABI in ``include/bwd.h``: each function checks and
marshals torch CUDA tensors into pointers and sizes and calls the library
entry point of the same name (prefix ``bwd_``); every step of the work runs in
the library's sm_103a kernels.  PyTorch supplies device memory and streams.

Method: "8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION" (summary on
wiki.neutronadmin.com/news/16836), sections 一 and 二.
"""

from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import numpy as np
import torch

from . import _abi
from ._abi import BLOCK, BwdError

__all__ = [
    "BLOCK",
    "BwdError",
    "num_blocks",
    "build_map",
    "init",
    "check_device",
    "quantize_blockwise",
    "dequantize_blockwise",
    "state_init",
    "adam8bit_step",
    "adam8bit_step_multi",
    "MultiTensorArgs",
    "Adam8bit",
    "AdamW8bit",
]

_KINDS = {"signed": _abi.BWD_MAP_SIGNED, "unsigned": _abi.BWD_MAP_UNSIGNED}
_GDT = {torch.float32: _abi.BWD_F32, torch.bfloat16: _abi.BWD_BF16, torch.float16: _abi.BWD_F16}


class _Lib:
    """Loads libbwd.so on first use; a missing build raises ImportError."""

    def __getattr__(self, name):
        return getattr(_abi.load(), name)


_lib = _Lib()


def num_blocks(n: int) -> int:
    """ceil(n / 2048): absmax entries of an n-element tensor."""
    return (int(n) + BLOCK - 1) // BLOCK


def _kind(kind) -> int:
    if isinstance(kind, str):
        if kind not in _KINDS:
            raise ValueError(f"map kind must be one of {sorted(_KINDS)}")
        return _KINDS[kind]
    return int(kind)


def _stream_handle(device: torch.device, stream) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _need(t: torch.Tensor, name: str, dtype, numel: Optional[int] = None,
          device: Optional[torch.device] = None) -> None:
    """Type, layout and size checks; with ``device`` given, the tensor must
    live on that device (the kernel is launched there, and a pointer into
    another GPU's memory would fault)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the call runs on {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} elements, got {t.numel()}")


def build_map(kind="signed"):
    """The 256-entry map and its 255 thresholds (host computation)."""
    m = np.empty(256, np.float32)
    t = np.empty(255, np.float32)
    _abi.check(_lib.bwd_build_map(_kind(kind), m.ctypes.data, t.ctypes.data), "bwd_build_map")
    return m, t


def check_device(device=None, stream=None) -> None:
    """Wait for the stream and raise BwdError if a bounded wait inside one of
    the library's kernels gave up since the last check (the flag is cleared)."""
    dev = torch.device(device if device is not None else torch.cuda.current_device())
    with torch.cuda.device(dev):
        _abi.check(_lib.bwd_check_device(_stream_handle(dev, stream)), "bwd_check_device")


def init(device=None) -> None:
    """Upload the code tables to ``device`` (blocking; do it before capture)."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _abi.check(_lib.bwd_init(), "bwd_init")


def quantize_blockwise(x: torch.Tensor, kind="signed", codes=None, absmax=None, stream=None):
    """Codes (uint8[n]) and per-2048-block absmax (float32) of flat fp32 ``x``."""
    n = x.numel()
    _need(x, "x", torch.float32)
    if codes is None:
        codes = torch.empty(n, dtype=torch.uint8, device=x.device)
    if absmax is None:
        absmax = torch.empty(num_blocks(n), dtype=torch.float32, device=x.device)
    _need(codes, "codes", torch.uint8, n, x.device)
    _need(absmax, "absmax", torch.float32, num_blocks(n), x.device)
    with torch.cuda.device(x.device):
        st = _lib.bwd_quantize_blockwise(
            x.data_ptr(), n, _kind(kind), codes.data_ptr(), absmax.data_ptr(), _stream_handle(x.device, stream)
        )
    _abi.check(st, "bwd_quantize_blockwise")
    return codes, absmax


def dequantize_blockwise(codes: torch.Tensor, absmax: torch.Tensor, kind="signed", out=None, stream=None):
    """map[code] * absmax[block] as a flat float32 tensor."""
    n = codes.numel()
    _need(codes, "codes", torch.uint8)
    _need(absmax, "absmax", torch.float32, num_blocks(n), codes.device)
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=codes.device)
    _need(out, "out", torch.float32, n, codes.device)
    with torch.cuda.device(codes.device):
        st = _lib.bwd_dequantize_blockwise(
            codes.data_ptr(), absmax.data_ptr(), n, _kind(kind), out.data_ptr(), _stream_handle(codes.device, stream)
        )
    _abi.check(st, "bwd_dequantize_blockwise")
    return out


def state_init(n: int, device, stream=None):
    """Fresh 8-bit state for n parameters: (m_codes, m_absmax, v_codes, v_absmax)."""
    device = torch.device(device)
    mc = torch.empty(n, dtype=torch.uint8, device=device)
    vc = torch.empty(n, dtype=torch.uint8, device=device)
    ma = torch.empty(num_blocks(n), dtype=torch.float32, device=device)
    va = torch.empty(num_blocks(n), dtype=torch.float32, device=device)
    with torch.cuda.device(device):
        st = _lib.bwd_state_init(
            mc.data_ptr(), ma.data_ptr(), vc.data_ptr(), va.data_ptr(), n, _stream_handle(device, stream)
        )
    _abi.check(st, "bwd_state_init")
    return mc, ma, vc, va


def _hparams(lr, beta1, beta2, eps, step, weight_decay=0.0) -> _abi.AdamHParams:
    return _abi.AdamHParams(float(lr), float(beta1), float(beta2), float(eps), float(weight_decay), int(step))


def adam8bit_step(p, g, m_codes, m_absmax, v_codes, v_absmax, *, lr=1e-3, beta1=0.9, beta2=0.999,
                  eps=1e-8, weight_decay=0.0, step, stream=None) -> None:
    """One 8-bit Adam step on one flat tensor, in place (``bwd_adam8bit_step``);
    ``weight_decay`` > 0 makes it AdamW (decoupled).  bf16 and fp16
    parameters go through ``bwd_adam8bit_step_multi_ex``."""
    if isinstance(p, torch.Tensor) and p.dtype in (torch.bfloat16, torch.float16):
        return adam8bit_step_multi([p], [g], [m_codes], [m_absmax], [v_codes], [v_absmax], lr=lr, beta1=beta1,
                                   beta2=beta2, eps=eps, weight_decay=weight_decay, step=step, stream=stream)
    n = p.numel()
    _need(p, "p", torch.float32)
    if g.dtype not in _GDT:
        raise TypeError("g must be float32, bfloat16 or float16")
    dev = p.device
    _need(g, "g", g.dtype, n, dev)
    _need(m_codes, "m_codes", torch.uint8, n, dev)
    _need(v_codes, "v_codes", torch.uint8, n, dev)
    _need(m_absmax, "m_absmax", torch.float32, num_blocks(n), dev)
    _need(v_absmax, "v_absmax", torch.float32, num_blocks(n), dev)
    hp = _hparams(lr, beta1, beta2, eps, step, weight_decay)
    with torch.cuda.device(p.device):
        st = _lib.bwd_adam8bit_step(
            p.data_ptr(), g.data_ptr(), _GDT[g.dtype], m_codes.data_ptr(), m_absmax.data_ptr(),
            v_codes.data_ptr(), v_absmax.data_ptr(), n, ctypes.byref(hp), _stream_handle(p.device, stream),
        )
    _abi.check(st, "bwd_adam8bit_step")


class MultiTensorArgs:
    """Host pointer arrays for ``bwd_adam8bit_step_multi``, built once for a
    fixed list of tensors and reused by every step."""

    def __init__(self, params: Sequence[torch.Tensor], grads: Sequence[torch.Tensor],
                 m_codes: Sequence[torch.Tensor], m_absmax: Sequence[torch.Tensor],
                 v_codes: Sequence[torch.Tensor], v_absmax: Sequence[torch.Tensor]):
        T = len(params)
        if not (len(grads) == len(m_codes) == len(m_absmax) == len(v_codes) == len(v_absmax) == T):
            raise ValueError("all lists must have the same length")
        gdt = {g.dtype for g in grads}
        pdt = {p.dtype for p in params}
        if len(gdt) > 1 or len(pdt) > 1:
            raise TypeError("all gradients (and all parameters) of one call must share a dtype")
        self.g_dtype = _GDT[gdt.pop()] if T else _abi.BWD_F32
        self.p_dtype = _GDT[pdt.pop()] if T else _abi.BWD_F32
        self.device = params[0].device if T else None
        dev = self.device
        for i in range(T):
            n = params[i].numel()
            _need(params[i], f"params[{i}]", params[i].dtype, None, dev)
            if params[i].dtype not in _GDT:
                raise TypeError("parameters must be float32, bfloat16 or float16")
            _need(grads[i], f"grads[{i}]", grads[i].dtype, n, dev)
            _need(m_codes[i], f"m_codes[{i}]", torch.uint8, n, dev)
            _need(v_codes[i], f"v_codes[{i}]", torch.uint8, n, dev)
            _need(m_absmax[i], f"m_absmax[{i}]", torch.float32, num_blocks(n), dev)
            _need(v_absmax[i], f"v_absmax[{i}]", torch.float32, num_blocks(n), dev)
        arr = ctypes.c_void_p * T
        self.T = T
        self._keep = (list(params), list(grads), list(m_codes), list(m_absmax), list(v_codes), list(v_absmax))
        self.p = arr(*[t.data_ptr() for t in params])
        self.g = arr(*[t.data_ptr() for t in grads])
        self.mc = arr(*[t.data_ptr() for t in m_codes])
        self.ma = arr(*[t.data_ptr() for t in m_absmax])
        self.vc = arr(*[t.data_ptr() for t in v_codes])
        self.va = arr(*[t.data_ptr() for t in v_absmax])
        self._sizes = [t.numel() for t in params]
        self.n = (ctypes.c_int64 * T)(*self._sizes)
        self.numel = int(sum(self._sizes))
        self._gdtype = grads[0].dtype if T else None

    def set_grads(self, grads: Sequence[torch.Tensor]) -> None:
        """Points the table at new gradient tensors (same sizes, dtype and
        device as before; non-contiguous ones are copied), leaving the
        parameter and state pointers as they are.  This is the per-step work
        when gradients are fresh tensors every step."""
        if len(grads) != self.T:
            raise ValueError(f"expected {self.T} gradients, got {len(grads)}")
        dev, gdt = self.device, self._gdtype
        if not all(isinstance(g, torch.Tensor) and g.dtype == gdt for g in grads):
            raise TypeError(f"every gradient must be a {gdt} tensor, as when the table was built")
        if [g.numel() for g in grads] != self._sizes:
            raise ValueError("gradient sizes differ from the parameters'")
        if not all(g.device == dev for g in grads):
            raise ValueError(f"every gradient must be on {dev}")
        if not all(g.is_contiguous() for g in grads):
            grads = [g if g.is_contiguous() else g.contiguous() for g in grads]
        self._keep = (self._keep[0], list(grads)) + self._keep[2:]
        self.g[:] = [g.data_ptr() for g in grads]

    def step(self, *, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, step,
             stream=None) -> None:
        if self.T == 0:
            return
        hp = _hparams(lr, beta1, beta2, eps, step, weight_decay)
        with torch.cuda.device(self.device):
            st = _lib.bwd_adam8bit_step_multi_ex(
                self.T, self.p, self.p_dtype, self.g, self.g_dtype, self.mc, self.ma, self.vc, self.va,
                self.n, ctypes.byref(hp), _stream_handle(self.device, stream),
            )
        _abi.check(st, "bwd_adam8bit_step_multi_ex")


def adam8bit_step_multi(params, grads, m_codes, m_absmax, v_codes, v_absmax, *, lr=1e-3, beta1=0.9,
                        beta2=0.999, eps=1e-8, weight_decay=0.0, step, stream=None) -> None:
    """One 8-bit Adam(W) step over a list of tensors (``bwd_adam8bit_step_multi_ex``);
    parameters fp32 or bf16, gradients fp32 or bf16."""
    MultiTensorArgs(params, grads, m_codes, m_absmax, v_codes, v_absmax).step(
        lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay, step=step, stream=stream
    )


from .optim import Adam8bit, AdamW8bit  # noqa: E402
