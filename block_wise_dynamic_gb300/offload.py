"""8-bit Adam steps whose gradients arrive from, and whose updated parameters
go back to, pinned host memory.

The page on "8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION" (section 一)
names offloading optimizer work to the CPU as the other way to save GPU
memory.  Here the 8-bit state stays on the GPU, and each step moves only the
gradients in and the parameters out.  The tensor list is cut into chunks;
chunk c's gradient copy, its multi-tensor step and its parameter copy run on
three streams ordered by events, so the host-to-device copy of chunk c + 1,
the step of chunk c and the device-to-host copy of chunk c - 1 overlap.
"""

from __future__ import annotations

from typing import List, Sequence

import torch

from . import MultiTensorArgs


class PipelinedHostStep:
    """One object per fixed list of tensors.

    ``dev_params``/``dev_grads``/states: the GPU tensors the step works on
    (as for :class:`MultiTensorArgs`).  ``host_grads``/``host_params``:
    pinned host tensors of the same shapes; every :meth:`step` reads the
    gradients from ``host_grads`` and leaves the updated parameters in
    ``host_params``.  ``chunk_bytes`` bounds the gradient bytes per chunk.
    """

    def __init__(self, dev_params: Sequence[torch.Tensor], dev_grads: Sequence[torch.Tensor],
                 m_codes, m_absmax, v_codes, v_absmax,
                 host_grads: Sequence[torch.Tensor], host_params: Sequence[torch.Tensor],
                 chunk_bytes: int = 256 << 20):
        T = len(dev_params)
        if not (len(dev_grads) == len(host_grads) == len(host_params) == T):
            raise ValueError("all lists must have the same length")
        for i in range(T):
            if not host_grads[i].is_pinned() or not host_params[i].is_pinned():
                raise ValueError("host buffers must be pinned (torch.empty(..., pin_memory=True))")
            if host_grads[i].shape != dev_grads[i].shape or host_params[i].shape != dev_params[i].shape:
                raise ValueError(f"host and device tensors {i} differ in shape")
        self.device = dev_params[0].device if T else None
        self.chunks: List[tuple] = []
        start, acc = 0, 0
        for i in range(T + 1):
            if i == T or (acc > 0 and acc + dev_grads[i].numel() * dev_grads[i].element_size() > chunk_bytes):
                if i > start:
                    sl = slice(start, i)
                    args = MultiTensorArgs(dev_params[sl], dev_grads[sl], m_codes[sl], m_absmax[sl],
                                           v_codes[sl], v_absmax[sl])
                    self.chunks.append((args, list(dev_params[sl]), list(dev_grads[sl]),
                                        list(host_grads[sl]), list(host_params[sl])))
                start, acc = i, 0
            if i < T:
                acc += dev_grads[i].numel() * dev_grads[i].element_size()
        if T:
            self.h2d = torch.cuda.Stream(self.device)
            self.d2h = torch.cuda.Stream(self.device)

    def step(self, *, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, step,
             stream=None) -> None:
        """Enqueue one step; the caller's stream (default: current) runs the
        kernels and, when it is done, the host parameters are complete."""
        if not self.chunks:
            return
        comp = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.h2d.wait_stream(comp)  # gradients may be overwritten only after earlier work
        self.d2h.wait_stream(comp)
        for args, dp, dg, hg, hp in self.chunks:
            with torch.cuda.stream(self.h2d):
                for d, h in zip(dg, hg):
                    d.copy_(h, non_blocking=True)
                arrived = torch.cuda.Event()
                arrived.record(self.h2d)
            comp.wait_event(arrived)
            args.step(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay, step=step,
                      stream=comp)
            stepped = torch.cuda.Event()
            stepped.record(comp)
            self.d2h.wait_event(stepped)
            with torch.cuda.stream(self.d2h):
                for d, h in zip(dp, hp):
                    h.copy_(d, non_blocking=True)
        comp.wait_stream(self.d2h)
