"""Drop-in replacement for ``torch.optim.Adam`` with 8-bit block-wise states.

The page on "8-BIT OPTIMIZERS VIA BLOCK-WISE QUANTIZATION" says switching to
the 8-bit optimizer takes two lines of code (introduction and 总结); this
class is that switch:

    from block_wise_dynamic_gb300 import Adam8bit
    opt = Adam8bit(model.parameters(), lr=1e-3, betas=(0.9, 0.999), eps=1e-8)

``AdamW8bit`` is the same with decoupled weight decay.

Parameters are fp32 (master weights), bf16 or fp16 CUDA tensors (widened for
the update, stored back rounded to nearest even); gradients fp32, bf16 or
fp16.  Per parameter the state holds ``step`` and the codes and absmax of
both moments; ``state_dict()`` / ``load_state_dict()`` round-trip them
exactly.  Each ``step()`` issues one multi-tensor launch per (device,
gradient dtype, step count) group.  The launch tables are built once per
parameter group and reused: when gradients are fresh tensors each step (the
default ``zero_grad(set_to_none=True)``), a step only re-reads the gradient
pointers.
"""

from __future__ import annotations

from collections import defaultdict

import torch

from . import MultiTensorArgs, num_blocks, state_init


class Adam8bit(torch.optim.Optimizer):
    """8-bit Adam (``weight_decay`` must be 0: torch.optim.Adam's coupled L2
    decay is not part of this step; use :class:`AdamW8bit` for decay)."""

    _decoupled = False

    def __init__(self, params, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.0):
        if lr < 0.0:
            raise ValueError(f"invalid learning rate {lr}")
        if not (0.0 <= betas[0] < 1.0 and 0.0 <= betas[1] < 1.0):
            raise ValueError(f"invalid betas {betas}")
        if eps < 0.0:
            raise ValueError(f"invalid eps {eps}")
        if weight_decay < 0.0 or (weight_decay != 0.0 and not self._decoupled):
            raise ValueError("Adam8bit takes no weight decay; AdamW8bit applies it decoupled")
        super().__init__(params, dict(lr=lr, betas=betas, eps=eps, weight_decay=weight_decay))
        self._args_cache = {}

    def _state_for(self, p: torch.Tensor):
        st = self.state[p]
        if len(st) == 0:
            mc, ma, vc, va = state_init(p.numel(), p.device)
            st["step"] = 0
            st["m_codes"], st["m_absmax"], st["v_codes"], st["v_absmax"] = mc, ma, vc, va
        return st

    def _plan(self, params, grads):
        """Launch plan of one parameter group: its parameters with a gradient,
        bucketed by (device, parameter dtype, gradient dtype, step count), each
        bucket with its argument table (parameter and state pointers fixed)."""
        buckets = defaultdict(list)
        for i, (p, g) in enumerate(zip(params, grads)):
            if g is None:
                continue
            if p.dtype not in (torch.float32, torch.bfloat16, torch.float16) or not p.is_cuda:
                raise TypeError("Adam8bit needs fp32, bf16 or fp16 CUDA parameters")
            if g.is_sparse:
                raise TypeError("sparse gradients are not supported")
            st = self._state_for(p)
            if st["m_absmax"].numel() != num_blocks(p.numel()):
                raise ValueError("state does not match the parameter size")
            buckets[(p.device, p.dtype, g.dtype, st["step"])].append(i)
        plan = []
        for (_, _, _, t), idx in buckets.items():
            sts = [self.state[params[i]] for i in idx]
            gs = [grads[i] if grads[i].is_contiguous() else grads[i].contiguous() for i in idx]
            args = MultiTensorArgs(
                [params[i].view(-1) for i in idx], [g.view(-1) for g in gs],
                [s["m_codes"] for s in sts], [s["m_absmax"] for s in sts],
                [s["v_codes"] for s in sts], [s["v_absmax"] for s in sts],
            )
            plan.append([idx, sts, args, t])
        return {"params": list(params), "has_grad": [g is not None for g in grads], "buckets": plan}

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        for gi, group in enumerate(self.param_groups):
            params = group["params"]
            grads = [p.grad for p in params]
            plan = self._args_cache.get(gi)
            fresh = (plan is None or len(plan["params"]) != len(params)
                     or not all(a is b for a, b in zip(plan["params"], params))
                     or plan["has_grad"] != [g is not None for g in grads])
            if fresh:
                plan = self._args_cache[gi] = self._plan(params, grads)
            b1, b2 = group["betas"]
            for bucket in plan["buckets"]:
                idx, sts, args, t = bucket
                if not fresh:
                    try:
                        args.set_grads([grads[i] for i in idx])
                    except (TypeError, ValueError):
                        # a gradient changed dtype or shape: rebuild this group's plan next step
                        self._args_cache.pop(gi, None)
                        raise
                args.step(lr=group["lr"], beta1=b1, beta2=b2, eps=group["eps"],
                          weight_decay=group["weight_decay"], step=t + 1)
                # the step count advances only once its launch went through
                bucket[3] = t + 1
                for s in sts:
                    s["step"] = t + 1
        return loss

    def _reset_plans(self):
        """Forget the cached launch plans (after the state was replaced)."""
        self._args_cache = {}

    def load_state_dict(self, state_dict):
        self._reset_plans()
        super().load_state_dict(state_dict)
        # torch casts every floating parameter's state tensors to the
        # parameter dtype; codes are integers 0..255, so casting back is exact
        for st in self.state.values():
            for k in ("m_codes", "v_codes"):
                if k in st and st[k].dtype != torch.uint8:
                    st[k] = st[k].to(torch.uint8)


class AdamW8bit(Adam8bit):
    """8-bit AdamW: decoupled weight decay, p <- p * (1 - lr * weight_decay)
    before the Adam update (torch.optim.AdamW's rule)."""

    _decoupled = True

    def __init__(self, params, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=1e-2):
        super().__init__(params, lr=lr, betas=betas, eps=eps, weight_decay=weight_decay)
