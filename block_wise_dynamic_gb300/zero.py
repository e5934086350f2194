"""ZeRO-style sharded 8-bit Adam over a torch.distributed process group.

"Яндекс Публикует ЯЛМ 100Б" (Yandex's YaLM-100B training notes), section
"ZeRO" under "Случай с несколькими графическими процессорами": each process
is given one group of the parameters, keeps their values and optimizer state
and is the only process that updates them; the step then costs O(N / P) per
process, the gradients are reduced before it and the parameters gathered by
every process after it.  The 8-bit optimizer page (section 二 / 逐块量化)
makes every 2048-element block independent, so the groups are cut on block
boundaries (``bwd_zero_shard``) and each rank's step, one multi-tensor launch
of the library's fused kernel over its pieces, gives exactly the elements the
unsharded step would.

Per step:
  1. reduce-scatter the flat gradient buffer: rank r receives the reduced
     gradients of its own blocks (the page reduces with all_reduce; only the
     owner reads a block's reduced gradient, and a reduce-scatter delivers
     exactly that at half the traffic);
  2. the fused 8-bit Adam step on the rank's pieces (state for them only);
  3. all-gather the updated parameters in place (optionally asynchronously,
     so the next forward pass can overlap it, as the page suggests).

Buffers: the parameters are copied into one flat padded buffer and replaced
by views of it (as the gradients are, when their dtype is the parameters'),
so every collective moves one contiguous tensor of world x K x 2048
elements, K the blocks per rank.
"""

from __future__ import annotations

import ctypes
from typing import Callable, List, Optional, Sequence, Tuple

import torch
import torch.distributed as dist

from . import _abi
from . import BLOCK, MultiTensorArgs, _lib, num_blocks, state_init

__all__ = ["ShardLayout", "ZeroAdam8bit"]


class ShardLayout:
    """Block-aligned split of a tensor list over ``world`` ranks
    (``bwd_zero_shard``).  Host computation only.

    ``offsets[i]``: start of tensor i in the padded flat space;
    ``pieces[r]``: the (tensor, element offset, element count) pieces of rank
    r, in tensor order; ``shard_numel``: K x 2048 elements per rank;
    ``flat_numel``: world x shard_numel."""

    def __init__(self, sizes: Sequence[int], world: int):
        self.sizes = [int(n) for n in sizes]
        self.world = int(world)
        T = len(self.sizes)
        n = (ctypes.c_int64 * max(T, 1))(*self.sizes)
        self.pieces: List[List[Tuple[int, int, int]]] = []
        k = ctypes.c_int64(0)
        for r in range(self.world):
            cnt = ctypes.c_int32(0)
            ti = (ctypes.c_int32 * max(T, 1))()
            off = (ctypes.c_int64 * max(T, 1))()
            c = (ctypes.c_int64 * max(T, 1))()
            _abi.check(_lib.bwd_zero_shard(T, n, self.world, r, ctypes.byref(k), ctypes.byref(cnt), ti, off, c),
                       "bwd_zero_shard")
            self.pieces.append([(ti[j], off[j], c[j]) for j in range(cnt.value)])
        self.blocks_per_rank = k.value
        self.shard_numel = self.blocks_per_rank * BLOCK
        self.flat_numel = self.world * self.shard_numel
        self.offsets = []
        pos = 0
        for s in self.sizes:
            self.offsets.append(pos)
            pos += num_blocks(s) * BLOCK

    def flat_start(self, rank: int, piece: Tuple[int, int, int]) -> int:
        """Position of a piece of ``rank`` inside that rank's shard slice."""
        ti, off, _ = piece
        return self.offsets[ti] + off - rank * self.shard_numel


class ZeroAdam8bit:
    """8-bit Adam(W) with optimizer state sharded over a process group.

    ``params``: tensors of one dtype (fp32, bf16 or fp16) on this rank's GPU,
    the same list on every rank.  They become views of ``flat_param``; when
    ``grad_dtype`` equals their dtype, ``p.grad`` becomes a view of
    ``flat_grad`` too, so autograd accumulates straight into the buffer the
    collective reads (zero it with :meth:`zero_grad`, not by setting grads to
    None).  Otherwise write the gradients into :meth:`grad_views`.

    ``reduce_op``: "avg" (data-parallel mean; NCCL) or "sum".
    ``local_step``: replaces the library's kernel for the rank's own pieces;
    called as ``local_step(param_views, grad_views, step, hparams)`` (used to
    check the collective plumbing against a reference step on CPU)."""

    def __init__(self, params: Sequence[torch.Tensor], *, group=None, lr=1e-3, betas=(0.9, 0.999), eps=1e-8,
                 weight_decay=0.0, grad_dtype: Optional[torch.dtype] = None, reduce_op: str = "avg",
                 local_step: Optional[Callable] = None):
        params = list(params)
        if not params:
            raise ValueError("no parameters")
        dtypes = {p.dtype for p in params}
        devices = {p.device for p in params}
        if len(dtypes) != 1 or len(devices) != 1:
            raise TypeError("all parameters must share one dtype and one device")
        if len({id(p) for p in params}) != len(params):
            raise ValueError("a parameter appears more than once")
        if reduce_op not in ("avg", "sum"):
            raise ValueError("reduce_op must be 'avg' or 'sum'")
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.params = params
        self.hparams = dict(lr=lr, beta1=betas[0], beta2=betas[1], eps=eps, weight_decay=weight_decay)
        self.op = dist.ReduceOp.AVG if reduce_op == "avg" else dist.ReduceOp.SUM
        self.local_step = local_step
        self.t = 0
        L = self.layout = ShardLayout([p.numel() for p in params], self.world)
        dev, pdt = params[0].device, params[0].dtype
        gdt = grad_dtype or pdt
        self.flat_param = torch.zeros(L.flat_numel, dtype=pdt, device=dev)
        self.flat_grad = torch.zeros(L.flat_numel, dtype=gdt, device=dev)
        self.grad_shard = torch.zeros(L.shard_numel, dtype=gdt, device=dev)
        with torch.no_grad():
            for p, off in zip(params, L.offsets):
                n = p.numel()
                self.flat_param[off:off + n].copy_(p.detach().reshape(-1))
                p.data = self.flat_param[off:off + n].view_as(p)
                # a gradient left elsewhere would be ignored by the step: either a
                # view of the flat buffer or nothing (then use grad_views())
                p.grad = self.flat_grad[off:off + n].view_as(p) if gdt == pdt else None
        s0 = self.rank * L.shard_numel
        self.param_shard = self.flat_param[s0:s0 + L.shard_numel]
        mine = L.pieces[self.rank]
        self.piece_params = [self.param_shard[L.flat_start(self.rank, pc):][:pc[2]] for pc in mine]
        self.piece_grads = [self.grad_shard[L.flat_start(self.rank, pc):][:pc[2]] for pc in mine]
        self.state = None
        self._args = None
        if local_step is None and mine:
            self.state = [state_init(pc[2], dev) for pc in mine]
            self._args = MultiTensorArgs(self.piece_params, self.piece_grads,
                                         *[[s[k] for s in self.state] for k in range(4)])

    def grad_views(self) -> List[torch.Tensor]:
        """Per parameter, its gradient's place in the flat gradient buffer."""
        return [self.flat_grad[o:o + p.numel()].view_as(p) for p, o in zip(self.params, self.layout.offsets)]

    def zero_grad(self) -> None:
        self.flat_grad.zero_()

    def reduce_gradients(self) -> None:
        """Phase 1: reduce-scatter the flat gradients; this rank's shard of
        the reduced gradients lands in ``grad_shard``."""
        dist.reduce_scatter_tensor(self.grad_shard, self.flat_grad, op=self.op, group=self.group)

    @torch.no_grad()
    def local_update(self) -> None:
        """Phase 2: the 8-bit Adam step on this rank's pieces (one
        multi-tensor launch of the library's fused kernel)."""
        t = self.t + 1
        if self.local_step is not None:
            self.local_step(self.piece_params, self.piece_grads, t, dict(self.hparams))
        elif self._args is not None:
            self._args.step(step=t, **self.hparams)
        self.t = t

    def gather_parameters(self, async_op: bool = False):
        """Phase 3: all-gather the updated parameter shards in place; with
        ``async_op`` the work handle of the gather in flight is returned."""
        return dist.all_gather_into_tensor(self.flat_param, self.param_shard, group=self.group, async_op=async_op)

    @torch.no_grad()
    def step(self, async_gather: bool = False):
        """Reduce-scatter, local 8-bit step, all-gather.  With
        ``async_gather`` the gather is left in flight and its work handle
        returned (wait on it before the parameters are read)."""
        self.reduce_gradients()
        self.local_update()
        work = self.gather_parameters(async_op=async_gather)
        return work if async_gather else None

    def state_dict(self) -> dict:
        """This rank's share: step count and the 8-bit state of its pieces."""
        keys = ("m_codes", "m_absmax", "v_codes", "v_absmax")
        return {"step": self.t, "rank": self.rank, "world": self.world,
                "pieces": list(self.layout.pieces[self.rank]),
                "state": [dict(zip(keys, (x.clone() for x in s))) for s in (self.state or [])]}

    def load_state_dict(self, sd: dict) -> None:
        if sd["world"] != self.world or sd["rank"] != self.rank or \
                [tuple(p) for p in sd["pieces"]] != self.layout.pieces[self.rank]:
            raise ValueError("state of a different sharding")
        keys = ("m_codes", "m_absmax", "v_codes", "v_absmax")
        for mine, saved in zip(self.state or [], sd["state"]):
            for k, dst in zip(keys, mine):
                dst.copy_(saved[k])
        self.t = int(sd["step"])
