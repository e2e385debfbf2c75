"""ZeRO-style sharded step: every rank updates only its own part of the
parameters and keeps optimizer state for that part alone.

"Fused Optimizers and State Precision", section 06: sharding (ZeRO / FSDP)
decides which rank owns which state, the fused optimizer decides how the local
state is updated, and the two compose. Here the partition is
``adamw_shard_ranges`` (C ABI, host only): the tensors end to end in one flat
buffer, each padded to whole 256-element blocks, cut into ``world`` equal
shards of whole blocks, so no 8-bit scale block is split between ranks.

One sharded step is the local fused step wrapped in the exchange a sharded
data-parallel step needs:

1. reduce-scatter of the flat gradient buffer: rank r receives the sum over
   ranks of its own shard;
2. all-reduce (max) of found_inf, so every rank skips the same steps;
3. the local update: ``adamw_step`` on a plan over the rank's slices (every
   tensor, empty slices included, so every rank advances every tensor's step
   count the same way);
4. all-gather of the parameter shards into every rank's flat buffer.

The collectives are plain ``torch.distributed`` calls (NCCL on GPUs); the
update itself is the CUDA library's. ``exchange_step`` holds the exchange and
takes the local update as a callable, so the exchange can be exercised on its
own.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence

import torch

from ._binding import (CS_INT8_BLOCK, EIGHT_BIT, Plan, adamw_plan_create, adamw_shard_ranges,
                       adamw_step, pack_present, tensor_desc)
from .torch_adapter import STATE_TORCH_DTYPES


class ShardLayout:
    """Rank ``rank``'s part of a tensor list (host arithmetic only)."""

    def __init__(self, numels: Sequence[int], world: int, rank: int):
        self.numels = [int(n) for n in numels]
        self.world = int(world)
        self.rank = int(rank)
        self.lo, self.hi, self.offsets, self.shard_elems = adamw_shard_ranges(
            self.numels, self.world, self.rank)
        self.flat_elems = self.world * self.shard_elems
        self.shard_start = self.rank * self.shard_elems

    def local_numel(self, i: int) -> int:
        return self.hi[i] - self.lo[i]

    def flat_range(self, i: int):
        """Tensor i's elements in the flat buffer."""
        return self.offsets[i], self.offsets[i] + self.numels[i]

    def shard_range(self, i: int):
        """Tensor i's local part within this rank's shard (empty if none)."""
        a = self.offsets[i] + self.lo[i] - self.shard_start
        return (a, a + self.local_numel(i)) if self.local_numel(i) else (0, 0)

    def block_range(self, i: int):
        """The 256-element blocks of tensor i that this rank owns."""
        b0 = self.lo[i] // CS_INT8_BLOCK
        return b0, b0 + -(-self.local_numel(i) // CS_INT8_BLOCK)


def exchange_step(layout: ShardLayout, flat_grad: torch.Tensor, grad_shard: torch.Tensor,
                  flat_param: torch.Tensor, found_inf: Optional[torch.Tensor],
                  local_step: Callable[[Optional[torch.Tensor]], None], group=None) -> None:
    """Reduce-scatter the gradients, agree on found_inf, run ``local_step``
    on this rank's shard, all-gather the parameters."""
    import torch.distributed as dist
    if flat_grad.numel() != layout.flat_elems or flat_param.numel() != layout.flat_elems:
        raise ValueError("flat buffers must hold world * shard_elems elements")
    if grad_shard.numel() != layout.shard_elems:
        raise ValueError("grad_shard must hold shard_elems elements")
    dist.reduce_scatter_tensor(grad_shard, flat_grad, op=dist.ReduceOp.SUM, group=group)
    fi = None
    if found_inf is not None:
        fi = found_inf.clone()
        dist.all_reduce(fi, op=dist.ReduceOp.MAX, group=group)
    local_step(fi)
    s0 = layout.shard_start
    dist.all_gather_into_tensor(flat_param, flat_param[s0:s0 + layout.shard_elems].clone(),
                                group=group)


class ShardedAdamW:
    """The sharded step on one rank: a full replica of the parameters in one
    flat buffer (views per tensor), the flat gradient buffer the backward
    pass fills, and moments, scales and step counts for this rank's part
    only.

    numels:     per-tensor element counts (the model's parameter list).
    param_dtype "f32" | "bf16" | "f16"; state_kind as for adamw_plan_create.
    group_of:   per-tensor group index.
    """

    def __init__(self, numels: Sequence[int], param_dtype: str, state_kind: str,
                 group_of: Optional[Sequence[int]], world: int, rank: int,
                 device, unit_elems: int = 0):
        pdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[param_dtype]
        self.layout = L = ShardLayout(numels, world, rank)
        self.state_kind = state_kind
        n = len(L.numels)
        self.group_of = list(group_of) if group_of is not None else [0] * n
        self.flat_param = torch.zeros(L.flat_elems, dtype=pdt, device=device)
        self.flat_grad = torch.zeros(L.flat_elems, dtype=pdt, device=device)
        self.grad_shard = torch.zeros(L.shard_elems, dtype=pdt, device=device)
        s0 = L.shard_start
        self.param_shard = self.flat_param[s0:s0 + L.shard_elems]
        mdt, vdt = STATE_TORCH_DTYPES[state_kind]
        self.m: List[torch.Tensor] = []
        self.v: List[torch.Tensor] = []
        self.m_scale: List[Optional[torch.Tensor]] = []
        self.v_scale: List[Optional[torch.Tensor]] = []
        descs = []
        for i in range(n):
            k = L.local_numel(i)
            a, b = L.shard_range(i)
            m = torch.zeros(k, dtype=mdt, device=device)
            v = torch.zeros(k, dtype=vdt, device=device)
            if state_kind in EIGHT_BIT:
                nb = max(1, -(-k // CS_INT8_BLOCK))
                ms = torch.zeros(nb, dtype=torch.float32, device=device)
                vs = torch.zeros(nb, dtype=torch.float32, device=device)
            else:
                ms = vs = None
            self.m.append(m)
            self.v.append(v)
            self.m_scale.append(ms)
            self.v_scale.append(vs)
            if k == 0:
                # the rank owns none of it: an empty slice still counts the step
                descs.append(tensor_desc(None, None, None, None, numel=0,
                                         param_dtype=param_dtype, group=self.group_of[i]))
            else:
                descs.append(tensor_desc(self.param_shard[a:b], self.grad_shard[a:b], m, v, ms,
                                         vs, group=self.group_of[i]))
        self.step_counts = torch.zeros(max(n, 1), dtype=torch.int32, device=device)
        self.plan: Plan = adamw_plan_create(descs, state_kind, unit_elems)

    def param(self, i: int) -> torch.Tensor:
        """Tensor i of the full replica (flat view; reshape as needed)."""
        a, b = self.layout.flat_range(i)
        return self.flat_param[a:b]

    def grad(self, i: int) -> torch.Tensor:
        a, b = self.layout.flat_range(i)
        return self.flat_grad[a:b]

    def local_step(self, groups, present=None, inv_scale=None, found_inf=None,
                   stream=None) -> None:
        """The fused step on this rank's part only; grad_shard must already
        hold the reduced gradients of the shard."""
        bits = None if present is None else pack_present(present, len(self.layout.numels))
        adamw_step(self.plan, groups, bits, self.step_counts, inv_scale, found_inf, stream)

    def step(self, groups, present=None, inv_scale=None, found_inf=None, group=None) -> None:
        """One sharded step on the current stream: reduce-scatter, found_inf
        agreement, local update, all-gather."""
        exchange_step(self.layout, self.flat_grad, self.grad_shard, self.flat_param, found_inf,
                      lambda fi: self.local_step(groups, present, inv_scale, fi), group)
