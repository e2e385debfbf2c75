"""Torch-side holder of one parameter set's optimizer state.

Allocates zeroed moment buffers (8-bit codes and their block scales for the
8-bit kinds, fp32 moments for tensors kept in fp32), optional fp32 master
weights, the per-tensor int32 step counters, and the plan, using torch only
for device memory; the step itself is ``adamw_step`` in the CUDA library.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import torch

from ._binding import (CS_INT8_BLOCK, CS_TENSOR_STATE_F32, EIGHT_BIT, Plan,
                       adamw_grad_prologue, adamw_plan_create, adamw_plan_set_grads,
                       adamw_step, pack_present, tensor_desc)

# storage dtype of (m, v) per state kind (8-bit codes are raw bytes)
STATE_TORCH_DTYPES = {"f32": (torch.float32, torch.float32),
                      "bf16": (torch.bfloat16, torch.bfloat16),
                      "int8": (torch.int8, torch.int8),
                      "int8uv": (torch.int8, torch.uint8),
                      "dyn8": (torch.uint8, torch.uint8)}
STATE_TORCH_DTYPE = {k: v[0] for k, v in STATE_TORCH_DTYPES.items()}


class AdamWState:
    """Moments, scales and step counts for ``params`` (flat per tensor).

    params, grads: same-length lists of CUDA tensors (grads same dtype/numel).
    group_of: per-tensor group index (default 0).
    master: keep fp32 master weights for the 16-bit params (initialised to
    their exact fp32 values); the step then updates the master and writes
    each 16-bit param as its rounding.
    min_8bit_size: with an 8-bit state kind, tensors with fewer elements keep
    fp32 moments (``fp32_state[i]`` tells which).
    """

    def __init__(self, params: Sequence[torch.Tensor], grads: Sequence[torch.Tensor],
                 state_kind: str = "f32", group_of: Optional[Sequence[int]] = None,
                 unit_elems: int = 0, master: bool = False, min_8bit_size: int = 0):
        if len(params) != len(grads):
            raise ValueError("params and grads differ in length")
        self.params = list(params)
        self.grads = list(grads)
        self.state_kind = state_kind
        n = len(self.params)
        self.group_of = list(group_of) if group_of is not None else [0] * n
        mdt, vdt = STATE_TORCH_DTYPES[state_kind]
        dev = self.params[0].device if n else torch.device("cuda")
        self.m: List[torch.Tensor] = []
        self.v: List[torch.Tensor] = []
        self.m_scale: List[Optional[torch.Tensor]] = []
        self.v_scale: List[Optional[torch.Tensor]] = []
        self.master: List[Optional[torch.Tensor]] = []
        self.fp32_state: List[bool] = []
        descs = []
        for p, g, grp in zip(self.params, self.grads, self.group_of):
            if p.numel() != g.numel() or p.dtype != g.dtype:
                raise ValueError("grad must match its param in numel and dtype")
            ne = p.numel()
            f32 = state_kind in EIGHT_BIT and ne < min_8bit_size
            m = torch.zeros(ne, dtype=torch.float32 if f32 else mdt, device=dev)
            v = torch.zeros(ne, dtype=torch.float32 if f32 else vdt, device=dev)
            self.fp32_state.append(f32)
            if state_kind in EIGHT_BIT and not f32:
                nb = -(-ne // CS_INT8_BLOCK)
                ms = torch.zeros(max(nb, 1), dtype=torch.float32, device=dev)
                vs = torch.zeros(max(nb, 1), dtype=torch.float32, device=dev)
            else:
                ms = vs = None
            self.m.append(m)
            self.v.append(v)
            self.m_scale.append(ms)
            self.v_scale.append(vs)
            mw = None
            if master and p.dtype != torch.float32:
                mw = p.detach().reshape(-1).to(torch.float32)
            self.master.append(mw)
            descs.append(tensor_desc(p, g, m, v, ms, vs, group=grp, master=mw,
                                     flags=CS_TENSOR_STATE_F32 if f32 else 0))
        self.step = torch.zeros(max(n, 1), dtype=torch.int32, device=dev)
        self.plan: Plan = adamw_plan_create(descs, state_kind, unit_elems)

    def run(self, groups, present=None, inv_scale=None, found_inf=None, stream=None):
        """One optimizer step (asynchronous on ``stream``)."""
        bits = None if present is None else pack_present(present, len(self.params))
        adamw_step(self.plan, groups, bits, self.step, inv_scale, found_inf, stream)

    def prologue(self, present=None, inv_scale=None, max_norm: float = 0.0, stream=None):
        """Non-finite flag, global norm and clip factor of this step's grads, as
        device fp32 tensors (found_inf, norm, scale); pass found_inf and scale
        to run() as found_inf and inv_scale."""
        dev = self.step.device
        if not hasattr(self, "_pro_out"):
            self._pro_out = torch.zeros(3, dtype=torch.float32, device=dev)
        o = self._pro_out
        bits = None if present is None else pack_present(present, len(self.params))
        adamw_grad_prologue(self.plan, bits, inv_scale, max_norm, o[0:1], o[1:2], o[2:3], stream)
        return o[0:1], o[1:2], o[2:3]

    def set_grads(self, grads: Sequence[torch.Tensor], stream=None) -> None:
        self.grads = list(grads)
        adamw_plan_set_grads(self.plan, self.grads, stream)

    def state_tensors(self, i: int):
        """(m, v, m_scale, v_scale, master) of tensor i (None where absent)."""
        return self.m[i], self.v[i], self.m_scale[i], self.v_scale[i], self.master[i]
