"""Seeded synthetic workloads for the fused multi-tensor AdamW step.

This module is shared by the CUDA path's tests and benchmark and by the oracle's
tests. It holds shapes, parameter-group tables, per-step schedules (which
tensors have a gradient, which step overflows) and seeded random fills. It holds
none of the optimizer's arithmetic.

Workload shapes follow the pages' own scenarios:

* ``tiny``        -- the worked example of "Fused Optimizers and State Precision"
                     section 02 (theta=[1,-2], g=[0.1,-0.2]) plus two small
                     tensors with ragged sizes.
* ``few_large``   -- eight 4096x4096 fp32 matrices ("few large tensors", the
                     ApexW news piece, where the fused path is said to win).
* ``llama3_8b``   -- the parameter list of an 8B Llama-3-shaped model, bf16
                     params and grads (``llama3_8b_layer``: one of its layers).
* ``many_small``  -- 20,000 tensors with log-uniform sizes in [1, 65536] plus 50
                     4096x1024 matrices ("many small tensors", where the ApexW
                     news piece says fused launches lose), three groups, 10% of
                     grads absent per step, one overflowing step.
* ``lora``        -- the rank-16 LoRA adapter set of the ApexW Unsloth
                     benchmark (24,313,856 params over 392 tensors).

Readings where the pages leave a choice (all stated once here):

* ``N(0, s)`` names a normal distribution with standard deviation ``s``.
* The LoRA benchmark states no weight decay; the AdamW default 0.01 is used.
  A matrices start ~N(0, 0.02), B matrices start at zero (LoRA convention).
* "1% of blocks all-zero" is a fixed seeded set of 256-element blocks, zero on
  every step.
* The overflowing step of ``many_small`` plants +inf and NaN at a few seeded
  positions of a few seeded gradients.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import List, Optional, Sequence

import numpy as np

PARAM_DTYPES = ("f32", "bf16", "f16")
STATE_KINDS = ("f32", "bf16", "int8")
INT8_BLOCK = 256


@dataclasses.dataclass(frozen=True)
class Group:
    lr: float
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0


@dataclasses.dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple
    group: int = 0

    @property
    def numel(self) -> int:
        return int(math.prod(self.shape)) if self.shape else 1


@dataclasses.dataclass
class Workload:
    name: str
    tensors: List[TensorSpec]
    groups: List[Group]
    param_dtype: str = "f32"
    steps: int = 10
    seed: int = 0
    param_std: float = 0.02
    grad_std: float = 1e-3
    grad_prescale: float = 1.0          # grads are stored multiplied by this
    none_fraction: float = 0.0          # fraction of tensors without grad per step
    found_inf_steps: Sequence[int] = ()  # 1-based steps whose found_inf flag is 1
    zero_block_fraction: float = 0.0    # fixed fraction of 256-blocks with zero grad
    zero_init: Sequence[str] = ()       # names of tensors that start at 0
    fixed_values: dict = dataclasses.field(default_factory=dict)
    # fixed_values: name -> {"theta": [...], "grad1": [...]} (page worked example)

    # ----- sizes --------------------------------------------------------
    @property
    def numels(self) -> List[int]:
        return [t.numel for t in self.tensors]

    @property
    def total_numel(self) -> int:
        return int(sum(self.numels))

    @property
    def inv_scale(self) -> float:
        return 1.0 / self.grad_prescale

    # ----- per-step schedule -------------------------------------------
    def present(self, step: int) -> np.ndarray:
        """Boolean mask of tensors that have a gradient at 1-based ``step``."""
        n = len(self.tensors)
        if self.none_fraction <= 0.0:
            return np.ones(n, dtype=bool)
        rng = np.random.default_rng(_seed(self.seed, "present", step))
        return rng.random(n) >= self.none_fraction

    def found_inf(self, step: int) -> bool:
        return int(step) in set(int(s) for s in self.found_inf_steps)

    def zero_blocks(self, i: int) -> np.ndarray:
        """Indices of the 256-element blocks of tensor ``i`` whose grad is 0."""
        if self.zero_block_fraction <= 0.0:
            return np.zeros(0, dtype=np.int64)
        nb = -(-self.tensors[i].numel // INT8_BLOCK)
        rng = np.random.default_rng(_seed(self.seed, "zeroblk", i))
        return np.nonzero(rng.random(nb) < self.zero_block_fraction)[0]

    def poison(self, step: int) -> List[tuple]:
        """(tensor, flat index, value) triples planted in grads of ``step``.

        Only overflowing steps are poisoned: +inf and NaN at a few seeded
        positions of a few seeded tensors, so a step that ignored found_inf
        would visibly corrupt state.
        """
        if not self.found_inf(step):
            return []
        rng = np.random.default_rng(_seed(self.seed, "poison", step))
        n = len(self.tensors)
        out = []
        for k, i in enumerate(rng.choice(n, size=min(4, n), replace=False)):
            j = int(rng.integers(0, self.tensors[int(i)].numel))
            out.append((int(i), j, math.inf if k % 2 == 0 else math.nan))
        return out


def _seed(*parts) -> int:
    h = hashlib.sha256(repr(parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


# ---------------------------------------------------------------------------
# workload definitions
# ---------------------------------------------------------------------------

def tiny(param_dtype: str = "f32") -> Workload:
    """Worked example plus ragged small tensors; one group, 10 steps."""
    g = Group(lr=0.01, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
    return Workload(
        name=f"tiny_{param_dtype}",
        tensors=[TensorSpec("worked", (2,)), TensorSpec("ragged", (257,)),
                 TensorSpec("matrix", (64, 33))],
        groups=[g], param_dtype=param_dtype, steps=10, seed=0,
        param_std=0.02, grad_std=1e-2,
        fixed_values={"worked": {"theta": [1.0, -2.0], "grad1": [0.1, -0.2]}})


def few_large(n: int = 8, rows: int = 4096, cols: int = 4096) -> Workload:
    return Workload(
        name=f"few_large_{n}x{rows}x{cols}",
        tensors=[TensorSpec(f"w{i}", (rows, cols)) for i in range(n)],
        groups=[Group(lr=1e-3, weight_decay=0.01)],
        param_dtype="f32", steps=110, seed=0, param_std=0.02, grad_std=1e-3)


def llama3_8b(layers: int = 32, hidden: int = 4096, kv: int = 1024,
              inter: int = 14336, vocab: int = 128256) -> Workload:
    t: List[TensorSpec] = [TensorSpec("embed", (vocab, hidden), 0)]
    for l in range(layers):
        p = f"layer{l}."
        t += [TensorSpec(p + "q", (hidden, hidden), 0),
              TensorSpec(p + "k", (kv, hidden), 0),
              TensorSpec(p + "v", (kv, hidden), 0),
              TensorSpec(p + "o", (hidden, hidden), 0),
              TensorSpec(p + "gate", (inter, hidden), 0),
              TensorSpec(p + "up", (inter, hidden), 0),
              TensorSpec(p + "down", (hidden, inter), 0),
              TensorSpec(p + "attn_norm", (hidden,), 1),
              TensorSpec(p + "mlp_norm", (hidden,), 1)]
    t += [TensorSpec("final_norm", (hidden,), 1),
          TensorSpec("lm_head", (vocab, hidden), 0)]
    groups = [Group(lr=3e-4, weight_decay=0.1), Group(lr=3e-4, weight_decay=0.0)]
    return Workload(name=f"llama3_8b_L{layers}", tensors=t, groups=groups,
                    param_dtype="bf16", steps=20, seed=0, param_std=0.02,
                    grad_std=1e-3)


def llama3_8b_layer(hidden: int = 4096, kv: int = 1024, inter: int = 14336) -> Workload:
    """One transformer layer of the ``llama3_8b`` list (9 tensors, 218,112,000
    elements): the same shapes, dtypes and groups, small enough (about 2.6 GB
    of state with fp32 moments) for detailed profiler captures."""
    full = llama3_8b(layers=1, hidden=hidden, kv=kv, inter=inter)
    t = [x for x in full.tensors if x.name.startswith("layer0.")]
    return dataclasses.replace(full, name="llama3_8b_layer", tensors=t)


def many_small(n_small: int = 20000, n_big: int = 50, big_shape=(4096, 1024),
               max_small: int = 65536) -> Workload:
    rng = np.random.default_rng(0)
    u = rng.random(n_small)
    sizes = np.clip(np.round(np.exp(u * math.log(max_small))), 1, max_small)
    t = [TensorSpec(f"s{i}", (int(s),), i % 3) for i, s in enumerate(sizes)]
    t += [TensorSpec(f"b{j}", tuple(big_shape), (n_small + j) % 3)
          for j in range(n_big)]
    groups = [Group(lr=1e-3, weight_decay=0.01), Group(lr=5e-4, weight_decay=0.0),
              Group(lr=1e-4, weight_decay=0.1)]
    return Workload(name=f"many_small_{n_small}+{n_big}", tensors=t, groups=groups,
                    param_dtype="f32", steps=20, seed=0, param_std=0.02,
                    grad_std=1e-3, grad_prescale=1024.0, none_fraction=0.10,
                    found_inf_steps=(5,))


def many_small_only(n_small: int = 20000) -> Workload:
    """The 20,000 log-uniform tensors of ``many_small`` without its 50 large
    matrices (about 118M elements): the small-tensor part on its own, with
    the same groups, absent-gradient schedule and overflow step."""
    full = many_small(n_small=n_small)
    return dataclasses.replace(full, name=f"many_small_only_{n_small}",
                               tensors=full.tensors[:n_small])


LORA_MODULES = (("q", 3072, 3072), ("k", 3072, 1024), ("v", 3072, 1024),
                ("o", 3072, 3072), ("gate", 3072, 8192), ("up", 3072, 8192),
                ("down", 8192, 3072))


def lora(layers: int = 28, rank: int = 16, steps: int = 250) -> Workload:
    t: List[TensorSpec] = []
    for l in range(layers):
        for name, fan_in, fan_out in LORA_MODULES:
            t.append(TensorSpec(f"l{l}.{name}.A", (rank, fan_in)))
            t.append(TensorSpec(f"l{l}.{name}.B", (fan_out, rank)))
    return Workload(name=f"lora_r{rank}_L{layers}", tensors=t,
                    groups=[Group(lr=2e-4, weight_decay=0.01)], param_dtype="f32",
                    steps=steps, seed=0, param_std=0.02, grad_std=1e-3,
                    zero_block_fraction=0.01,
                    zero_init=tuple(x.name for x in t if x.name.endswith(".B")))


def mixed(sizes: Sequence[int], param_dtype: str = "f32", groups: int = 2,
          steps: int = 6, none_fraction: float = 0.0, seed: int = 1,
          found_inf_steps: Sequence[int] = (), grad_prescale: float = 1.0,
          zero_block_fraction: float = 0.0) -> Workload:
    """Ad-hoc list of 1-D tensors for parity cases (ragged tails, many tiles)."""
    grp = [Group(lr=1e-3 * (k + 1), beta1=0.9 - 0.05 * k, beta2=0.999 - 0.004 * k,
                 eps=1e-8 * (10 ** k), weight_decay=0.01 * k) for k in range(groups)]
    t = [TensorSpec(f"t{i}", (int(n),), i % groups) for i, n in enumerate(sizes)]
    return Workload(name=f"mixed_{len(sizes)}", tensors=t, groups=grp,
                    param_dtype=param_dtype, steps=steps, seed=seed,
                    param_std=0.02, grad_std=1e-3, grad_prescale=grad_prescale,
                    none_fraction=none_fraction, found_inf_steps=found_inf_steps,
                    zero_block_fraction=zero_block_fraction)


# ---------------------------------------------------------------------------
# seeded fills (torch; CPU or CUDA generator)
# ---------------------------------------------------------------------------

TORCH_DTYPE = {"f32": "float32", "bf16": "bfloat16", "f16": "float16"}


def torch_dtype(name: str):
    import torch
    return getattr(torch, TORCH_DTYPE[name])


def _gen(device, *parts):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


def init_param(wl: Workload, i: int, device="cpu", dtype: Optional[str] = None):
    """Initial parameter tensor ``i`` (seeded per tensor)."""
    import torch
    spec = wl.tensors[i]
    dt = torch_dtype(dtype or wl.param_dtype)
    if spec.name in wl.fixed_values:
        return torch.tensor(wl.fixed_values[spec.name]["theta"],
                            dtype=torch.float32).to(dt).to(device).reshape(spec.shape)
    if spec.name in wl.zero_init:
        return torch.zeros(spec.shape, dtype=dt, device=device)
    x = torch.empty(spec.shape, dtype=torch.float32, device=device)
    x.normal_(0.0, wl.param_std, generator=_gen(device, wl.seed, "param", i))
    return x.to(dt)


def fill_grad(wl: Workload, i: int, step: int, out, scratch=None) -> None:
    """Write the stored (pre-scaled) gradient of tensor ``i`` at 1-based ``step``
    into ``out`` (any device/dtype; values are generated in fp32 and cast)."""
    import torch
    spec = wl.tensors[i]
    device = out.device
    fixed = wl.fixed_values.get(spec.name)
    if fixed is not None and step == 1 and "grad1" in fixed:
        v = torch.tensor(fixed["grad1"], dtype=torch.float32) * wl.grad_prescale
        out.copy_(v.reshape(spec.shape).to(out.dtype))
        return
    x = scratch if scratch is not None else torch.empty(
        spec.shape, dtype=torch.float32, device=device)
    x = x.view(-1)[: spec.numel].view(spec.shape)
    x.normal_(0.0, wl.grad_std, generator=_gen(device, wl.seed, "grad", i, step))
    if wl.grad_prescale != 1.0:
        x.mul_(wl.grad_prescale)
    zb = wl.zero_blocks(i)
    if zb.size:
        flat = x.view(-1)
        idx = torch.from_numpy(zb).to(device)
        offs = torch.arange(INT8_BLOCK, device=device)
        el = (idx[:, None] * INT8_BLOCK + offs[None, :]).reshape(-1)
        el = el[el < spec.numel]
        flat[el] = 0.0
    for (ti, j, val) in wl.poison(step):
        if ti == i:
            x.view(-1)[j] = val
    out.copy_(x.to(out.dtype))


def grad(wl: Workload, i: int, step: int, device="cpu", dtype: Optional[str] = None):
    import torch
    spec = wl.tensors[i]
    out = torch.empty(spec.shape, dtype=torch_dtype(dtype or wl.param_dtype),
                      device=device)
    fill_grad(wl, i, step, out)
    return out
