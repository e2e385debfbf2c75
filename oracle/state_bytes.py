"""Optimizer-state byte ledger.

"Fused Optimizers and State Precision", section 05: for 100M parameters two
fp32 moments are an 800 MB payload, two 16-bit moments 400 MB, two 8-bit codes
200 MB plus low-bit metadata. The ApexW Unsloth benchmark page reports the
optimizer state of a 24.3M-parameter LoRA run as 185.501 MB (AdamW),
92.751 MB (compact) and 47.101 MB (8-bit).

Layout counted here (one step counter of 4 bytes per tensor):

* "f32":  two fp32 moments              -> 8 bytes per element
* "bf16": two bf16 moments              -> 4 bytes per element
* "int8": two int8 codes + two fp32 scales per 256-element block of each tensor
* "int8uv", "dyn8": the same bytes (other codecs, section 05 variants)

Selective precision (section 05 cites bitsandbytes' selective high-precision
settings): with ``min_8bit_size``, tensors smaller than it keep fp32 moments.
"""
from __future__ import annotations

from typing import Iterable

BYTES_PER_ELEM = {"f32": 8, "bf16": 4, "int8": 2, "int8uv": 2, "dyn8": 2}
EIGHT_BIT = ("int8", "int8uv", "dyn8")
STEP_BYTES = 4
BLOCK = 256
SCALE_BYTES = 4


def tensor_state_bytes(n: int, state_kind: str, with_step: bool = True) -> int:
    b = BYTES_PER_ELEM[state_kind] * int(n)
    if state_kind in EIGHT_BIT:
        b += 2 * SCALE_BYTES * (-(-int(n) // BLOCK))
    if with_step:
        b += STEP_BYTES
    return b


def kind_for(n: int, state_kind: str, min_8bit_size: int = 0) -> str:
    """Selective precision: an 8-bit plan keeps fp32 moments for tensors with
    fewer than ``min_8bit_size`` elements."""
    return "f32" if state_kind in EIGHT_BIT and int(n) < min_8bit_size else state_kind


def state_bytes(numels: Iterable[int], state_kind: str, with_step: bool = True,
                min_8bit_size: int = 0) -> int:
    return sum(tensor_state_bytes(n, kind_for(n, state_kind, min_8bit_size), with_step)
               for n in numels)
