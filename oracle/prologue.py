"""Gradient prologue before the update: unscale, non-finite check, clipping.

"Fused Optimizers and State Precision", section 06: mixed-precision training
first unscales the gradients, checks them for non-finite values and clips them
(as the recipe says), then runs the update; a step skipped by that check must
leave parameters, moments and step counts untouched. The Apex fused-optimizers
guide (FusedAdam capturable path, section 4.3; FusedLAMB global gradient norm,
section 5.3) does the check and the global L2 norm on the device.

Readings (the pages give no formulas for these):

* found_inf is 1 when any unscaled gradient value g*inv_scale of a tensor that
  has a gradient is NaN or infinite, else 0. This flag is decided by floating
  point, so it is decided in fp32, the kernel's precision: a stored value that
  overflows fp32 once unscaled counts as infinite.
* The global norm is the L2 norm of all unscaled gradient values of the tensors
  that have a gradient.
* Clipping follows the usual global-norm rule: coefficient
  min(1, max_norm / (norm + 1e-6)); max_norm <= 0 disables clipping. The
  update then sees g * inv_scale * coefficient, so the combined factor is
  handed to the step as its inverse scale. When found_inf is set the factor
  is inv_scale (the step is skipped anyway).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

CLIP_EPS = 1e-6


def grad_prologue(grads: Sequence[Optional[np.ndarray]], inv_scale: float,
                  max_norm: float):
    """Returns (found_inf, norm, scale) in float64 from stored gradients
    (None for tensors without a gradient)."""
    found = False
    total = 0.0
    for g in grads:
        if g is None:
            continue
        g = np.asarray(g).reshape(-1)
        with np.errstate(over="ignore", invalid="ignore"):
            x32 = g.astype(np.float32) * np.float32(inv_scale)
        if not np.all(np.isfinite(x32)):
            found = True
        else:
            x = g.astype(np.float64) * float(np.float32(inv_scale))
            total += float(np.sum(x * x))
    if found:
        return 1.0, float("nan"), float(inv_scale)
    norm = float(np.sqrt(total))
    coef = 1.0
    if max_norm > 0.0:
        coef = min(1.0, float(max_norm) / (norm + CLIP_EPS))
    return 0.0, norm, float(inv_scale) * coef
