"""The AdamW step as "Fused Optimizers and State Precision" defines it.

Section 02 gives one AdamW update, without AMSGrad, minimising, per parameter:

    t = t + 1
    m = beta1*m + (1-beta1)*g
    v = beta2*v + (1-beta2)*g*g
    m_hat = m / (1-beta1**t)
    v_hat = v / (1-beta2**t)
    theta = theta*(1-lr*weight_decay) - lr*m_hat/(sqrt(v_hat)+eps)

``adamw_update`` writes exactly that, in that order, in float64.

The contract around it (sections 02, 03, 06, and the Apex FusedAdam article's
capturable path, section 4.3):

* every parameter group keeps its own lr, betas, eps and weight decay;
* a tensor whose grad is None is not updated at all this step: no decay, no
  moment advance, no step advance (a zero grad is a full update);
* if the whole step is skipped for overflow (found_inf != 0), parameters,
  moments and step counts are all left untouched;
* a grad-scaler's inverse scale multiplies the stored gradient before any use.

Readings (the pages leave these open):

* The step count t is kept per tensor and advances only when that tensor is
  updated ("effective step", sections 03 and 07).
* Hyper-parameters are used exactly as given (the caller passes the values the
  GPU sees, i.e. fp32-rounded ones, when comparing against the GPU).
* The theta update uses the freshly updated moments before they are stored
  (decode -> update -> re-encode); with compact or 8-bit state the stored
  moments are rounded afterwards.
* Stored values are rounded once, from float64, on every store: theta to the
  param format, moments to the state format (``formats``, ``int8_block``).

fp32 master weights (the Apex fused-optimizers guide, FusedAdam
``master_weights``, sections 4.2 and 4.3): a 16-bit model parameter may carry an
fp32 master copy. The update then works on the master, not on the 16-bit
value: the new theta is stored to the master in fp32, and the model parameter
becomes the master rounded to its 16-bit format (round to nearest even), so
updates smaller than half a 16-bit ulp still accumulate. The gradient stays in
the model's format. Reading: the master starts as the exact fp32 value of the
model parameter, as Apex creates it from the model's parameters.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np

from . import dynamic8, int8_block
from .formats import round_to

# 8-bit state kinds: (encode, decode, code dtype) for m, then for v.
#   "int8"   -- the signed linear block codec for both moments (section 05);
#   "int8uv" -- signed linear m, unsigned linear v (scale max/255);
#   "dyn8"   -- the dynamic-exponent codebook, signed for m, unsigned for v.
CODECS = {
    "int8": ((int8_block.encode, int8_block.decode, np.int8),
             (int8_block.encode, int8_block.decode, np.int8)),
    "int8uv": ((int8_block.encode, int8_block.decode, np.int8),
               (int8_block.encode_unsigned, int8_block.decode_unsigned, np.uint8)),
    "dyn8": ((dynamic8.encode_signed, dynamic8.decode_signed, np.uint8),
             (dynamic8.encode_unsigned, dynamic8.decode_unsigned, np.uint8)),
}


def adamw_update(theta, g, m, v, t, lr, beta1, beta2, eps, weight_decay):
    """One AdamW update of section 02 in float64; returns (theta, m, v)."""
    theta = np.asarray(theta, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m = np.asarray(m, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    theta = theta * (1.0 - lr * weight_decay) - lr * m_hat / (np.sqrt(v_hat) + eps)
    return theta, m, v


@dataclasses.dataclass
class TensorState:
    """One parameter tensor and its optimizer state, as stored.

    ``theta`` holds float64 values representable in ``param_fmt``. For state
    kinds "f32"/"bf16", ``m``/``v`` hold float64 values representable in that
    format; for the 8-bit kinds (``CODECS``) they hold 8-bit codes and
    ``m_scale``/``v_scale`` fp32 per-block scales.
    """
    theta: np.ndarray
    param_fmt: str
    state_kind: str
    m: np.ndarray
    v: np.ndarray
    m_scale: Optional[np.ndarray] = None
    v_scale: Optional[np.ndarray] = None
    step: int = 0
    group: int = 0
    master: Optional[np.ndarray] = None   # fp32 master weights (float64 values)

    def copy(self) -> "TensorState":
        c = lambda a: None if a is None else np.array(a, copy=True)
        return TensorState(c(self.theta), self.param_fmt, self.state_kind,
                           c(self.m), c(self.v), c(self.m_scale), c(self.v_scale),
                           int(self.step), int(self.group), c(self.master))

    def weights(self) -> np.ndarray:
        """The values the update works on: the master when there is one."""
        return self.theta if self.master is None else self.master

    # -- decode / encode ---------------------------------------------------
    def moments(self):
        if self.state_kind in CODECS:
            (_, dec_m, _), (_, dec_v, _) = CODECS[self.state_kind]
            return dec_m(self.m, self.m_scale), dec_v(self.v, self.v_scale)
        return (np.asarray(self.m, dtype=np.float64),
                np.asarray(self.v, dtype=np.float64))

    def store(self, theta, m, v) -> None:
        if self.master is None:
            self.theta = round_to(theta, self.param_fmt)
        else:
            self.master = round_to(theta, "f32")
            self.theta = round_to(self.master, self.param_fmt)
        if self.state_kind in CODECS:
            (enc_m, _, _), (enc_v, _, _) = CODECS[self.state_kind]
            self.m, self.m_scale = enc_m(m)
            self.v, self.v_scale = enc_v(v)
        else:
            self.m = round_to(m, self.state_kind)
            self.v = round_to(v, self.state_kind)


def new_state(theta, param_fmt: str, state_kind: str, group: int = 0,
              step: int = 0, master: bool = False) -> TensorState:
    """Zero moments (the optimizer's lazy zero initialisation); with
    ``master``, an fp32 master equal to the (16-bit) parameter's value."""
    theta = round_to(np.asarray(theta, dtype=np.float64).reshape(-1), param_fmt)
    n = theta.size
    mw = np.array(theta, copy=True) if master else None
    if state_kind in CODECS:
        nb = int8_block.n_blocks(n)
        (_, _, dm), (_, _, dv) = CODECS[state_kind]
        return TensorState(theta, param_fmt, state_kind, np.zeros(n, dm),
                           np.zeros(n, dv), np.zeros(nb, np.float32),
                           np.zeros(nb, np.float32), step, group, mw)
    return TensorState(theta, param_fmt, state_kind, np.zeros(n), np.zeros(n),
                       None, None, step, group, mw)


def _hyper(group):
    if isinstance(group, dict):
        return (group["lr"], group["beta1"], group["beta2"], group["eps"],
                group["weight_decay"])
    return (group.lr, group.beta1, group.beta2, group.eps, group.weight_decay)


def oracle_step(states: List[TensorState], groups: Sequence,
                grads: Sequence[Optional[np.ndarray]], inv_scale: float = 1.0,
                found_inf: float = 0.0) -> None:
    """One optimizer step over a tensor list, in place, fused form.

    ``grads[i]`` is the stored gradient of tensor i (float64 values), or None
    when that tensor has no gradient this step.
    """
    if found_inf != 0.0:
        return
    for st, g in zip(states, grads):
        if g is None:
            continue
        lr, b1, b2, eps, wd = _hyper(groups[st.group])
        t = st.step + 1
        m, v = st.moments()
        g = np.asarray(g, dtype=np.float64).reshape(-1) * float(inv_scale)
        theta, m, v = adamw_update(st.weights(), g, m, v, t, lr, b1, b2, eps, wd)
        st.store(theta, m, v)
        st.step = t


def oracle_step_three_loops(states: List[TensorState], groups: Sequence,
                            grads: Sequence[Optional[np.ndarray]],
                            inv_scale: float = 1.0, found_inf: float = 0.0) -> None:
    """The same step as three separate passes (section 04's byte ledger).

    Pass 1 updates every m, pass 2 every v, pass 3 every theta from the updated
    moments; intermediate moments live in float64 arrays and are stored once at
    the end, so the result must equal the fused form bit for bit.
    """
    if found_inf != 0.0:
        return
    live = [(st, np.asarray(g, dtype=np.float64).reshape(-1) * float(inv_scale))
            for st, g in zip(states, grads) if g is not None]
    new_m, new_v = [], []
    for st, g in live:                                     # pass 1: m
        _, b1, _, _, _ = _hyper(groups[st.group])
        m, _ = st.moments()
        new_m.append(b1 * m + (1.0 - b1) * g)
    for st, g in live:                                     # pass 2: v
        _, _, b2, _, _ = _hyper(groups[st.group])
        _, v = st.moments()
        new_v.append(b2 * v + (1.0 - b2) * g * g)
    for (st, _), m, v in zip(live, new_m, new_v):          # pass 3: theta
        lr, b1, b2, eps, wd = _hyper(groups[st.group])
        t = st.step + 1
        m_hat = m / (1.0 - b1 ** t)
        v_hat = v / (1.0 - b2 ** t)
        theta = st.weights() * (1.0 - lr * wd) - lr * m_hat / (np.sqrt(v_hat) + eps)
        st.store(theta, m, v)
        st.step = t
