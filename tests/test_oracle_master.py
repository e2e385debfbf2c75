"""Pins of the oracle's fp32 master-weight path against facts outside the oracle.

With a master (the Apex fused-optimizers guide, FusedAdam ``master_weights``,
sections 4.2 and 4.3) the update works on an fp32 copy and the 16-bit model
parameter is that copy rounded to nearest even:

* the master sequence is exactly fp32-parameter training from the same start
  and the same gradients, a path pinned by the closed forms of the AdamW
  tests; the model parameter equals torch's fp32 -> bf16 / fp16 cast of it;
* constant gradient: the master follows the closed form
  theta_t = d^t theta_0 - lr*s*sum_{k<t} d^k (s = g/(|g|+eps)), and updates
  below half a 16-bit ulp, which a 16-bit parameter alone never takes, add up
  to whole ulps of the model parameter;
* a skipped step (found_inf) or a missing gradient leaves master and model
  parameter bit-identical;
* a planted mistake, updating from the 16-bit value instead of the master,
  fails the closed form;
* without a master, a 16-bit parameter follows the constant-gradient
  recurrence from its stored value, rounded by torch's casts, step by step.
"""
import numpy as np
import pytest
import torch

from oracle import adamw as oadamw
from oracle.adamw import new_state, oracle_step
from oracle.formats import round_to

GROUP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)


def _torch_cast(x, fmt):
    dt = {"bf16": torch.bfloat16, "f16": torch.float16}[fmt]
    return torch.from_numpy(np.asarray(x, np.float32)).to(dt).to(torch.float64).numpy()


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
@pytest.mark.parametrize("state_kind", ["f32", "bf16", "int8"])
def test_master_is_fp32_training_and_model_is_its_cast(fmt, state_kind):
    rng = np.random.default_rng(7)
    n = 700
    theta0 = round_to(rng.normal(0, 0.02, n), fmt)
    groups = [dict(GROUP, weight_decay=0.01)]
    a = new_state(theta0, fmt, state_kind, master=True)
    b = new_state(theta0, "f32", state_kind)          # plain fp32 parameters
    assert np.array_equal(a.master, b.theta)
    for s in range(12):
        g = round_to(rng.normal(0, 1e-3, n), fmt)     # gradients in the model format
        oracle_step([a], groups, [g])
        oracle_step([b], groups, [g])
        assert np.array_equal(a.master, b.theta), s
        assert np.array_equal(a.theta, _torch_cast(a.master, fmt)), s
        assert a.step == b.step == s + 1


def _closed_form(theta0, t, lr, wd, g, eps):
    d = 1.0 - lr * wd
    s = g / (abs(g) + eps)
    return d ** t * theta0 - lr * s * sum(d ** k for k in range(t))


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
@pytest.mark.parametrize("wd", [0.0, 0.05])
def test_sub_ulp_updates_accumulate_in_the_master(fmt, wd):
    lr, eps, g = 1e-3, 1e-8, 2.0 ** -10
    group = [dict(GROUP, lr=lr, weight_decay=wd, eps=eps)]
    with_master = new_state(np.array([1.0]), fmt, "f32", master=True)
    without = new_state(np.array([1.0]), fmt, "f32")
    ulp_below_one = 2.0 ** -8 if fmt == "bf16" else 2.0 ** -11
    moved = 0
    for t in range(1, 21):
        oracle_step([with_master, without], group * 1, [np.array([g]), np.array([g])])
        exact = _closed_form(1.0, t, lr, wd, g, eps)
        # fp32 rounding of the master: at most half an ulp per step
        assert abs(with_master.master[0] - exact) <= t * 2.0 ** -24
        assert with_master.theta[0] == _torch_cast([exact], fmt)[0]
        moved = max(moved, round((1.0 - with_master.theta[0]) / ulp_below_one))
        if fmt == "bf16" and wd == 0.0:
            # every update (about 1e-3) is below half a bf16 ulp under 1.0
            assert without.theta[0] == 1.0
    assert moved >= 2


def test_skip_and_missing_grad_leave_master_untouched():
    rng = np.random.default_rng(3)
    a = new_state(rng.normal(0, 0.02, 300), "bf16", "f32", master=True)
    oracle_step([a], [GROUP], [round_to(rng.normal(0, 1e-3, 300), "bf16")])
    snap = a.copy()
    oracle_step([a], [GROUP], [round_to(rng.normal(0, 1e-3, 300), "bf16")], found_inf=1.0)
    oracle_step([a], [GROUP], [None])
    assert np.array_equal(a.master, snap.master) and np.array_equal(a.theta, snap.theta)
    assert a.step == snap.step == 1


def test_planted_update_from_the_16bit_value_fails(monkeypatch):
    monkeypatch.setattr(oadamw.TensorState, "weights", lambda self: self.theta)
    with pytest.raises(AssertionError):
        test_sub_ulp_updates_accumulate_in_the_master("bf16", 0.0)


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_16bit_params_without_master_follow_rounded_recurrence(fmt, wd):
    """16-bit params without a master: with a constant gradient (m_hat = g,
    v_hat = g^2 at every t), each step is theta <- cast(theta*(1 - lr*wd) -
    lr*g/(|g| + eps)) from the stored value, the cast being torch's
    fp64 -> fp32 -> 16-bit rounding; the oracle's sequence must equal it."""
    lr, eps = 3e-3, 1e-8
    rng = np.random.default_rng(4)
    theta0 = _torch_cast(rng.normal(0, 0.5, 64), fmt)
    g = _torch_cast(rng.normal(0, 1e-2, 64), fmt)
    st = new_state(theta0, fmt, "f32")
    grp = [dict(GROUP, lr=lr, weight_decay=wd, eps=eps)]
    th = theta0.copy()
    for t in range(1, 31):
        oracle_step([st], grp, [g])
        # float64 recurrence with the constant-gradient moments, then the casts
        exact = th * (1.0 - lr * wd) - lr * g / (np.abs(g) + eps)
        th = _torch_cast(exact.astype(np.float32), fmt)
        # one 16-bit ulp allowed where the float64 value sits on a rounding
        # boundary between the fp32 and direct roundings
        ulp = np.abs(th) * (2.0 ** -7 if fmt == "bf16" else 2.0 ** -10)
        assert np.all(np.abs(st.theta - th) <= ulp), t
        th = st.theta.copy()                  # continue from the stored value
    assert not np.array_equal(st.theta, theta0)
