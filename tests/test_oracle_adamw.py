"""Pins of the oracle's AdamW step against facts that do not come from the oracle.

* the worked example printed in "Fused Optimizers and State Precision" section 02
  (tests/golden/worked_example.txt);
* the constant-gradient closed form (m_t=(1-b1^t)g, v_t=(1-b2^t)g^2, so
  m_hat=g, v_hat=g^2 at every t, and theta solves a linear recurrence);
* the unrolled-sum closed form of the moments for arbitrary gradients, evaluated
  in exact rational arithmetic, and theta as the solution of its linear
  recurrence in 60-digit decimal arithmetic;
* the step contract of sections 02, 03 and 06 (grad=None, zero grad, overflow
  skip, per-tensor step counts) and the power-of-two unscale identity;
* section 04: three separate passes give the same result as the fused pass;
* a planted coupled-L2 mutant (section 02 says it is not a valid substitute)
  fails the pins, so they have teeth.
"""
import decimal
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import adamw as oadamw
from oracle.adamw import adamw_update, new_state, oracle_step, oracle_step_three_loops
from tests.conftest import load_golden


GOLD = load_golden("worked_example.txt")


def _worked(update=adamw_update):
    g = GOLD
    return update(np.array(g["theta0"]), np.array(g["grad"]), np.array(g["m0"]),
                  np.array(g["v0"]), 1, g["lr"], g["beta1"], g["beta2"], g["eps"],
                  g["weight_decay"])


def _check_worked(update=adamw_update):
    theta, m, v = _worked(update)
    np.testing.assert_allclose(m, GOLD["m1"], rtol=1e-12, atol=0)
    np.testing.assert_allclose(v, GOLD["v1"], rtol=1e-12, atol=0)
    np.testing.assert_allclose(m / (1 - GOLD["beta1"]), GOLD["m_hat1"], rtol=1e-12)
    np.testing.assert_allclose(v / (1 - GOLD["beta2"]), GOLD["v_hat1"], rtol=1e-12)
    half = 0.5 * 10.0 ** -GOLD["theta1_approx_decimals"]
    assert np.all(np.abs(theta - np.array(GOLD["theta1_approx"])) <= half)
    # with m_hat = g and v_hat = g^2 (page), theta1 = theta0*(1-lr*wd) - lr*g/(|g|+eps)
    g = np.array(GOLD["grad"])
    exact = (np.array(GOLD["theta0"]) * (1 - GOLD["lr"] * GOLD["weight_decay"])
             - GOLD["lr"] * g / (np.abs(g) + GOLD["eps"]))
    np.testing.assert_allclose(theta, exact, rtol=1e-14, atol=0)
    return theta


def test_worked_example_matches_page():
    theta = _check_worked()
    # exact value in the page's notation: [0.999 - 0.001/(0.1+1e-8), ...]
    assert abs(theta[0] - 0.98900000099999990) < 1e-15
    assert abs(theta[1] - (-1.98800000049999998)) < 1e-15


def test_worked_example_through_tensor_step():
    st = new_state(GOLD["theta0"], "f64", "f32")
    grp = dict(lr=GOLD["lr"], beta1=GOLD["beta1"], beta2=GOLD["beta2"],
               eps=GOLD["eps"], weight_decay=GOLD["weight_decay"])
    oracle_step([st], [grp], [np.array(GOLD["grad"])])
    assert st.step == 1
    np.testing.assert_allclose(st.m, GOLD["m1"], rtol=1e-7)   # stored in fp32
    np.testing.assert_allclose(st.v, GOLD["v1"], rtol=1e-7)
    half = 0.5 * 10.0 ** -GOLD["theta1_approx_decimals"]
    assert np.all(np.abs(st.theta - np.array(GOLD["theta1_approx"])) <= half)


@pytest.mark.parametrize("b1,b2,lr,wd,eps", [
    (0.9, 0.999, 1e-3, 0.01, 1e-8),
    (0.8, 0.95, 3e-2, 0.0, 1e-6),
    (0.5, 0.9, 1e-2, 0.3, 1e-3),
])
def test_constant_gradient_closed_form(b1, b2, lr, wd, eps):
    rng = np.random.default_rng(3)
    n, T = 64, 200
    theta0 = rng.normal(0, 0.5, n)
    g = rng.normal(0, 1e-2, n) * np.where(rng.random(n) < 0.1, 1e-4, 1.0)
    theta, m, v = theta0.copy(), np.zeros(n), np.zeros(n)
    for t in range(1, T + 1):
        theta, m, v = adamw_update(theta, g, m, v, t, lr, b1, b2, eps, wd)
        if t in (1, 2, 7, 50, T):
            np.testing.assert_allclose(m, (1 - b1 ** t) * g, rtol=1e-12)
            np.testing.assert_allclose(v, (1 - b2 ** t) * g * g, rtol=1e-12)
            d = 1.0 - lr * wd
            s = g / (np.abs(g) + eps)
            geo = t if wd == 0 else (1 - d ** t) / (1 - d)
            expect = d ** t * theta0 - lr * s * geo
            np.testing.assert_allclose(theta, expect, rtol=1e-11, atol=1e-13)


def _exact_reference(theta0, gs, lr, b1, b2, eps, wd):
    """Moments from the unrolled sums (exact rationals); theta from the solution
    of theta_t = d*theta_{t-1} - lr*u_t, i.e. theta_T = d^T theta_0 -
    lr*sum_k d^(T-k) u_k, with u_k = m_hat_k/(sqrt(v_hat_k)+eps) in decimal."""
    ctx = decimal.Context(prec=60)
    F = Fraction
    B1, B2, LR, WD, EPS = F(b1), F(b2), F(lr), F(wd), F(eps)
    T = len(gs)
    out = []
    for j in range(len(theta0)):
        u = []
        for t in range(1, T + 1):
            m_t = (1 - B1) * sum(B1 ** (t - k) * F(gs[k - 1][j]) for k in range(1, t + 1))
            v_t = (1 - B2) * sum(B2 ** (t - k) * F(gs[k - 1][j]) ** 2 for k in range(1, t + 1))
            mh = m_t / (1 - B1 ** t)
            vh = v_t / (1 - B2 ** t)
            dm = ctx.divide(decimal.Decimal(mh.numerator), decimal.Decimal(mh.denominator))
            dv = ctx.divide(decimal.Decimal(vh.numerator), decimal.Decimal(vh.denominator))
            de = ctx.divide(decimal.Decimal(EPS.numerator), decimal.Decimal(EPS.denominator))
            u.append(ctx.divide(dm, ctx.add(ctx.sqrt(dv), de)))
        D = 1 - LR * WD
        dd = ctx.divide(decimal.Decimal(D.numerator), decimal.Decimal(D.denominator))
        dl = ctx.divide(decimal.Decimal(LR.numerator), decimal.Decimal(LR.denominator))
        th = ctx.multiply(ctx.power(dd, T), decimal.Decimal(F(theta0[j]).numerator)
                          / decimal.Decimal(F(theta0[j]).denominator))
        for k in range(1, T + 1):
            th = ctx.subtract(th, ctx.multiply(dl, ctx.multiply(ctx.power(dd, T - k), u[k - 1])))
        out.append((float(m_t), float(v_t), float(th)))
    return np.array(out)


def test_unrolled_sum_closed_form_varying_grads():
    rng = np.random.default_rng(11)
    n, T = 6, 7
    lr, b1, b2, eps, wd = 0.01, 0.85, 0.99, 1e-6, 0.05
    theta0 = rng.normal(0, 0.1, n)
    gs = [rng.normal(0, 1e-2, n) for _ in range(T)]
    gs[3][2] = 0.0          # a zero gradient mid-run is a full update
    theta, m, v = theta0.copy(), np.zeros(n), np.zeros(n)
    for t in range(1, T + 1):
        theta, m, v = adamw_update(theta, gs[t - 1], m, v, t, lr, b1, b2, eps, wd)
    ref = _exact_reference(theta0, gs, lr, b1, b2, eps, wd)
    np.testing.assert_allclose(m, ref[:, 0], rtol=1e-13)
    np.testing.assert_allclose(v, ref[:, 1], rtol=1e-13)
    np.testing.assert_allclose(theta, ref[:, 2], rtol=1e-13)


def test_grad_none_untouched_zero_grad_updates():
    rng = np.random.default_rng(5)
    grp = [dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)]
    a = new_state(rng.normal(0, 0.02, 33), "f32", "f32")
    b = new_state(rng.normal(0, 0.02, 33), "f32", "f32")
    for s in range(3):        # build up non-zero moments
        oracle_step([a, b], grp, [rng.normal(0, 1e-2, 33)] * 2)
    a0, b0 = a.copy(), b.copy()
    oracle_step([a, b], grp, [None, np.zeros(33)])
    # None: bit-identical everything
    assert a.step == a0.step == 3
    for x, y in [(a.theta, a0.theta), (a.m, a0.m), (a.v, a0.v)]:
        assert x.tobytes() == y.tobytes()
    # zero grad: moments decay, theta decays and moves by the decayed moments
    lr, b1, b2, eps, wd = 1e-2, 0.9, 0.999, 1e-8, 0.1
    t = 4
    m = b1 * b0.m
    v = b2 * b0.v
    exp_theta = b0.theta * (1 - lr * wd) - lr * (m / (1 - b1 ** t)) / (
        np.sqrt(v / (1 - b2 ** t)) + eps)
    assert b.step == 4
    np.testing.assert_allclose(b.m, m, rtol=1e-7)
    np.testing.assert_allclose(b.v, v, rtol=1e-7)
    np.testing.assert_allclose(b.theta, exp_theta, rtol=1e-7)
    assert not np.array_equal(b.theta, b0.theta)


@pytest.mark.parametrize("state_kind", ["f32", "bf16", "int8", "int8uv", "dyn8"])
def test_found_inf_leaves_everything_untouched(state_kind):
    rng = np.random.default_rng(6)
    grp = [dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)]
    sts = [new_state(rng.normal(0, 0.02, n), "bf16", state_kind) for n in (5, 300)]
    oracle_step(sts, grp, [rng.normal(0, 1e-2, 5), rng.normal(0, 1e-2, 300)])
    before = [s.copy() for s in sts]
    bad = [np.full(5, np.inf), np.full(300, np.nan)]
    oracle_step(sts, grp, bad, inv_scale=1.0, found_inf=1.0)
    for s, s0 in zip(sts, before):
        assert s.step == s0.step == 1
        for f in ("theta", "m", "v", "m_scale", "v_scale"):
            x, y = getattr(s, f), getattr(s0, f)
            assert (x is None and y is None) or x.tobytes() == y.tobytes()


@pytest.mark.parametrize("state_kind", ["f32", "bf16", "int8", "int8uv", "dyn8"])
def test_power_of_two_unscale_is_exact(state_kind):
    rng = np.random.default_rng(8)
    grp = [dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)]
    th = rng.normal(0, 0.02, 700)
    a = [new_state(th, "f32", state_kind)]
    b = [new_state(th, "f32", state_kind)]
    for s in range(4):
        g = rng.normal(0, 1e-3, 700)
        oracle_step(a, grp, [g])
        oracle_step(b, grp, [g * 1024.0], inv_scale=1.0 / 1024.0)
    for f in ("theta", "m", "v"):
        assert getattr(a[0], f).tobytes() == getattr(b[0], f).tobytes()


@pytest.mark.parametrize("state_kind", ["f32", "bf16", "int8", "int8uv", "dyn8"])
def test_three_loops_equal_fused(state_kind):
    rng = np.random.default_rng(9)
    groups = [dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01),
              dict(lr=5e-4, beta1=0.8, beta2=0.99, eps=1e-6, weight_decay=0.0)]
    sizes = [1, 7, 256, 513]
    fused = [new_state(rng.normal(0, 0.02, n), "f32", state_kind, group=i % 2)
             for i, n in enumerate(sizes)]
    loops = [s.copy() for s in fused]
    for step in range(12):
        grads = [None if (step + i) % 5 == 0 else rng.normal(0, 1e-3, n)
                 for i, n in enumerate(sizes)]
        fi = 1.0 if step == 6 else 0.0
        oracle_step(fused, groups, grads, found_inf=fi)
        oracle_step_three_loops(loops, groups, grads, found_inf=fi)
    for a, b in zip(fused, loops):
        assert a.step == b.step
        for f in ("theta", "m", "v", "m_scale", "v_scale"):
            x, y = getattr(a, f), getattr(b, f)
            assert (x is None and y is None) or x.tobytes() == y.tobytes()


def test_per_tensor_step_counts_follow_schedule():
    rng = np.random.default_rng(10)
    grp = [dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)]
    sizes = [3, 4, 5, 6]
    sts = [new_state(np.zeros(n), "f32", "f32") for n in sizes]
    expect = [0] * len(sizes)
    for step in range(1, 21):
        present = rng.random(len(sizes)) >= 0.3
        fi = 1.0 if step == 5 else 0.0
        oracle_step(sts, grp, [rng.normal(0, 1, n) if p else None
                               for n, p in zip(sizes, present)], found_inf=fi)
        for i, p in enumerate(present):
            expect[i] += int(p and fi == 0.0)
    assert [s.step for s in sts] == expect


def _coupled_l2(theta, g, m, v, t, lr, beta1, beta2, eps, weight_decay):
    """Planted mistake: weight decay added to the gradient (coupled L2), which
    section 02 says is not a substitute for decoupled AdamW decay."""
    g = np.asarray(g, dtype=np.float64) + weight_decay * np.asarray(theta)
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    return theta - lr * m_hat / (np.sqrt(v_hat) + eps), m, v


def test_planted_coupled_l2_mutant_fails_the_pins(monkeypatch):
    with pytest.raises(AssertionError):
        _check_worked(_coupled_l2)
    # and through the tensor step, on the moments of the worked example
    monkeypatch.setattr(oadamw, "adamw_update", _coupled_l2)
    st = new_state(GOLD["theta0"], "f64", "f32")
    grp = dict(lr=GOLD["lr"], beta1=GOLD["beta1"], beta2=GOLD["beta2"],
               eps=GOLD["eps"], weight_decay=GOLD["weight_decay"])
    oadamw.oracle_step([st], [grp], [np.array(GOLD["grad"])])
    assert not np.allclose(st.m, GOLD["m1"], rtol=1e-6)


@pytest.mark.parametrize("mutation", ["old_m", "t_minus_1", "eps_inside"])
def test_other_planted_mistakes_fail_closed_forms(mutation):
    def bad(theta, g, m, v, t, lr, beta1, beta2, eps, weight_decay):
        m_new = beta1 * m + (1.0 - beta1) * g
        v_new = beta2 * v + (1.0 - beta2) * g * g
        tt = t - 1 if mutation == "t_minus_1" else t
        mm = m if mutation == "old_m" else m_new
        with np.errstate(divide="ignore", invalid="ignore"):
            m_hat = mm / (1.0 - beta1 ** max(tt, 1)) if tt else mm
            v_hat = v_new / (1.0 - beta2 ** max(tt, 1)) if tt else v_new
        den = np.sqrt(v_hat + eps) if mutation == "eps_inside" else np.sqrt(v_hat) + eps
        return theta * (1 - lr * weight_decay) - lr * m_hat / den, m_new, v_new

    rng = np.random.default_rng(12)
    n, T = 6, 7
    lr, b1, b2, eps, wd = 0.01, 0.85, 0.99, 1e-6, 0.05
    theta0 = rng.normal(0, 0.1, n)
    gs = [rng.normal(0, 1e-2, n) for _ in range(T)]
    theta, m, v = theta0.copy(), np.zeros(n), np.zeros(n)
    for t in range(1, T + 1):
        theta, m, v = bad(theta, gs[t - 1], m, v, t, lr, b1, b2, eps, wd)
    ref = _exact_reference(theta0, gs, lr, b1, b2, eps, wd)
    with pytest.raises(AssertionError):
        np.testing.assert_allclose(theta, ref[:, 2], rtol=1e-9)
