"""Pins of the oracle's gradient prologue (unscale, non-finite check, clip).

Closed forms and hand values, none re-typing the oracle's own formula:
a constant gradient c over n elements has norm |c|*sqrt(n); gradients [3, 4]
have norm 5; the clip coefficient of the usual global-norm rule is
max_norm/(norm + 1e-6) below the threshold and 1 above it; a planted inf or
NaN anywhere in a present gradient sets found_inf, in an absent one it does not.
"""
import math

import numpy as np
import pytest

from oracle.prologue import grad_prologue


def test_constant_gradient_norm():
    for n, c in [(1, 3.0), (1000, -0.25), (257, 1e-3)]:
        fi, norm, scale = grad_prologue([np.full(n, c)], 1.0, 0.0)
        assert fi == 0.0 and scale == 1.0
        assert norm == pytest.approx(abs(c) * math.sqrt(n), rel=1e-14)


def test_pythagorean_norm_and_clip_coefficient():
    fi, norm, scale = grad_prologue([np.array([3.0]), np.array([4.0])], 1.0, 1.0)
    assert norm == 5.0
    assert scale == pytest.approx(1.0 / (5.0 + 1e-6), rel=1e-15)
    # below the threshold: no clipping
    fi, norm, scale = grad_prologue([np.array([3.0, 4.0])], 1.0, 10.0)
    assert scale == 1.0


def test_unscale_applies_before_norm_and_clip():
    g = np.array([3.0, 4.0]) * 1024.0
    fi, norm, scale = grad_prologue([g], 1.0 / 1024.0, 2.5)
    assert norm == 5.0
    assert scale == pytest.approx((1.0 / 1024.0) * 2.5 / (5.0 + 1e-6), rel=1e-15)


def test_nonfinite_sets_found_inf_only_in_present_grads():
    g = np.ones(10)
    for bad in (np.inf, -np.inf, np.nan):
        h = g.copy()
        h[7] = bad
        fi, _, scale = grad_prologue([g, h], 0.5, 1.0)
        assert fi == 1.0 and scale == 0.5
        fi, norm, _ = grad_prologue([g, None], 0.5, 1.0)
        assert fi == 0.0 and norm == pytest.approx(math.sqrt(10) * 0.5)


def test_overflow_after_unscale_counts_as_nonfinite():
    # 3e38 is a finite fp32 value; unscaled by 4 it overflows fp32, where the
    # flag is decided
    fi, _, _ = grad_prologue([np.array([3e38], dtype=np.float32)], 4.0, 0.0)
    assert fi == 1.0
    fi, _, _ = grad_prologue([np.array([3e38], dtype=np.float32)], 1.0, 0.0)
    assert fi == 0.0
