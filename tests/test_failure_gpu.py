"""Failure detection on the GPU without a GPU fault.

Every wait inside the step kernel is bounded. A test hook leaves the first
CTA's first tile unsignalled, so its compute warps' wait runs out (a flag that
nothing sets); the kernel must record that in the plan's error word, return,
and leave the context usable: the next normal step runs clean and matches a
plan that never saw the hook.
"""
import pytest
import torch

import workloads
from tests.parity_harness import _bits_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compact_state_gb300 import build
    build.build()


def _state(wl, kind):
    from compact_state_gb300.torch_adapter import AdamWState
    ps = [workloads.init_param(wl, i).reshape(-1).cuda() for i in range(len(wl.tensors))]
    gs = [workloads.grad(wl, i, 1).reshape(-1).cuda() for i in range(len(wl.tensors))]
    return AdamWState(ps, gs, kind, [t.group for t in wl.tensors])


@pytest.mark.parametrize("kind", ["f32", "int8"])
def test_wait_that_runs_out_reports_and_context_survives(kind):
    from compact_state_gb300 import adamw_plan_error, adamw_plan_set_debug
    wl = workloads.mixed([70001, 300000, 5], steps=1)
    groups = [dict(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                   weight_decay=g.weight_decay) for g in wl.groups]
    st = _state(wl, kind)
    assert adamw_plan_error(st.plan) == 0
    adamw_plan_set_debug(st.plan, wait_ns=50_000_000, flags=1)
    st.run(groups)
    torch.cuda.synchronize()
    err = adamw_plan_error(st.plan)
    assert err & 1, f"compute warps should report the wait that ran out (got {err})"
    assert adamw_plan_error(st.plan) == 0, "reading clears the error word"
    # normal steps afterwards: no error, and the same result as a clean plan
    adamw_plan_set_debug(st.plan, 0, 0)
    ref = _state(wl, kind)
    for i in range(3):
        st.params[i].copy_(ref.params[i])
        st.m[i].copy_(ref.m[i])
        st.v[i].copy_(ref.v[i])
        if st.m_scale[i] is not None:
            st.m_scale[i].copy_(ref.m_scale[i])
            st.v_scale[i].copy_(ref.v_scale[i])
    st.step.copy_(ref.step)
    st.run(groups)
    ref.run(groups)
    torch.cuda.synchronize()
    assert adamw_plan_error(st.plan) == 0 and adamw_plan_error(ref.plan) == 0
    for i in range(3):
        assert _bits_equal(st.params[i], ref.params[i])
        assert _bits_equal(st.m[i], ref.m[i]) and _bits_equal(st.v[i], ref.v[i])


def test_set_debug_rejects_unknown_flags():
    from compact_state_gb300 import CompactStateError, adamw_plan_set_debug
    st = _state(workloads.mixed([10], steps=1), "f32")
    with pytest.raises(CompactStateError):
        adamw_plan_set_debug(st.plan, 0, 2)
    with pytest.raises(CompactStateError):
        adamw_plan_set_debug(st.plan, 61 * 10 ** 9, 0)
