"""GPU parity: the CUDA step through the C ABI against the CPU oracle.

Small cases (whole tensors, several work units per tensor, ragged tails) for
every param dtype x state kind, free-running and oracle-forced; the page's
worked example; the step contract (grad=None, found_inf, step counts); the
scalar path for misaligned buffers; unit-size and graph-capture invariance.
Full-size workloads are in test_parity_full_gpu.py.
"""
import numpy as np
import pytest
import torch

import workloads
from tests.conftest import load_golden
from tests.parity_harness import Harness, _bits_equal, check_bars

pytestmark = pytest.mark.gpu

KINDS = ["f32", "bf16", "int8"]
DTYPES = ["f32", "bf16", "f16"]
RAGGED = [1, 3, 4, 5, 255, 256, 257, 1000, 4099, 70001]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compact_state_gb300 import build
    build.build()


def test_worked_example_on_gpu():
    gold = load_golden("worked_example.txt")
    wl = workloads.tiny("f32")
    h = Harness(wl, "f32")
    res = h.run(steps=1)
    th = h.params[0].double().cpu().numpy()
    half = 0.5 * 10.0 ** -gold["theta1_approx_decimals"]
    assert np.all(np.abs(th - np.array(gold["theta1_approx"])) <= half)
    # the GPU takes hyper-parameters as fp32: 1-fp32(0.9) and 1-fp32(0.999) differ
    # from 0.1 and 0.001 by 2.4e-7 and 1.3e-5 relative, which bounds m1 and v1
    np.testing.assert_allclose(h.state.m[0].double().cpu().numpy(), gold["m1"], rtol=1e-6)
    np.testing.assert_allclose(h.state.v[0].double().cpu().numpy(), gold["v1"], rtol=2e-5)
    check_bars(res, "f32", "f32", forced=False)


@pytest.mark.parametrize("dtype", DTYPES)
def test_tiny_free_run_fp32_state(dtype, record_property):
    wl = workloads.tiny(dtype)
    h = Harness(wl, "f32")
    res = h.run()
    if dtype == "f32":
        check_bars(res, "f32", "f32", forced=False)
    else:
        # 16-bit params drift by rounding in a free run: reported. m and v do
        # not depend on theta, and each step's 16-bit rounding can add at most
        # one ulp of distance, so K steps stay within K ulps.
        record_property("theta16_drift", res.free["theta16_excess"])
        assert res.free["theta16_excess"] <= wl.steps, res.free
        assert res.free["m_excess"] <= 1 and res.free["v_excess"] <= 1, res.free


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("dtype", DTYPES)
def test_ragged_multi_unit_forced(kind, dtype):
    wl = workloads.mixed(RAGGED, param_dtype=dtype, groups=3, steps=6,
                         none_fraction=0.2, found_inf_steps=(3,), grad_prescale=1024.0)
    h = Harness(wl, kind, unit_elems=1024)
    res = h.run(forced=True)
    check_bars(res, kind, dtype, forced=True)


@pytest.mark.parametrize("dtype", DTYPES)
def test_ragged_multi_unit_free_run_fp32_state(dtype):
    wl = workloads.mixed(RAGGED, param_dtype=dtype, groups=3, steps=20,
                         none_fraction=0.2, found_inf_steps=(5,), grad_prescale=1024.0)
    h = Harness(wl, "f32", unit_elems=256)
    res = h.run()
    if dtype == "f32":
        check_bars(res, "f32", "f32", forced=False)
    else:
        assert res.free["m_excess"] <= 1 and res.free["v_excess"] <= 1, res.free


@pytest.mark.parametrize("kind", ["f32", "bf16", "int8", "int8uv", "dyn8"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_packed_small_units(kind, dtype):
    """Hundreds of small tensors (1 to 1536 elements, most not a multiple of
    16, so with a direct remainder; for the 8-bit kinds most end in a ragged
    block) share stages several at a time, between larger tensors that take
    stages of their own; groups, absent gradients and a skipped step as in the
    ragged cases. (The codebook kind packs with 16-bit params only.)"""
    rng = np.random.default_rng(5)
    sizes = [int(n) for n in rng.integers(1, 1537, 300)]
    sizes += [1, 15, 16, 17, 1535, 1536, 1537, 3072, 50000, 9]
    wl = workloads.mixed(sizes, param_dtype=dtype, groups=3, steps=4, none_fraction=0.2,
                         found_inf_steps=(2,), grad_prescale=1024.0)
    h = Harness(wl, kind)
    forced = kind != "f32" or dtype != "f32"
    res = h.run(forced=forced)
    check_bars(res, kind, dtype, forced=forced)


@pytest.mark.parametrize("kind", KINDS)
def test_misaligned_buffers_use_scalar_path(kind):
    wl = workloads.mixed([5, 300, 2049], param_dtype="bf16", groups=2, steps=4,
                         none_fraction=0.0)
    h = Harness(wl, kind, misalign=True)
    res = h.run(forced=True)
    check_bars(res, kind, "bf16", forced=True)


@pytest.mark.parametrize("kind", KINDS)
def test_zero_grad_blocks_and_zero_init(kind):
    wl = workloads.lora(layers=1, steps=5)
    h = Harness(wl, kind)
    res = h.run(forced=(kind != "f32"))
    check_bars(res, kind, "f32", forced=(kind != "f32"))
    if kind == "int8":
        for i in range(len(wl.tensors)):
            zb = wl.zero_blocks(i)
            ms = h.state.m_scale[i].cpu().numpy()
            assert np.all(ms[zb] == 0), "zero-grad blocks keep scale 0"


def test_found_inf_step_is_bit_exact_noop_with_poisoned_grads():
    wl = workloads.mixed([7, 300, 5000], param_dtype="f32", groups=2, steps=4,
                         found_inf_steps=(2, 3), grad_prescale=1024.0)
    for kind in KINDS:
        h = Harness(wl, kind, unit_elems=256)
        h.run(forced=(kind != "f32"))       # snapshots compared inside
        assert h.state.step.cpu().tolist()[:3] == [2, 2, 2]


def test_none_tensors_and_step_counts():
    sizes = [1, 17, 256, 3000, 70000]
    wl = workloads.mixed(sizes, steps=15, none_fraction=0.4, found_inf_steps=(4, 9))
    h = Harness(wl, "f32", unit_elems=256)
    h.run()
    expect = np.zeros(len(sizes), dtype=int)
    for s in range(1, 16):
        if not wl.found_inf(s):
            expect += wl.present(s).astype(int)
    assert h.state.step.cpu().numpy()[:len(sizes)].tolist() == expect.tolist()


def test_empty_and_zero_numel_tensors():
    from compact_state_gb300 import adamw_plan_info
    wl = workloads.mixed([0, 5, 0, 300], steps=3)
    h = Harness(wl, "f32")
    res = h.run()
    check_bars(res, "f32", "f32", forced=False)
    assert adamw_plan_info(h.state.plan)["n_units"] == 4
    only_empty = workloads.mixed([0, 0], steps=2)
    h2 = Harness(only_empty, "int8")
    h2.run()                       # nothing to touch, but the steps are counted
    assert h2.state.step.cpu().tolist()[:2] == [2, 2]


def _run_gpu_only(wl, kind, unit, steps, inv=None, prescale=1.0):
    from compact_state_gb300.torch_adapter import AdamWState
    ps = [workloads.init_param(wl, i).reshape(-1).cuda() for i in range(len(wl.tensors))]
    gs = [torch.empty_like(p) for p in ps]
    st = AdamWState(ps, gs, kind, [t.group for t in wl.tensors], unit)
    groups = [dict(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                   weight_decay=g.weight_decay) for g in wl.groups]
    inv_t = None if inv is None else torch.tensor([inv], dtype=torch.float32, device="cuda")
    for s in range(1, steps + 1):
        for i, g in enumerate(gs):
            g.copy_(workloads.grad(wl, i, s).reshape(-1).cuda() * prescale)
        st.run(groups, None, inv_t, None)
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("kind", KINDS)
def test_unit_size_does_not_change_results(kind):
    wl = workloads.mixed([3, 1000, 40000, 70001], param_dtype="bf16", steps=4)
    runs = [_run_gpu_only(wl, kind, u, 4) for u in (256, 4096, 32768, 1 << 20)]
    for st in runs[1:]:
        for i in range(4):
            assert _bits_equal(st.params[i], runs[0].params[i])
            assert _bits_equal(st.m[i], runs[0].m[i]) and _bits_equal(st.v[i], runs[0].v[i])


@pytest.mark.parametrize("kind", KINDS)
def test_power_of_two_unscale_bit_identical(kind):
    wl = workloads.mixed([1000, 5000], steps=3)
    a = _run_gpu_only(wl, kind, 0, 3)
    b = _run_gpu_only(wl, kind, 0, 3, inv=1.0 / 1024.0, prescale=1024.0)
    for i in range(2):
        assert _bits_equal(a.params[i], b.params[i])
        assert _bits_equal(a.m[i], b.m[i]) and _bits_equal(a.v[i], b.v[i])


def test_set_grads_swaps_gradient_buffers():
    from compact_state_gb300.torch_adapter import AdamWState
    wl = workloads.mixed([100, 3000], steps=3)
    ref = _run_gpu_only(wl, "f32", 0, 3)
    ps = [workloads.init_param(wl, i).reshape(-1).cuda() for i in range(2)]
    gs = [torch.empty_like(p) for p in ps]
    st = AdamWState(ps, gs, "f32", [t.group for t in wl.tensors])
    groups = [dict(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                   weight_decay=g.weight_decay) for g in wl.groups]
    for s in range(1, 4):
        fresh = [workloads.grad(wl, i, s).reshape(-1).cuda() for i in range(2)]
        st.set_grads(fresh)
        st.run(groups)
    torch.cuda.synchronize()
    for i in range(2):
        assert _bits_equal(st.params[i], ref.params[i])


def test_graph_capture_replays_like_direct_calls():
    from compact_state_gb300.torch_adapter import AdamWState
    wl = workloads.mixed([100, 3000, 70001], steps=5)
    ref = _run_gpu_only(wl, "bf16", 0, 5)
    ps = [workloads.init_param(wl, i).reshape(-1).cuda() for i in range(3)]
    gs = [torch.empty_like(p) for p in ps]
    st = AdamWState(ps, gs, "bf16", [t.group for t in wl.tensors])
    groups = [dict(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                   weight_decay=g.weight_decay) for g in wl.groups]
    s_ = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s_):
        with torch.cuda.graph(graph, stream=s_):
            st.run(groups, None, None, None, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert st.step.cpu().tolist()[:3] == [0, 0, 0], "capture must not execute"
    for s in range(1, 6):
        for i, g in enumerate(gs):
            g.copy_(workloads.grad(wl, i, s).reshape(-1).cuda())
        graph.replay()
    torch.cuda.synchronize()
    for i in range(3):
        assert _bits_equal(st.params[i], ref.params[i])
        assert _bits_equal(st.m[i], ref.m[i]) and _bits_equal(st.v[i], ref.v[i])
    assert st.step.cpu().tolist()[:3] == [5, 5, 5]


def test_many_units_commit_exactly_once_per_step():
    wl = workloads.mixed([256 * 3001, 5], steps=1)
    st = _run_gpu_only(wl, "f32", 256, 1)
    groups = [dict(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                   weight_decay=g.weight_decay) for g in wl.groups]
    for _ in range(49):
        st.run(groups)
    torch.cuda.synchronize()
    assert st.step.cpu().tolist()[:2] == [50, 50]


def test_step_rejects_bad_hyperparameters_without_launch():
    from compact_state_gb300 import CompactStateError
    from compact_state_gb300.torch_adapter import AdamWState
    p = torch.zeros(10, device="cuda")
    st = AdamWState([p], [torch.zeros_like(p)], "f32")
    bad = [dict(lr=1e-3, beta1=1.0, beta2=0.999, eps=1e-8, weight_decay=0.0)]
    with pytest.raises(CompactStateError):
        st.run(bad)
    with pytest.raises(CompactStateError):
        st.run([dict(lr=float("nan"), beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)])
    torch.cuda.synchronize()
    assert st.step.cpu().tolist() == [0]
