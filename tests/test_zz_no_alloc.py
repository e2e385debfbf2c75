"""The step entry point that allocates nothing (adamw_step_noalloc).

Some callers cannot call cudaMalloc: an allocator or memory pool that runs the
optimizer step from its own callbacks must not re-enter the device allocator,
and a runtime that hands all device memory to its own pool at start-up has
none left for a plan. adamw_step_noalloc keeps its scratch in a fixed-size
device array instead. Through the C ABI, this checks that it gives the same
results as a plan's adamw_step on the same inputs, on two calls in a row; that
it rejects sizes beyond its fixed scratch without touching the device (every
pointer handed to it is a real device buffer, so a validation slip could not
launch on made-up addresses); that a bounded wait that runs out inside it is
reported through adamw_noalloc_error; and that it refuses a stream that is
being captured.

Collected last on purpose, so a run that stops at the first failure has run
every other test first.
"""
import ctypes

import numpy as np
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


def _buffers(wl, kind):
    sdt = {"f32": torch.float32, "bf16": torch.bfloat16, "int8": torch.int8}[kind]
    params = [workloads.init_param(wl, i).reshape(-1).cuda() for i in range(len(wl.tensors))]
    grads = [torch.zeros_like(p) for p in params]
    m = [torch.zeros(p.numel(), dtype=sdt, device="cuda") for p in params]
    v = [torch.zeros(p.numel(), dtype=sdt, device="cuda") for p in params]
    nb = [max(1, -(-p.numel() // 256)) for p in params]
    ms = [torch.zeros(n, device="cuda") if kind == "int8" else None for n in nb]
    vs = [torch.zeros(n, device="cuda") if kind == "int8" else None for n in nb]
    step = torch.zeros(len(params), dtype=torch.int32, device="cuda")
    return params, grads, m, v, ms, vs, step


def _groups(wl):
    return [dict(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                 weight_decay=g.weight_decay) for g in wl.groups]


def _descs(cs, X, grp_of):
    return [cs.tensor_desc(p, g, m, v, a, b, group=k)
            for p, g, m, v, a, b, k in zip(*X[:6], grp_of)]


@pytest.mark.parametrize("kind", ["f32", "bf16", "int8"])
def test_noalloc_step_matches_plan_step_on_two_calls(kind):
    import compact_state_gb300 as cs
    wl = workloads.mixed([1, 300, 70001, 40000, 0], param_dtype="bf16" if kind == "int8" else "f32",
                         groups=2, steps=2)
    groups = _groups(wl)
    grp_of = [t.group for t in wl.tensors]
    A = _buffers(wl, kind)      # stepped through a plan
    B = _buffers(wl, kind)      # stepped through the entry point that allocates nothing
    plan = cs.adamw_plan_create(_descs(cs, A, grp_of), kind)
    inv = torch.tensor([1.0 / 1024.0], device="cuda")
    fi = torch.zeros(1, device="cuda")
    presents = [None, [True, False, True, True, True]]
    for call in range(2):
        for i in range(len(wl.tensors)):
            g = workloads.grad(wl, i, call + 1).reshape(-1).cuda() * 1024.0
            A[1][i].copy_(g)
            B[1][i].copy_(g)
        cs.adamw_step(plan, groups, presents[call], A[6], inv, fi)
        cs.adamw_step_noalloc(_descs(cs, B, grp_of), kind, groups, presents[call], B[6], inv, fi)
        torch.cuda.synchronize()
        for i in range(len(wl.tensors)):
            assert _bits_equal(A[0][i], B[0][i]), f"call {call}: theta {i}"
            assert _bits_equal(A[2][i], B[2][i]) and _bits_equal(A[3][i], B[3][i]), f"m/v {i}"
            if kind == "int8":
                assert _bits_equal(A[4][i], B[4][i]) and _bits_equal(A[5][i], B[5][i])
        assert torch.equal(A[6], B[6])
    assert B[6].cpu().tolist() == [2, 1, 2, 2, 2]
    assert cs.adamw_noalloc_error() == 0
    cs.adamw_plan_destroy(plan)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import compact_state_gb300 as cs
    L = cs.lib()
    grp = cs.adamw_group_t(1e-3, 0.9, 0.999, 1e-8, 0.0)
    g = (cs.adamw_group_t * 1)(grp)
    # real device buffers, shared by every descriptor below: if validation ever
    # let a call through, its kernel would still stay inside them
    n_unit = cs.CS_NOALLOC_UNIT
    per = 17 * n_unit                       # 17 work units per tensor
    p = torch.zeros(per, device="cuda")
    gr = torch.zeros(per, device="cuda")
    m = torch.zeros(per, device="cuda")
    v = torch.zeros(per, device="cuda")
    before = [x.clone() for x in (p, m, v)]

    def desc(numel):
        return cs.tensor_desc(p, gr, m, v, numel=numel, param_dtype="f32")

    nt = cs.CS_NOALLOC_MAX_TENSORS + 1
    step = torch.zeros(nt, dtype=torch.int32, device="cuda")
    many = (cs.adamw_tensor_t * nt)(*[desc(16)] * nt)
    assert L.adamw_step_noalloc(many, nt, 0, g, 1, None, step.data_ptr(), None, None,
                                None) == cs._binding.CS_ERR_LIMIT
    # 4096 tensors of 17 units each: 69,632 units, more than the scratch holds
    nt = cs.CS_NOALLOC_MAX_TENSORS
    assert nt * 17 > cs.CS_NOALLOC_MAX_UNITS
    wide = (cs.adamw_tensor_t * nt)(*[desc(per)] * nt)
    assert L.adamw_step_noalloc(wide, nt, 0, g, 1, None, step.data_ptr(), None, None,
                                None) == cs._binding.CS_ERR_LIMIT
    # more groups than a step takes
    g65 = (cs.adamw_group_t * 65)(*[grp] * 65)
    one = (cs.adamw_tensor_t * 1)(desc(16))
    assert L.adamw_step_noalloc(one, 1, 0, g65, 65, None, step.data_ptr(), None, None,
                                None) == cs._binding.CS_ERR_LIMIT
    torch.cuda.synchronize()
    assert int(step.abs().sum()) == 0
    for a, b in zip((p, m, v), before):
        assert torch.equal(a, b), "a rejected call touched a buffer"


@pytest.mark.parametrize("kind", ["f32", "int8"])
def test_noalloc_wait_that_runs_out_is_reported(kind):
    """The test hook leaves the first tile unsignalled, so the bounded waits of
    the CTA holding it run out: adamw_noalloc_error reports it once, and the
    next normal call runs clean and equals a plan's step."""
    import compact_state_gb300 as cs
    wl = workloads.mixed([70001, 300000, 5], param_dtype="f32", steps=1)
    groups = _groups(wl)
    grp_of = [t.group for t in wl.tensors]
    X = _buffers(wl, kind)
    for i in range(len(wl.tensors)):
        X[1][i].copy_(workloads.grad(wl, i, 1).reshape(-1).cuda())
    assert cs.adamw_noalloc_error() == 0
    cs.adamw_noalloc_set_debug(wait_ns=50_000_000, flags=1)
    try:
        cs.adamw_step_noalloc(_descs(cs, X, grp_of), kind, groups, None, X[6])
        torch.cuda.synchronize()
    finally:
        cs.adamw_noalloc_set_debug(0, 0)
    err = cs.adamw_noalloc_error()
    assert err & 1, f"compute warps should report the wait that ran out (got {err})"
    assert cs.adamw_noalloc_error() == 0, "reading clears the error word"
    # a clean call afterwards equals a plan's step on fresh buffers
    A, B = _buffers(wl, kind), _buffers(wl, kind)
    for i in range(len(wl.tensors)):
        A[1][i].copy_(X[1][i])
        B[1][i].copy_(X[1][i])
    plan = cs.adamw_plan_create(_descs(cs, A, grp_of), kind)
    cs.adamw_step(plan, groups, None, A[6])
    cs.adamw_step_noalloc(_descs(cs, B, grp_of), kind, groups, None, B[6])
    torch.cuda.synchronize()
    assert cs.adamw_noalloc_error() == 0
    for i in range(len(wl.tensors)):
        assert _bits_equal(A[0][i], B[0][i]) and _bits_equal(A[2][i], B[2][i])
        assert _bits_equal(A[3][i], B[3][i])
    assert torch.equal(A[6], B[6])
    cs.adamw_plan_destroy(plan)


def test_noalloc_refuses_a_capturing_stream():
    import compact_state_gb300 as cs
    wl = workloads.mixed([1000], steps=1)
    X = _buffers(wl, "f32")
    descs = _descs(cs, X, [0])
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    cs.adamw_step_noalloc(descs, "f32", _groups(wl), None, X[6], stream=s)   # set-up first
    torch.cuda.synchronize()
    before = X[0][0].clone()
    with pytest.raises(cs.CompactStateError) as e:
        with torch.cuda.graph(g, stream=s):
            cs.adamw_step_noalloc(descs, "f32", _groups(wl), None, X[6], stream=s)
    assert e.value.code == cs._binding.CS_ERR_INVALID_ARGUMENT
    torch.cuda.synchronize()
    assert torch.equal(before, X[0][0])
