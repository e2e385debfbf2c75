"""The step entry point that allocates nothing (adamw_step_noalloc).

Some callers cannot call cudaMalloc: an allocator or memory pool that runs the
optimizer step from its own callbacks must not re-enter the device allocator,
and a runtime that hands all device memory to its own pool at start-up has
none left for a plan. adamw_step_noalloc keeps its scratch in a fixed-size
device array instead. Through the C ABI, this checks that it gives the same
results as a plan's adamw_step on the same inputs, on two calls in a row, and
that it rejects sizes beyond its fixed scratch without touching the device.

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


@pytest.mark.parametrize("kind", ["f32", "bf16", "int8"])
def test_noalloc_step_matches_plan_step_on_two_calls(kind):
    import compact_state_gb300 as cs
    wl = workloads.mixed([1, 300, 70001, 40000, 0], param_dtype="bf16" if kind == "int8" else "f32",
                         groups=2, steps=2)
    groups = [dict(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                   weight_decay=g.weight_decay) for g in wl.groups]
    grp_of = [t.group for t in wl.tensors]
    A = _buffers(wl, kind)      # stepped through a plan
    B = _buffers(wl, kind)      # stepped through the entry point that allocates nothing
    descs = lambda X: [cs.tensor_desc(p, g, m, v, a, b, group=k)
                       for p, g, m, v, a, b, k in zip(*X[:6], grp_of)]
    plan = cs.adamw_plan_create(descs(A), kind)
    inv = torch.tensor([1.0 / 1024.0], device="cuda")
    fi = torch.zeros(1, device="cuda")
    presents = [None, [True, False, True, True, True]]
    for call in range(2):
        for i in range(len(wl.tensors)):
            g = workloads.grad(wl, i, call + 1).reshape(-1).cuda() * 1024.0
            A[1][i].copy_(g)
            B[1][i].copy_(g)
        cs.adamw_step(plan, groups, presents[call], A[6], inv, fi)
        cs.adamw_step_noalloc(descs(B), kind, groups, presents[call], B[6], inv, fi)
        torch.cuda.synchronize()
        for i in range(len(wl.tensors)):
            assert _bits_equal(A[0][i], B[0][i]), f"call {call}: theta {i}"
            assert _bits_equal(A[2][i], B[2][i]) and _bits_equal(A[3][i], B[3][i]), f"m/v {i}"
            if kind == "int8":
                assert _bits_equal(A[4][i], B[4][i]) and _bits_equal(A[5][i], B[5][i])
        assert torch.equal(A[6], B[6])
    assert B[6].cpu().tolist() == [2, 1, 2, 2, 2]
    cs.adamw_plan_destroy(plan)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import compact_state_gb300 as cs
    L = cs.lib()
    g = (cs.adamw_group_t * 1)(cs.adamw_group_t(1e-3, 0.9, 0.999, 1e-8, 0.0))
    fake = dict(param=0x10000, grad=0x20000, m=0x30000, v=0x40000, m_scale=0x50000,
                v_scale=0x60000, param_dtype=0, group=0)
    many = (cs.adamw_tensor_t * (cs.CS_NOALLOC_MAX_TENSORS + 1))(
        *[cs.adamw_tensor_t(numel=16, **fake)] * (cs.CS_NOALLOC_MAX_TENSORS + 1))
    rc = L.adamw_step_noalloc(many, cs.CS_NOALLOC_MAX_TENSORS + 1, 0, g, 1, None, 0x1000,
                              None, None, None)
    assert rc == cs._binding.CS_ERR_LIMIT
    huge = (cs.adamw_tensor_t * 1)(cs.adamw_tensor_t(
        numel=(cs.CS_NOALLOC_MAX_UNITS + 1) * cs.CS_NOALLOC_UNIT, **fake))
    rc = L.adamw_step_noalloc(huge, 1, 0, g, 1, None, 0x1000, None, None, None)
    assert rc == cs._binding.CS_ERR_LIMIT
