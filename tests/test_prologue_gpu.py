"""GPU parity of the gradient prologue (adamw_grad_prologue) and of prologue + step.

The prologue's outputs are compared with the oracle's (found_inf exactly, norm
and clip factor to 1e-6 relative); then the pipeline prologue -> step, where
the step takes the prologue's found_inf and scale, is compared with the
oracle's prologue -> oracle step over several steps, one of them overflowing.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle.adamw import oracle_step
from oracle.prologue import grad_prologue
from tests.parity_harness import Harness, _bits_equal, check_bars

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compact_state_gb300 import build
    build.build()


def _rel(a, b):
    return abs(a - b) / max(abs(b), 1e-300)


def _oracle_grads(h, s, present):
    gv = h._fill_grads(s)
    return [g if p else None for g, p in zip(gv, present)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("max_norm", [0.0, 1e-3, 1e6])
def test_prologue_matches_oracle(dtype, max_norm):
    wl = workloads.mixed([1, 5, 255, 256, 1000, 4099, 70001, 0], param_dtype=dtype, groups=2,
                         steps=3, none_fraction=0.3, grad_prescale=1024.0)
    h = Harness(wl, "f32", unit_elems=1024)
    for s in range(1, 4):
        present = wl.present(s)
        og = _oracle_grads(h, s, present)
        fo, no, so = h.state.prologue(present, h.inv_scale_t, max_norm)
        torch.cuda.synchronize()
        fi, norm, scale = grad_prologue(og, float(np.float32(wl.inv_scale)), max_norm)
        assert float(fo) == fi == 0.0
        assert _rel(float(no), norm) <= 1e-6, (float(no), norm)
        assert _rel(float(so), scale) <= 1e-6, (float(so), scale)
        if max_norm == 1e-3:
            assert float(so) < float(h.inv_scale_t)   # clipping is active


def test_prologue_flags_nonfinite_only_in_present_grads():
    wl = workloads.mixed([300, 5000, 70001], steps=1)
    h = Harness(wl, "f32")
    h._fill_grads(1)
    for bad in (float("inf"), float("nan")):
        h.grads[1][1234] = bad
        fo, no, so = h.state.prologue(None, None, 1.0)
        torch.cuda.synchronize()
        assert float(fo) == 1.0 and float(so) == 1.0 and np.isnan(float(no))
        fo, no, so = h.state.prologue([True, False, True], None, 1.0)
        torch.cuda.synchronize()
        assert float(fo) == 0.0 and np.isfinite(float(no))
    # an fp32 overflow after unscaling counts, as in the oracle
    h.grads[1][1234] = 3e38
    inv4 = torch.tensor([4.0], device="cuda")
    fo, _, _ = h.state.prologue(None, inv4, 0.0)
    torch.cuda.synchronize()
    assert float(fo) == 1.0


@pytest.mark.parametrize("kind", ["f32", "bf16", "int8"])
def test_prologue_then_step_against_oracle(kind):
    wl = workloads.mixed([3, 300, 5000, 70001], steps=8, none_fraction=0.2, groups=2,
                         found_inf_steps=(4,), grad_prescale=1024.0)
    h = Harness(wl, kind, unit_elems=2048)
    max_norm = 0.05            # the seeded grads have norm ~0.27: clipping is active
    worst = {}
    for s in range(1, wl.steps + 1):
        present = wl.present(s)
        og = _oracle_grads(h, s, present)
        forced = kind != "f32"
        if forced:
            h._upload_oracle_state()
        fo, no, so = h.state.prologue(present, h.inv_scale_t, max_norm)
        h.state.run(h.gpu_groups, None if present.all() else present, so, fo)
        torch.cuda.synchronize()
        fi, norm, scale = grad_prologue(og, float(np.float32(wl.inv_scale)), max_norm)
        assert float(fo) == fi, s
        poisoned_present = any(present[i] for i, _, _ in wl.poison(s))
        assert fi == (1.0 if poisoned_present else 0.0)
        oracle_step(h.ostates, h.gpu_groups, og, inv_scale=float(np.float32(scale)),
                    found_inf=fi)
        assert h.state.step.cpu().tolist()[:4] == [o.step for o in h.ostates]
        if forced:
            h._compare(worst, final=False)
    if kind == "f32":
        h._compare(worst, final=True)
    res = type("R", (), {"free": worst, "forced": worst})()
    check_bars(res, kind, "f32", forced=(kind != "f32"))


def test_prologue_full_size_norm_and_determinism():
    wl = workloads.few_large()
    h = Harness(wl, "f32", sample=16, grad_device="cuda", param_device_init="cuda")
    h._fill_grads(1)
    a = h.state.prologue(None, None, 1.0)
    first = [float(x) for x in a]
    b = h.state.prologue(None, None, 1.0)
    torch.cuda.synchronize()
    assert [float(x) for x in b] == first, "same inputs give the same bits"
    total = sum(float(torch.sum(g.double() ** 2)) for g in h.grads)
    assert _rel(first[1], float(np.sqrt(total))) <= 1e-6
    assert _rel(first[2], 1.0 / (np.sqrt(total) + 1e-6)) <= 1e-6


def test_prologue_and_step_in_one_graph():
    wl = workloads.mixed([100, 3000, 70001], steps=4, grad_prescale=1024.0)
    runs = []
    for use_graph in (False, True):
        h = Harness(wl, "bf16")
        h._fill_grads(1)
        h.state.prologue(None, h.inv_scale_t, 0.01)      # outputs allocated before capture
        torch.cuda.synchronize()
        if use_graph:
            s_ = torch.cuda.Stream()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s_):
                with torch.cuda.graph(graph, stream=s_):
                    cur = torch.cuda.current_stream()
                    fo, no, so = h.state.prologue(None, h.inv_scale_t, 0.01, stream=cur)
                    h.state.run(h.gpu_groups, None, so, fo, stream=cur)
            torch.cuda.synchronize()
        for s in range(1, wl.steps + 1):
            h._fill_grads(s)
            if use_graph:
                graph.replay()
            else:
                fo, no, so = h.state.prologue(None, h.inv_scale_t, 0.01)
                h.state.run(h.gpu_groups, None, so, fo)
        torch.cuda.synchronize()
        runs.append(h)
    for i in range(3):
        assert _bits_equal(runs[0].params[i], runs[1].params[i])
        assert _bits_equal(runs[0].state.m[i], runs[1].state.m[i])
    assert runs[1].state.step.cpu().tolist()[:3] == [4, 4, 4]
