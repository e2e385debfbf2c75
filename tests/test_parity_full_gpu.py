"""GPU parity at the full sizes of the benchmark workloads, on sampled elements.

The step runs over every element of the workload in the same launch shape the
benchmark times; the oracle follows a seeded sample of positions (whole
256-element blocks for int8 state). Inputs are generated on the device by the
seeded generators and gathered at the sampled positions for the oracle.
"""
import numpy as np
import pytest
import torch

import workloads
from tests.parity_harness import Harness, check_bars

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compact_state_gb300 import build
    build.build()


def _free_gb():
    free, _ = torch.cuda.mem_get_info()
    return free / 2 ** 30


def _harness(wl, kind, sample):
    return Harness(wl, kind, sample=sample, grad_device="cuda", param_device_init="cuda")


def test_few_large_fp32_free_run_10_steps():
    wl = workloads.few_large()
    h = _harness(wl, "f32", 4096)
    res = h.run(steps=10)
    check_bars(res, "f32", "f32", forced=False)


@pytest.mark.parametrize("kind", ["bf16", "int8"])
def test_few_large_compact_state_forced(kind):
    wl = workloads.few_large()
    h = _harness(wl, kind, 4096)
    res = h.run(steps=4, forced=True)
    check_bars(res, kind, "f32", forced=True)


def test_many_small_fp32_free_run_20_steps():
    wl = workloads.many_small()
    h = _harness(wl, "f32", 64)
    res = h.run(steps=20)
    check_bars(res, "f32", "f32", forced=False)


@pytest.mark.parametrize("kind", ["bf16", "int8"])
def test_lora_compact_states_forced_250_steps(kind):
    wl = workloads.lora()
    h = _harness(wl, kind, 512)
    res = h.run(steps=250, forced=True)
    check_bars(res, kind, "f32", forced=True)


@pytest.mark.parametrize("kind", ["f32", "int8"])
def test_llama3_8b_forced_3_steps(kind):
    need = 100 if kind == "f32" else 52
    if _free_gb() < need:
        pytest.skip(f"needs {need} GiB free")
    wl = workloads.llama3_8b()
    h = _harness(wl, kind, 2048)
    res = h.run(steps=3, forced=True)
    check_bars(res, kind, "bf16", forced=True)
    del h
    torch.cuda.empty_cache()


def test_tensor_beyond_2_31_elements():
    n = (1 << 31) + 1000 + 3
    if _free_gb() < 20:
        pytest.skip("needs 20 GiB free")
    wl = workloads.mixed([n, 7], param_dtype="bf16", groups=1, steps=2)
    h = _harness(wl, "bf16", 4096)
    res = h.run(steps=2, forced=True)
    check_bars(res, "bf16", "bf16", forced=True)
    del h
    torch.cuda.empty_cache()
