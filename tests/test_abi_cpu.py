"""Host-side checks of the C ABI that need no GPU.

* the library builds, loads, and exports every function include/compact_state.h
  declares; the binding's constants equal the header's;
* adamw_state_bytes reproduces the oracle's ledger and the pages' figures;
* the work-unit table covers every tensor exactly once;
* invalid plans and steps are rejected with status codes before any CUDA call.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import workloads
from oracle import state_bytes as ostate

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "compact_state.h")


@pytest.fixture(scope="module")
def cs():
    from compact_state_gb300 import build
    build.build()
    import compact_state_gb300 as m
    m.lib()
    return m


def _header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(adamw_\w+)\s*\(", src, re.M)))


def _header_defines():
    out = {}
    for name, val in re.findall(r"#define\s+(CS_\w+)\s+\(?(-?\d+)\)?", open(HEADER).read()):
        out[name] = int(val)
    return out


def test_exports_every_declared_symbol(cs):
    declared = _header_functions()
    assert len(declared) == 16, declared
    assert sorted(cs.EXPORTS) == declared
    L = cs.lib()
    for name in declared:
        assert hasattr(L, name), name
    out = os.popen(f"nm -D {cs.lib()._name}").read()
    for name in declared:
        assert re.search(rf"\bT {name}\b", out), name


def test_constants_match_header(cs):
    import compact_state_gb300._binding as b
    defs = _header_defines()
    assert defs, "no #defines parsed"
    for name, val in defs.items():
        assert getattr(b, name) == val, name


def test_strerror_names_every_code(cs):
    for code in range(0, -9, -1):
        s = cs.adamw_strerror(code)
        assert s and s != "unknown status"
    assert cs.adamw_strerror(-99) == "unknown status"


@pytest.mark.parametrize("kind", ["f32", "bf16", "int8", "int8uv", "dyn8"])
def test_state_bytes_equals_oracle_ledger(cs, kind):
    rng = np.random.default_rng(0)
    numels = [0, 1, 255, 256, 257] + list(rng.integers(1, 10 ** 6, 50))
    assert cs.adamw_state_bytes(numels, kind) == ostate.state_bytes(numels, kind)
    lora = workloads.lora()
    mib = round(cs.adamw_state_bytes(lora.numels, kind) / 2 ** 20, 3)
    assert mib == {"f32": 185.501, "bf16": 92.751}.get(kind, 47.101)


def test_state_bytes_rejects_bad_input(cs):
    with pytest.raises(cs.CompactStateError):
        cs.adamw_state_bytes([5, -1], "f32")
    with pytest.raises(KeyError):
        cs.adamw_state_bytes([5], "f8")
    assert cs.lib().adamw_state_bytes(None, None, 0, 7, ctypes.byref(ctypes.c_int64())) == -2
    assert cs.lib().adamw_state_bytes(None, None, 0, 5, ctypes.byref(ctypes.c_int64())) == -2
    with pytest.raises(cs.CompactStateError):      # fp32 flag outside an 8-bit kind
        cs.adamw_state_bytes([5], "bf16", flags=[1])
    with pytest.raises(cs.CompactStateError):      # unknown flag
        cs.adamw_state_bytes([5], "int8", flags=[2])


@pytest.mark.parametrize("kind", ["int8", "int8uv", "dyn8"])
@pytest.mark.parametrize("threshold", [0, 1, 4096, 65537, 10 ** 9])
def test_selective_state_bytes_equal_oracle_ledger(cs, kind, threshold):
    """With selective fp32 moments the ABI ledger follows the oracle's."""
    numels = workloads.many_small().numels + [0, 1, 255, 256, 257]
    got = cs.adamw_state_bytes(numels, kind, min_8bit_size=threshold)
    assert got == ostate.state_bytes(numels, kind, min_8bit_size=threshold)
    flags = [1 if n < threshold else 0 for n in numels]
    assert cs.adamw_state_bytes(numels, kind, flags=flags) == got


@pytest.mark.parametrize("unit", [256, 1024, 32768])
def test_work_units_tile_every_tensor_once(cs, unit):
    rng = np.random.default_rng(unit)
    numels = [0, 1, 3, unit - 1, unit, unit + 1, 3 * unit + 17] + list(
        rng.integers(1, 20 * unit, 40))
    t, s, ln = cs.adamw_build_units(numels, unit)
    t, s, ln = np.array(t), np.array(s), np.array(ln)
    assert ln.sum() == sum(numels)
    assert np.all(ln <= unit) and np.all(s % unit == 0)
    assert np.all((ln > 0) | (np.array(numels)[t] == 0))
    assert np.all(np.diff(ln) <= 0), "units must be ordered longest first"
    for i, n in enumerate(numels):
        sel = t == i
        order = np.argsort(s[sel])
        ss, ll = s[sel][order], ln[sel][order]
        if n == 0:
            assert sel.sum() == 1 and ln[sel][0] == 0
            continue
        assert ss[0] == 0 and np.all(ss[1:] == ss[:-1] + ll[:-1]) and ss[-1] + ll[-1] == n


def test_work_units_reject_bad_unit_size(cs):
    for bad in (-256, 100, 257):
        with pytest.raises(cs.CompactStateError):
            cs.adamw_build_units([10], bad)


def _desc(cs, **kw):
    base = dict(param=0x10000, grad=0x20000, m=0x30000, v=0x40000, m_scale=0x50000,
                v_scale=0x60000, numel=100, param_dtype=0, group=0)
    base.update(kw)
    return cs.adamw_tensor_t(**base)


@pytest.mark.parametrize("kw,state,code", [
    (dict(param_dtype=5), "f32", -2),
    (dict(numel=-1), "f32", -1),
    (dict(group=-1), "f32", -1),
    (dict(group=64), "f32", -4),
    (dict(param=0), "f32", -1),
    (dict(grad=0x20002), "f32", -3),          # fp32 grad not 4-byte aligned
    (dict(param=0x10001, param_dtype=1), "bf16", -3),
    (dict(m=0x30002), "f32", -3),
    (dict(m_scale=0), "int8", -1),
    (dict(v_scale=0x60002), "int8", -3),
    (dict(master=0x70000), "f32", -1),        # a master needs a 16-bit param
    (dict(master=0x70002, param_dtype=1), "f32", -3),   # master not 4-byte aligned
    (dict(flags=2), "int8", -1),                        # unknown tensor flag
    (dict(flags=1), "f32", -1),                         # fp32 moments outside an 8-bit plan
    (dict(flags=1, m=0x30002), "dyn8", -3),             # fp32 moments need 4-byte alignment
    (dict(m_scale=0), "int8uv", -1),
    (dict(v_scale=0x60002), "dyn8", -3),
])
def test_plan_create_rejects_invalid_tensors(cs, kw, state, code):
    arr = (cs.adamw_tensor_t * 2)(_desc(cs), _desc(cs, **kw))
    out = ctypes.c_void_p(123)
    rc = cs.lib().adamw_plan_create(arr, 2, cs.STATE_CODES[state], 0, ctypes.byref(out))
    assert rc == code and out.value is None


def test_plan_create_rejects_bad_arguments(cs):
    L = cs.lib()
    arr = (cs.adamw_tensor_t * 1)(_desc(cs))
    out = ctypes.c_void_p()
    assert L.adamw_plan_create(None, 1, 0, 0, ctypes.byref(out)) == -1
    assert L.adamw_plan_create(arr, 0, 0, 0, ctypes.byref(out)) == -1
    assert L.adamw_plan_create(arr, 1, 5, 0, ctypes.byref(out)) == -2
    assert L.adamw_plan_create(arr, 1, 0, 100, ctypes.byref(out)) == -1
    assert L.adamw_plan_create(arr, 1, 0, 0, None) == -1
    assert L.adamw_plan_create(arr, 245761, 0, 0, ctypes.byref(out)) == -4


def test_step_rejects_null_plan(cs):
    g = (cs.adamw_group_t * 1)(cs.adamw_group_t(1e-3, 0.9, 0.999, 1e-8, 0.0))
    assert cs.lib().adamw_step(None, g, 1, None, 0x1000, None, None, None) == -1
    assert cs.lib().adamw_plan_info(None, None) == -1
    assert cs.lib().adamw_plan_error(None, None) == -1
    assert cs.lib().adamw_plan_set_debug(None, 0, 0) == -1
    assert cs.lib().adamw_grad_prologue(None, None, None, 1.0, 0x10, None, 0x20, None) == -1
    assert cs.lib().adamw_plan_destroy(None) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_plan_without_gpu_reports_cuda_error(cs):
    arr = (cs.adamw_tensor_t * 1)(_desc(cs))
    out = ctypes.c_void_p()
    assert cs.lib().adamw_plan_create(arr, 1, 0, 0, ctypes.byref(out)) == -5
    assert out.value is None


def test_tensor_struct_layout_matches_header(cs):
    # the C struct: six pointers, int64 numel, two int32, then the master pointer
    assert ctypes.sizeof(cs.adamw_tensor_t) == 80
    assert cs.adamw_tensor_t.master.offset == 64
    assert cs.adamw_tensor_t.flags.offset == 72


def test_selective_fp32_tensor_needs_no_scales(cs):
    # an fp32-moment tensor in an 8-bit plan validates without scale arrays
    # (then fails only for want of a GPU here)
    arr = (cs.adamw_tensor_t * 1)(_desc(cs, m_scale=0, v_scale=0, flags=1))
    out = ctypes.c_void_p()
    rc = cs.lib().adamw_plan_create(arr, 1, cs.STATE_CODES["dyn8"], 0, ctypes.byref(out))
    assert rc in (0, -5)
    if rc == 0:
        cs.adamw_plan_destroy(cs.Plan(out.value, 1))


def _check_cover(numels, t, s, ln):
    t, s, ln = np.array(t), np.array(s), np.array(ln)
    for i, n in enumerate(numels):
        sel = t == i
        order = np.argsort(s[sel])
        ss, ll = s[sel][order], ln[sel][order]
        if n == 0:
            assert sel.sum() == 1 and ll[0] == 0
            continue
        assert ss[0] == 0 and np.all(ss[1:] == ss[:-1] + ll[:-1]) and ss[-1] + ll[-1] == n
    return t, s, ln


@pytest.mark.parametrize("kind,tile", [("f32", 3072), ("bf16", 3072), ("int8", 4096),
                                       ("dyn8", 4096)])
@pytest.mark.parametrize("wl", ["lora", "few_large", "many_small", "mixed"])
def test_plan_queue_recuts_the_last_two_waves(cs, kind, tile, wl):
    """The plan's queue: every tensor covered once, longest first, starts on
    256-element blocks; it is the plain cut up to a point, after which every
    unit is at most four tiles long, and that re-cut region holds the last
    two waves' worth of elements (at most one unit more)."""
    if wl == "mixed":
        numels = [0, 1, 255, 5000, 49152, 49153, 200000, 1 << 20]
    else:
        numels = getattr(workloads, wl)().numels
    ctas, unit = 152, 49152
    piece = min(unit, 4 * tile)
    t, s, ln = _check_cover(numels, *cs.adamw_build_queue(numels, kind, ctas))
    assert np.all(np.diff(ln) <= 0) and np.all(s % 256 == 0)
    # the queue is the plain cut up to some position p, then re-cut pieces
    bt, bs, bl = (np.array(x) for x in cs.adamw_build_units(numels))
    n = min(len(ln), len(bl))
    diff = np.flatnonzero((t[:n] != bt[:n]) | (s[:n] != bs[:n]) | (ln[:n] != bl[:n]))
    p = int(diff[0]) if diff.size else n
    assert np.all(ln[p:] <= piece)
    region, total, waves = int(ln[p:].sum()), int(ln.sum()), 2 * ctas * unit
    assert region >= min(total, waves) or np.all(bl[p:] <= piece)
    assert region <= waves + unit
    # the last two waves' worth of elements hold no unit longer than a piece,
    # and, for the 8-bit kinds, the last ctas pieces' worth none longer than
    # two tiles
    suffix = np.cumsum(ln[::-1])[::-1]
    assert np.all(ln[suffix <= waves] <= piece)
    if kind in ("int8", "dyn8"):
        assert np.all(ln[suffix <= ctas * piece] <= 2 * tile)


def test_plan_queue_small_plan_is_all_pieces(cs):
    numels = [3 * 49152 + 7, 100]
    t, s, ln = _check_cover(numels, *cs.adamw_build_queue(numels, "int8", 152))
    assert ln.max() <= 2 * 4096
    with pytest.raises(cs.CompactStateError):
        cs.adamw_build_queue(numels, "int8", 0)
    with pytest.raises(KeyError):
        cs.adamw_build_queue(numels, "f8", 152)


def test_descriptors_reject_strided_and_host_tensors(cs):
    t = torch.zeros(8, 8)
    with pytest.raises(ValueError, match="contiguous"):
        cs.tensor_desc(t[:, 0], 0x20000, 0x30000, 0x40000, numel=8, param_dtype="f32")
    with pytest.raises(ValueError, match="CUDA"):
        cs.tensor_desc(t.reshape(-1), 0x20000, 0x30000, 0x40000, numel=64, param_dtype="f32")


@pytest.mark.parametrize("bad", [
    dict(eps=0.0), dict(eps=-1e-8), dict(eps=float("nan")), dict(beta1=1.0),
    dict(beta2=-0.1), dict(lr=float("inf")), dict(weight_decay=float("nan")),
])
def test_step_rejects_bad_hyperparameters_before_any_cuda_call(cs, bad):
    """Group validation comes first: eps must be positive (it keeps
    sqrt(v_hat) + eps away from zero), betas in [0, 1), everything finite.
    The no-allocation entry point checks groups before touching a device, so
    this runs without a GPU."""
    g = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    g.update(bad)
    ga = (cs.adamw_group_t * 1)(cs.adamw_group_t(g["lr"], g["beta1"], g["beta2"], g["eps"],
                                                 g["weight_decay"]))
    arr = (cs.adamw_tensor_t * 1)(_desc(cs))
    rc = cs.lib().adamw_step_noalloc(arr, 1, 0, ga, 1, None, 0x1000, None, None, None)
    assert rc == cs._binding.CS_ERR_HYPERPARAM


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_tiny_positive_eps_passes_validation(cs):
    ga = (cs.adamw_group_t * 1)(cs.adamw_group_t(1e-3, 0.9, 0.999, 1e-30, 0.0))
    arr = (cs.adamw_tensor_t * 1)(_desc(cs))
    rc = cs.lib().adamw_step_noalloc(arr, 1, 0, ga, 1, None, 0x1000, None, None, None)
    assert rc == cs._binding.CS_ERR_CUDA      # past validation, then no device here


def test_noalloc_readback_without_gpu_reports_cuda_error(cs):
    if torch.cuda.is_available():
        pytest.skip("checks the no-GPU path")
    out = ctypes.c_uint32(7)
    assert cs.lib().adamw_noalloc_error(None) == -1
    assert cs.lib().adamw_noalloc_error(ctypes.byref(out)) == -5
    assert cs.lib().adamw_noalloc_set_debug(0, 2) == -1
    assert cs.lib().adamw_noalloc_set_debug(61 * 10 ** 9, 0) == -1
    assert cs.lib().adamw_noalloc_set_debug(0, 0) == 0
