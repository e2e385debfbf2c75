"""ctypes binding of include/compact_state.h: the same entry points, argument
marshalling only. Every step of the optimizer runs in the CUDA library; if the
library is missing this module raises instead of falling back to anything."""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, Optional, Sequence

from . import build as _build

# ---- constants (values of include/compact_state.h) -------------------------
CS_OK = 0
CS_ERR_INVALID_ARGUMENT = -1
CS_ERR_UNSUPPORTED = -2
CS_ERR_MISALIGNED = -3
CS_ERR_LIMIT = -4
CS_ERR_CUDA = -5
CS_ERR_OUT_OF_MEMORY = -6
CS_ERR_HYPERPARAM = -7
CS_ERR_WRONG_DEVICE = -8

CS_DTYPE_F32 = 0
CS_DTYPE_BF16 = 1
CS_DTYPE_F16 = 2
CS_STATE_F32 = 0
CS_STATE_BF16 = 1
CS_STATE_INT8 = 2
CS_STATE_INT8_UV = 3
CS_STATE_DYN8 = 4
CS_TENSOR_STATE_F32 = 1
CS_INT8_BLOCK = 256
CS_MAX_GROUPS = 64
CS_MAX_TENSORS = 245760
CS_NOALLOC_MAX_TENSORS = 4096
CS_NOALLOC_MAX_UNITS = 65536
CS_NOALLOC_UNIT = 49152

DTYPE_CODES = {"f32": CS_DTYPE_F32, "bf16": CS_DTYPE_BF16, "f16": CS_DTYPE_F16}
STATE_CODES = {"f32": CS_STATE_F32, "bf16": CS_STATE_BF16, "int8": CS_STATE_INT8,
               "int8uv": CS_STATE_INT8_UV, "dyn8": CS_STATE_DYN8}
EIGHT_BIT = ("int8", "int8uv", "dyn8")


class adamw_group_t(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
                ("weight_decay", ctypes.c_float)]


class adamw_tensor_t(ctypes.Structure):
    _fields_ = [("param", ctypes.c_void_p), ("grad", ctypes.c_void_p),
                ("m", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("m_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("numel", ctypes.c_int64), ("param_dtype", ctypes.c_int32),
                ("group", ctypes.c_int32), ("master", ctypes.c_void_p),
                ("flags", ctypes.c_int32)]


class adamw_plan_info_t(ctypes.Structure):
    _fields_ = [("n_units", ctypes.c_int64), ("total_numel", ctypes.c_int64),
                ("device_bytes", ctypes.c_int64), ("n_tensors", ctypes.c_int32),
                ("state_kind", ctypes.c_int32), ("unit_elems", ctypes.c_int32),
                ("grid_blocks", ctypes.c_int32), ("block_threads", ctypes.c_int32),
                ("device", ctypes.c_int32)]


class CompactStateError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {adamw_strerror(code)} ({code})")


_LIB = None
EXPORTS = ("adamw_plan_create", "adamw_step", "adamw_plan_set_grads", "adamw_plan_info",
           "adamw_plan_destroy", "adamw_state_bytes", "adamw_build_units", "adamw_strerror",
           "adamw_plan_error", "adamw_plan_set_debug", "adamw_step_noalloc",
           "adamw_grad_prologue", "adamw_build_queue", "adamw_noalloc_error",
           "adamw_noalloc_set_debug", "adamw_shard_ranges")


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m compact_state_gb300.build` (needs nvcc)")
    L = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    L.adamw_plan_create.argtypes = [ctypes.POINTER(adamw_tensor_t), i32, i32, i32,
                                    ctypes.POINTER(vp)]
    L.adamw_step.argtypes = [vp, ctypes.POINTER(adamw_group_t), i32,
                             ctypes.POINTER(ctypes.c_uint32), vp, vp, vp, vp]
    L.adamw_plan_set_grads.argtypes = [vp, ctypes.POINTER(vp), vp]
    L.adamw_plan_info.argtypes = [vp, ctypes.POINTER(adamw_plan_info_t)]
    L.adamw_plan_destroy.argtypes = [vp]
    L.adamw_state_bytes.argtypes = [ctypes.POINTER(i64), ctypes.POINTER(i32), i32, i32,
                                    ctypes.POINTER(i64)]
    L.adamw_build_units.argtypes = [ctypes.POINTER(i64), i32, i32, ctypes.POINTER(i32),
                                    ctypes.POINTER(i64), ctypes.POINTER(i32), i64,
                                    ctypes.POINTER(i64)]
    L.adamw_build_queue.argtypes = [ctypes.POINTER(i64), i32, i32, i32, i32,
                                    ctypes.POINTER(i32), ctypes.POINTER(i64),
                                    ctypes.POINTER(i32), i64, ctypes.POINTER(i64)]
    L.adamw_plan_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    L.adamw_plan_set_debug.argtypes = [vp, ctypes.c_uint64, ctypes.c_uint32]
    L.adamw_step_noalloc.argtypes = [ctypes.POINTER(adamw_tensor_t), i32, i32,
                                     ctypes.POINTER(adamw_group_t), i32,
                                     ctypes.POINTER(ctypes.c_uint32), vp, vp, vp, vp]
    L.adamw_noalloc_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.adamw_shard_ranges.argtypes = [ctypes.POINTER(i64), i32, i32, i32, ctypes.POINTER(i64),
                                     ctypes.POINTER(i64), ctypes.POINTER(i64),
                                     ctypes.POINTER(i64)]
    L.adamw_noalloc_set_debug.argtypes = [ctypes.c_uint64, ctypes.c_uint32]
    L.adamw_grad_prologue.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp, ctypes.c_float,
                                      vp, vp, vp, vp]
    L.adamw_strerror.argtypes = [ctypes.c_int]
    L.adamw_strerror.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name != "adamw_strerror":
            getattr(L, name).restype = ctypes.c_int
    _LIB = L
    return L


def _check(rc: int, where: str) -> None:
    if rc != CS_OK:
        raise CompactStateError(rc, where)


def _ptr(x) -> Optional[int]:
    """Device pointer of a torch tensor, an int address, or None. Tensors must
    be contiguous CUDA tensors: the kernels address them as flat arrays."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("buffers passed to the step must be contiguous")
    if x.device.type != "cuda":
        raise ValueError(f"buffers passed to the step must be CUDA tensors, got {x.device}")
    return int(x.data_ptr())


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


class Plan:
    """Owner of an ``adamw_plan_t*``; ``adamw_plan_destroy`` frees it."""

    def __init__(self, handle: int, n_tensors: int, keepalive=None):
        self.handle = handle
        self.n_tensors = n_tensors
        self._keepalive = keepalive

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        adamw_plan_destroy(self)

    def __del__(self):
        try:
            if self.handle:
                adamw_plan_destroy(self)
        except Exception:
            pass


# ---- entry points ------------------------------------------------------------

def adamw_strerror(code: int) -> str:
    return lib().adamw_strerror(int(code)).decode()


def tensor_desc(param, grad, m, v, m_scale=None, v_scale=None, group: int = 0,
                numel: Optional[int] = None, param_dtype: Optional[str] = None,
                master=None, flags: int = 0) -> adamw_tensor_t:
    """An ``adamw_tensor_t`` from torch tensors (or int addresses + numel/dtype);
    ``master``: optional fp32 master weights of a 16-bit param; ``flags``:
    CS_TENSOR_* bits."""
    if numel is None:
        numel = int(param.numel())
    if param_dtype is None:
        param_dtype = {"torch.float32": "f32", "torch.bfloat16": "bf16",
                       "torch.float16": "f16"}[str(param.dtype)]
    return adamw_tensor_t(_ptr(param), _ptr(grad), _ptr(m), _ptr(v), _ptr(m_scale),
                          _ptr(v_scale), int(numel), DTYPE_CODES[param_dtype], int(group),
                          _ptr(master), int(flags))


def adamw_plan_create(tensors: Sequence[adamw_tensor_t], state_kind="f32",
                      unit_elems: int = 0, keepalive=None) -> Plan:
    sk = STATE_CODES[state_kind] if isinstance(state_kind, str) else int(state_kind)
    arr = (adamw_tensor_t * max(len(tensors), 1))(*tensors)
    out = ctypes.c_void_p()
    rc = lib().adamw_plan_create(arr if tensors else None, len(tensors), sk, int(unit_elems),
                                 ctypes.byref(out))
    _check(rc, "adamw_plan_create")
    return Plan(out.value, len(tensors), keepalive)


def pack_present(present: Optional[Iterable[bool]], n_tensors: int):
    """Bitmask words (ctypes uint32 array) from per-tensor booleans; None -> None."""
    if present is None:
        return None
    words = (ctypes.c_uint32 * ((n_tensors + 31) // 32))()
    for i, p in enumerate(present):
        if p:
            words[i >> 5] |= (1 << (i & 31))
    return words


def groups_array(groups) -> ctypes.Array:
    def one(g):
        if isinstance(g, adamw_group_t):
            return g
        if isinstance(g, dict):
            return adamw_group_t(g["lr"], g["beta1"], g["beta2"], g["eps"], g["weight_decay"])
        if isinstance(g, (tuple, list)):
            return adamw_group_t(*g)
        return adamw_group_t(g.lr, g.beta1, g.beta2, g.eps, g.weight_decay)
    gs = [one(g) for g in groups]
    return (adamw_group_t * max(len(gs), 1))(*gs)


def adamw_step(plan: Plan, groups, grad_present=None, step=None, inv_scale=None,
               found_inf=None, stream=None) -> None:
    """Enqueue one fused AdamW step (asynchronous on ``stream``).

    ``groups``: adamw_group_t array, or a sequence of dicts / tuples / objects
    with lr, beta1, beta2, eps, weight_decay. ``grad_present``: None, a ctypes
    uint32 bitmask, or per-tensor booleans. ``step``: device int32 [n_tensors].
    ``inv_scale`` / ``found_inf``: device fp32 scalars or None.
    """
    ga = groups if isinstance(groups, ctypes.Array) else groups_array(groups)
    n_groups = len(groups)
    if grad_present is not None and not isinstance(grad_present, ctypes.Array):
        grad_present = pack_present(grad_present, plan.n_tensors)
    rc = lib().adamw_step(plan.handle, ga, n_groups, grad_present, _ptr(step),
                          _ptr(inv_scale), _ptr(found_inf), _stream(stream))
    _check(rc, "adamw_step")


def adamw_step_noalloc(tensors: Sequence[adamw_tensor_t], state_kind, groups,
                       grad_present=None, step=None, inv_scale=None, found_inf=None,
                       stream=None) -> None:
    """One step without a plan and without any device allocation (see the
    header: shared fixed-size scratch, first call per device sets it up)."""
    sk = STATE_CODES[state_kind] if isinstance(state_kind, str) else int(state_kind)
    arr = (adamw_tensor_t * max(len(tensors), 1))(*tensors)
    ga = groups if isinstance(groups, ctypes.Array) else groups_array(groups)
    if grad_present is not None and not isinstance(grad_present, ctypes.Array):
        grad_present = pack_present(grad_present, len(tensors))
    rc = lib().adamw_step_noalloc(arr, len(tensors), sk, ga, len(groups), grad_present,
                                  _ptr(step), _ptr(inv_scale), _ptr(found_inf),
                                  _stream(stream))
    _check(rc, "adamw_step_noalloc")


def adamw_noalloc_error() -> int:
    """Read and clear the no-allocation step's error word on the current
    device (synchronises the device)."""
    out = ctypes.c_uint32()
    _check(lib().adamw_noalloc_error(ctypes.byref(out)), "adamw_noalloc_error")
    return out.value


def adamw_noalloc_set_debug(wait_ns: int = 0, flags: int = 0) -> None:
    """Test hook: bound on every in-kernel wait and debug flags of later
    no-allocation steps."""
    _check(lib().adamw_noalloc_set_debug(int(wait_ns), int(flags)), "adamw_noalloc_set_debug")


def adamw_grad_prologue(plan: Plan, grad_present=None, inv_scale=None, max_norm: float = 0.0,
                        found_inf_out=None, grad_norm_out=None, scale_out=None,
                        stream=None) -> None:
    """Enqueue the gradient checks before a step: non-finite flag, global L2
    norm and clip factor into device fp32 scalars (asynchronous)."""
    if grad_present is not None and not isinstance(grad_present, ctypes.Array):
        grad_present = pack_present(grad_present, plan.n_tensors)
    rc = lib().adamw_grad_prologue(plan.handle, grad_present, _ptr(inv_scale),
                                   float(max_norm), _ptr(found_inf_out), _ptr(grad_norm_out),
                                   _ptr(scale_out), _stream(stream))
    _check(rc, "adamw_grad_prologue")


def adamw_plan_set_grads(plan: Plan, grads: Sequence, stream=None) -> None:
    arr = (ctypes.c_void_p * max(len(grads), 1))(*[_ptr(g) for g in grads])
    _check(lib().adamw_plan_set_grads(plan.handle, arr, _stream(stream)),
           "adamw_plan_set_grads")


def adamw_plan_info(plan: Plan) -> dict:
    info = adamw_plan_info_t()
    _check(lib().adamw_plan_info(plan.handle, ctypes.byref(info)), "adamw_plan_info")
    return {k: getattr(info, k) for k, _ in adamw_plan_info_t._fields_}


def adamw_plan_error(plan: Plan) -> int:
    """Read and clear the plan's device error word (synchronises the device)."""
    out = ctypes.c_uint32()
    _check(lib().adamw_plan_error(plan.handle, ctypes.byref(out)), "adamw_plan_error")
    return out.value


def adamw_plan_set_debug(plan: Plan, wait_ns: int = 0, flags: int = 0) -> None:
    """Test hook: bound on every in-kernel wait and debug flags."""
    _check(lib().adamw_plan_set_debug(plan.handle, int(wait_ns), int(flags)),
           "adamw_plan_set_debug")


def adamw_plan_destroy(plan: Plan) -> None:
    if plan.handle:
        h, plan.handle = plan.handle, None
        _check(lib().adamw_plan_destroy(h), "adamw_plan_destroy")


def adamw_state_bytes(numels: Sequence[int], state_kind="f32", flags=None,
                      min_8bit_size: int = 0) -> int:
    """Optimizer-state bytes of a tensor list. ``flags``: per-tensor
    adamw_tensor_t.flags values; ``min_8bit_size`` (8-bit kinds) sets
    CS_TENSOR_STATE_F32 on tensors with fewer elements, as AdamWState does."""
    sk = STATE_CODES[state_kind] if isinstance(state_kind, str) else int(state_kind)
    n = len(numels)
    arr = (ctypes.c_int64 * max(n, 1))(*[int(x) for x in numels])
    if flags is None and min_8bit_size and state_kind in EIGHT_BIT:
        flags = [CS_TENSOR_STATE_F32 if int(x) < min_8bit_size else 0 for x in numels]
    fa = None if flags is None else (ctypes.c_int32 * max(n, 1))(*[int(f) for f in flags])
    out = ctypes.c_int64()
    _check(lib().adamw_state_bytes(arr, fa, n, sk, ctypes.byref(out)), "adamw_state_bytes")
    return out.value


def _unit_table(name, call, numels):
    n = len(numels)
    arr = (ctypes.c_int64 * max(n, 1))(*[int(x) for x in numels])
    cnt = ctypes.c_int64()
    _check(call(arr, n, None, None, None, 0, ctypes.byref(cnt)), name)
    k = cnt.value
    t = (ctypes.c_int32 * max(k, 1))()
    s = (ctypes.c_int64 * max(k, 1))()
    ln = (ctypes.c_int32 * max(k, 1))()
    _check(call(arr, n, t, s, ln, k, ctypes.byref(cnt)), name)
    return list(t[:k]), list(s[:k]), list(ln[:k])


def adamw_build_units(numels: Sequence[int], unit_elems: int = 0):
    """(tensor, start, len) lists of the work-unit cut, computed on the host."""
    L = lib()
    return _unit_table("adamw_build_units",
                       lambda a, n, t, s, ln, cap, cnt: L.adamw_build_units(
                           a, n, int(unit_elems), t, s, ln, cap, cnt), numels)


def adamw_build_queue(numels: Sequence[int], state_kind, ctas: int, unit_elems: int = 0):
    """(tensor, start, len) lists of the queue a plan builds for ``ctas`` CTAs."""
    L = lib()
    sk = STATE_CODES[state_kind] if isinstance(state_kind, str) else int(state_kind)
    return _unit_table("adamw_build_queue",
                       lambda a, n, t, s, ln, cap, cnt: L.adamw_build_queue(
                           a, n, sk, int(unit_elems), int(ctas), t, s, ln, cap, cnt), numels)


def adamw_shard_ranges(numels: Sequence[int], world: int, rank: int):
    """(lo, hi, offsets, shard_elems) of rank ``rank`` of ``world``: the part
    [lo[i], hi[i]) of every tensor the rank updates, each tensor's offset in
    the flat padded buffer, and the elements per shard (host only)."""
    n = len(numels)
    arr = (ctypes.c_int64 * max(n, 1))(*[int(x) for x in numels])
    lo = (ctypes.c_int64 * max(n, 1))()
    hi = (ctypes.c_int64 * max(n, 1))()
    off = (ctypes.c_int64 * max(n, 1))()
    sh = ctypes.c_int64()
    _check(lib().adamw_shard_ranges(arr, n, int(world), int(rank), lo, hi, off,
                                    ctypes.byref(sh)), "adamw_shard_ranges")
    return list(lo[:n]), list(hi[:n]), list(off[:n]), sh.value
