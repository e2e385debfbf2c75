"""Parity harness: the CUDA step (through the C ABI) against the CPU oracle.

Two modes, both on the same seeded inputs (``workloads``):

* free run  -- GPU and oracle each run every step from the same initial state;
               compared at the end (the fp32-state bar: |gpu-ref| <=
               2e-6 * (|ref| + rms(ref)) on theta, m, v after all steps).
* forced    -- before every step the oracle's stored state (theta, moments,
               scales, step counts) is uploaded into the GPU buffers at the
               compared positions, one GPU step runs, and its outputs are
               compared with one oracle step. Inputs flow from the oracle to
               the GPU only. Bars: bf16 values <= 1 ulp, int8 codes +-1 and
               scales <= 1e-6 relative, fp32 values by the fp32 rule,
               bf16/fp16 params <= 1 ulp of their format, step counts exact.

With fp32 master weights (``master=True``, 16-bit params) the master is
compared by the fp32 rule, and the 16-bit param must equal torch's rounding of
the GPU's own master bit for bit, besides the 16-bit param bar against the
oracle.

Positions are either whole tensors or a seeded sample (whole 256-element blocks
for int8 state), so full-size workloads can be checked element by element.
Steps whose found_inf flag is set and tensors without a gradient are checked
bit for bit against a snapshot of the GPU buffers taken before the step.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np
import torch

import workloads
from oracle import formats as ofmt
from oracle.adamw import TensorState, new_state, oracle_step

F32_RTOL = 2e-6
EIGHT_BIT = ("int8", "int8uv", "dyn8")
# fp32 values are graded per tensor, relative to |ref| + the tensor's own rms.
# A tensor with fewer compared positions than this has no reliable scale of
# its own (one element near a zero crossing has rms ~ 0), so its rms is
# floored at the rms of all compared positions of the same quantity.
SMALL_TENSOR = 32


# --------------------------------------------------------------------- metrics

def _ordered_bits(x: np.ndarray, fmt: str) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    if fmt == "f32":
        b = x.astype(np.float32).view(np.int32).astype(np.int64)
        sign, mag = b < 0, b & 0x7FFFFFFF
    elif fmt == "bf16":
        b = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.int64)
        sign, mag = (b & 0x8000) != 0, b & 0x7FFF
    elif fmt == "f16":
        b = x.astype(np.float16).view(np.uint16).astype(np.int64)
        sign, mag = (b & 0x8000) != 0, b & 0x7FFF
    else:
        raise ValueError(fmt)
    return np.where(sign, -mag, mag)


def ulp_diff(a, b, fmt: str) -> np.ndarray:
    """Distance in units in the last place of ``fmt`` (values must be
    representable in ``fmt``); NaN positions must agree (else a huge value)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    d = np.abs(_ordered_bits(a, fmt) - _ordered_bits(b, fmt))
    na, nb = np.isnan(a), np.isnan(b)
    d = np.where(na & nb, 0, d)
    d = np.where(na ^ nb, 1 << 40, d)
    return d


def ulp_of(x, fmt: str) -> np.ndarray:
    """Spacing of ``fmt`` values at |x| (the finest quantum at zero)."""
    f = ofmt.FORMATS[fmt]
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(x > 0, x, 1.0))
    q = np.maximum(e - f.p, f.q_min)
    return np.where(x > 0, np.ldexp(1.0, q), np.ldexp(1.0, f.q_min))


def param16_excess(gpu, ref, fmt: str) -> float:
    """16-bit params: max |gpu-ref| / (ulp(ref) + 2^-20 * rms(ref)); <= 1 passes.
    One ulp covers fp32 -> 16-bit double rounding; the rms term covers the fp32
    rounding of theta*decay - update where the two nearly cancel."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    fin = np.isfinite(ref)
    if not np.array_equal(fin, np.isfinite(gpu)):
        return float("inf")
    if not fin.any():
        return 0.0
    rms = float(np.sqrt(np.mean(ref[fin] ** 2)))
    den = ulp_of(ref[fin], fmt) + 2.0 ** -20 * rms
    return float(np.max(np.abs(gpu[fin] - ref[fin]) / den))


def _rms(x) -> float:
    x = np.asarray(x, dtype=np.float64)
    x = x[np.isfinite(x)]
    return float(np.sqrt(np.mean(x ** 2))) if x.size else 0.0


def f32_excess(gpu, ref, rtol=F32_RTOL, rms_floor: float = 0.0) -> float:
    """max |gpu-ref| / (rtol*(|ref|+rms)); <= 1 passes. rms is the rms of
    ``ref`` itself, or ``rms_floor`` when that is larger."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    fin = np.isfinite(ref)
    if not np.array_equal(fin, np.isfinite(gpu)):
        return float("inf")
    if not fin.any():
        return 0.0
    rms = max(float(np.sqrt(np.mean(ref[fin] ** 2))), rms_floor)
    den = rtol * (np.abs(ref[fin]) + rms)
    den = np.where(den == 0, np.finfo(np.float64).tiny, den)
    return float(np.max(np.abs(gpu[fin] - ref[fin]) / den))


def f32_max_rel(gpu, ref) -> float:
    """max relative error over elements with |ref| >= rms(ref) (reported)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    if not fin.any():
        return 0.0
    rms = float(np.sqrt(np.mean(ref[fin] ** 2)))
    sel = fin & (np.abs(ref) >= rms) & (ref != 0)
    if not sel.any():
        return 0.0
    return float(np.max(np.abs(gpu[sel] - ref[sel]) / np.abs(ref[sel])))


# ----------------------------------------------------------------------- setup

def torch_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy().reshape(-1)


def f64_to_torch(x: np.ndarray, dtype, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(dtype).to(device)


@dataclasses.dataclass
class Result:
    free: Dict[str, float] = dataclasses.field(default_factory=dict)
    forced: Dict[str, float] = dataclasses.field(default_factory=dict)
    steps_checked: int = 0


class Harness:
    """GPU buffers + oracle states for one workload and state kind."""

    def __init__(self, wl: workloads.Workload, state_kind: str, unit_elems: int = 0,
                 sample: Optional[int] = None, grad_device: str = "cpu",
                 param_device_init: str = "cpu", misalign: bool = False,
                 device: str = "cuda", seed: int = 0, master: bool = False,
                 min_8bit_size: int = 0):
        from compact_state_gb300.torch_adapter import AdamWState
        self.wl = wl
        self.kind = state_kind
        self.dev = torch.device(device)
        self.grad_device = grad_device
        self.fmt = wl.param_dtype
        pdt = workloads.torch_dtype(wl.param_dtype)
        n = len(wl.tensors)
        self._storage = []            # keeps misaligned backing buffers alive
        self.params, self.grads = [], []
        for i, spec in enumerate(wl.tensors):
            p0 = workloads.init_param(wl, i, device=param_device_init)
            if misalign:
                bp = torch.empty(spec.numel + 1, dtype=pdt, device=self.dev)
                bg = torch.empty(spec.numel + 1, dtype=pdt, device=self.dev)
                self._storage += [bp, bg]
                p, g = bp[1:], bg[1:]
            else:
                p = torch.empty(spec.numel, dtype=pdt, device=self.dev)
                g = torch.empty(spec.numel, dtype=pdt, device=self.dev)
            p.copy_(p0.reshape(-1).to(self.dev))
            g.zero_()
            self.params.append(p)
            self.grads.append(g)
        self.master = master
        self.state = AdamWState(self.params, self.grads, state_kind,
                                [t.group for t in wl.tensors], unit_elems, master=master,
                                min_8bit_size=min_8bit_size)
        # per-tensor state kind: fp32 for tensors an 8-bit plan keeps in fp32
        self.kinds = ["f32" if f else state_kind for f in self.state.fp32_state]
        if misalign:
            # moments of the misaligned case start one element into a buffer too
            self._misalign_state(pdt)
        # compared positions
        rng = np.random.default_rng(seed + 12345)
        self.idx: List[np.ndarray] = []
        for spec in wl.tensors:
            ne = spec.numel
            if sample is None or ne <= sample:
                self.idx.append(np.arange(ne, dtype=np.int64))
            elif state_kind in EIGHT_BIT:
                nb = -(-ne // 256)
                k = max(1, sample // 256)
                blocks = np.sort(rng.choice(nb, size=min(k, nb), replace=False))
                blocks[-1] = nb - 1                      # keep the ragged tail block
                blocks = np.unique(blocks)
                el = (blocks[:, None] * 256 + np.arange(256)[None, :]).reshape(-1)
                self.idx.append(el[el < ne])
            else:
                el = np.sort(rng.choice(ne, size=sample, replace=False))
                el[-1] = ne - 1
                self.idx.append(np.unique(el))
        self.tidx = [torch.from_numpy(ix).to(self.dev) for ix in self.idx]
        # oracle states over the compared positions
        self.ostates: List[TensorState] = []
        for i, spec in enumerate(wl.tensors):
            th = torch_to_f64(self.params[i].view(-1)[self.tidx[i]])
            self.ostates.append(new_state(th, self.fmt, self.kinds[i], group=spec.group,
                                          master=master))
        self.gpu_groups = self._gpu_groups()
        self.inv_scale_t = torch.tensor([wl.inv_scale], dtype=torch.float32, device=self.dev)
        self.found_inf_t = torch.zeros(1, dtype=torch.float32, device=self.dev)
        self.scratch = None
        self.last_step = 0

    def _misalign_state(self, pdt):
        from compact_state_gb300 import adamw_plan_create, adamw_plan_destroy, tensor_desc
        st = self.state
        adamw_plan_destroy(st.plan)
        descs = []
        for i, spec in enumerate(self.wl.tensors):
            bm = torch.zeros(spec.numel + 1, dtype=st.m[i].dtype, device=self.dev)
            bv = torch.zeros(spec.numel + 1, dtype=st.v[i].dtype, device=self.dev)
            self._storage += [bm, bv]
            st.m[i], st.v[i] = bm[1:], bv[1:]
            if st.master[i] is not None:
                bw = torch.empty(spec.numel + 1, dtype=torch.float32, device=self.dev)
                bw[1:].copy_(st.master[i])
                self._storage.append(bw)
                st.master[i] = bw[1:]
            descs.append(tensor_desc(self.params[i], self.grads[i], st.m[i], st.v[i],
                                     st.m_scale[i], st.v_scale[i], group=spec.group,
                                     master=st.master[i],
                                     flags=1 if st.fp32_state[i] else 0))
        st.plan = adamw_plan_create(descs, self.kind, 0)

    def _gpu_groups(self):
        # the GPU sees fp32 hyper-parameters; the oracle uses the same fp32 values
        f = lambda x: float(np.float32(x))
        return [dict(lr=f(g.lr), beta1=f(g.beta1), beta2=f(g.beta2), eps=f(g.eps),
                     weight_decay=f(g.weight_decay)) for g in self.wl.groups]

    # ---------------------------------------------------------------- steps
    def _fill_grads(self, s: int) -> List[np.ndarray]:
        """Write step ``s`` grads into the GPU buffers; return them at the
        compared positions (float64, as stored)."""
        out = []
        for i, spec in enumerate(self.wl.tensors):
            if self.grad_device == "cpu":
                g = workloads.grad(self.wl, i, s, device="cpu")
                self.grads[i].copy_(g.reshape(-1).to(self.dev))
                gv = g.reshape(-1).to(torch.float64).numpy()[self.idx[i]]
            else:
                if self.scratch is None or self.scratch.numel() < spec.numel:
                    big = max(t.numel for t in self.wl.tensors)
                    self.scratch = torch.empty(big, dtype=torch.float32, device=self.dev)
                workloads.fill_grad(self.wl, i, s, self.grads[i].view(spec.shape),
                                    scratch=self.scratch)
                gv = torch_to_f64(self.grads[i].view(-1)[self.tidx[i]])
            out.append(gv)
        return out

    def _upload_oracle_state(self):
        """Forced mode: oracle state -> GPU buffers at the compared positions."""
        st = self.state
        pdt = workloads.torch_dtype(self.fmt)
        steps = st.step.clone()
        for i, o in enumerate(self.ostates):
            ix = self.tidx[i]
            self.params[i].view(-1)[ix] = f64_to_torch(o.theta, pdt, self.dev)
            if o.master is not None:
                st.master[i][ix] = f64_to_torch(o.master, torch.float32, self.dev)
            if o.state_kind in EIGHT_BIT:
                st.m[i][ix] = torch.from_numpy(o.m).to(self.dev)
                st.v[i][ix] = torch.from_numpy(o.v).to(self.dev)
                blk = torch.unique(ix // 256)
                st.m_scale[i][blk] = torch.from_numpy(o.m_scale).to(self.dev)[
                    self._oblk(i, blk)]
                st.v_scale[i][blk] = torch.from_numpy(o.v_scale).to(self.dev)[
                    self._oblk(i, blk)]
            else:
                sdt = st.m[i].dtype
                st.m[i][ix] = f64_to_torch(o.m, sdt, self.dev)
                st.v[i][ix] = f64_to_torch(o.v, sdt, self.dev)
            steps[i] = o.step
        st.step.copy_(steps)

    def _oblk(self, i, blk):
        """Map absolute block ids of tensor i to indices into the oracle's
        per-sample scale arrays (the sample holds whole blocks, in order)."""
        ob = np.unique(self.idx[i] // 256)
        pos = {int(b): k for k, b in enumerate(ob)}
        return torch.tensor([pos[int(b)] for b in blk.cpu().numpy()], dtype=torch.long,
                            device=self.dev)

    def _gpu_state(self, i):
        st = self.state
        ix = self.tidx[i]
        th = torch_to_f64(self.params[i].view(-1)[ix])
        if self.kinds[i] in EIGHT_BIT:
            m = st.m[i][ix].cpu().numpy()
            v = st.v[i][ix].cpu().numpy()
            blk = torch.from_numpy(np.unique(self.idx[i] // 256)).to(self.dev)
            ms = st.m_scale[i][blk].cpu().numpy()
            vs = st.v_scale[i][blk].cpu().numpy()
            return th, m, v, ms, vs
        return th, torch_to_f64(st.m[i][ix]), torch_to_f64(st.v[i][ix]), None, None

    def snapshot(self):
        st = self.state
        c = lambda x: None if x is None else x.clone()
        return [(self.params[i].clone(), st.m[i].clone(), st.v[i].clone(),
                 c(st.m_scale[i]), c(st.v_scale[i]), c(st.master[i]))
                for i in range(len(self.params))], st.step.clone()

    def assert_unchanged(self, snap, tensors):
        bufs, steps = snap
        st = self.state
        cur_steps = st.step
        for i in tensors:
            p, m, v, ms, vs, mw = bufs[i]
            assert _bits_equal(p, self.params[i]), f"param {i} changed"
            if mw is not None:
                assert _bits_equal(mw, st.master[i]), f"master {i} changed"
            assert _bits_equal(m, st.m[i]), f"m {i} changed"
            assert _bits_equal(v, st.v[i]), f"v {i} changed"
            if ms is not None:
                assert _bits_equal(ms, st.m_scale[i]) and _bits_equal(vs, st.v_scale[i])
            assert int(cur_steps[i]) == int(steps[i]), f"step {i} changed"

    def gpu_step(self, s: int, present: np.ndarray, fi: bool):
        self.found_inf_t.fill_(1.0 if fi else 0.0)
        self.state.run(self.gpu_groups, None if present.all() else present,
                       self.inv_scale_t, self.found_inf_t)

    def run(self, steps: Optional[int] = None, forced: bool = False,
            check_invariants: bool = True) -> Result:
        res = Result()
        steps = steps or self.wl.steps
        worst: Dict[str, float] = {}
        for s in range(1, steps + 1):
            present = self.wl.present(s)
            fi = self.wl.found_inf(s)
            gv = self._fill_grads(s)
            if forced:
                self._upload_oracle_state()
            snap = self.snapshot() if (check_invariants and (fi or not present.all())) else None
            torch.cuda.synchronize()
            self.gpu_step(s, present, fi)
            torch.cuda.synchronize()
            oracle_step(self.ostates, self.gpu_groups,
                        [g if p else None for g, p in zip(gv, present)],
                        inv_scale=float(np.float32(self.wl.inv_scale)),
                        found_inf=1.0 if fi else 0.0)
            if snap is not None:
                self.assert_unchanged(snap, range(len(self.params)) if fi
                                      else np.nonzero(~present)[0])
            gsteps = self.state.step.cpu().numpy()
            osteps = np.array([o.step for o in self.ostates])
            assert np.array_equal(gsteps[:len(osteps)], osteps), "step counts differ"
            if forced:
                self._compare(worst, final=False)
            res.steps_checked += 1
        if forced:
            res.forced = worst
        else:
            self._compare(worst, final=True)
            res.free = worst
        return res

    # ----------------------------------------------------------- comparison
    def _compare(self, worst: Dict[str, float], final: bool):
        upd = lambda k, x: worst.__setitem__(k, max(worst.get(k, 0.0), float(x)))
        th_all, thr_all, th16, th16r = [], [], [], []
        mv = {"m": ([], []), "v": ([], [])}
        for i, o in enumerate(self.ostates):
            th, m, v, ms, vs = self._gpu_state(i)
            if o.master is not None:
                # the master by the fp32 rule; the 16-bit param is exactly the
                # rounding of the GPU's own master
                mw = self.state.master[i][self.tidx[i]]
                th_all.append(torch_to_f64(mw))
                thr_all.append(o.master)
                cast = torch_to_f64(mw.to(workloads.torch_dtype(self.fmt)))
                upd("copy_mismatch", int(np.sum(~((cast == th) | (np.isnan(cast) &
                                                                   np.isnan(th))))))
            if self.fmt == "f32":
                th_all.append(th)
                thr_all.append(o.theta)
            else:
                upd("theta_ulp", ulp_diff(th, o.theta, self.fmt).max(initial=0))
                th16.append(th)
                th16r.append(o.theta)
            kind = self.kinds[i]
            if kind == "f32":
                # graded per tensor (see SMALL_TENSOR)
                mv["m"][0].append(m)
                mv["m"][1].append(o.m)
                mv["v"][0].append(v)
                mv["v"][1].append(o.v)
            elif kind == "bf16":
                upd("m_ulp", ulp_diff(m, o.m, "bf16").max(initial=0))
                upd("v_ulp", ulp_diff(v, o.v, "bf16").max(initial=0))
            else:
                upd("m_code", np.abs(code_index(m, kind, "m") -
                                     code_index(o.m, kind, "m")).max(initial=0))
                upd("v_code", np.abs(code_index(v, kind, "v") -
                                     code_index(o.v, kind, "v")).max(initial=0))
                upd("m_scale_rel", _scale_rel(ms, o.m_scale))
                upd("v_scale_rel", _scale_rel(vs, o.v_scale))
        if th_all:
            _grade_f32(upd, "theta", th_all, thr_all)
        if th16:
            upd("theta16_excess", max(param16_excess(g, r, self.fmt)
                                      for g, r in zip(th16, th16r)))
        for k, (g, r) in mv.items():
            if g:
                _grade_f32(upd, k, g, r)


def _grade_f32(upd, key, gpu_list, ref_list) -> None:
    """fp32 bar per tensor: each tensor against its own rms, floored at the
    pooled rms for tensors with fewer than SMALL_TENSOR compared positions."""
    pooled = _rms(np.concatenate(ref_list)) if ref_list else 0.0
    for g, r in zip(gpu_list, ref_list):
        floor = pooled if np.asarray(r).size < SMALL_TENSOR else 0.0
        upd(f"{key}_excess", f32_excess(g, r, rms_floor=floor))
        upd(f"{key}_maxrel", f32_max_rel(g, r))


def _scale_rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.size == 0:
        return 0.0
    na, nb = ~np.isfinite(a), ~np.isfinite(b)
    if not np.array_equal(np.isnan(a), np.isnan(b)) or not np.array_equal(na, nb):
        return float("inf")
    zero = (b == 0) | nb
    if np.any(a[zero & ~nb] != 0):
        return float("inf")
    sel = ~zero
    if not sel.any():
        return 0.0
    return float(np.max(np.abs(a[sel] - b[sel]) / np.abs(b[sel])))


def _bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    if a.dtype.itemsize == 1:
        return torch.equal(a.view(torch.int8), b.view(torch.int8))
    view = {2: torch.int16, 4: torch.int32}[a.element_size()]
    return torch.equal(a.contiguous().view(view), b.contiguous().view(view))


def code_index(codes, kind: str, which: str) -> np.ndarray:
    """Codes as positions on their codebook's axis, so neighbouring values
    differ by one: signed linear codes as themselves, unsigned bytes as
    0..255, signed codebook bytes (sign<<7 | r) as +-r."""
    c = np.asarray(codes)
    if kind == "dyn8" and which == "m":
        b = c.astype(np.uint8).astype(np.int64)
        return np.where(b & 0x80, -(b & 0x7F), b & 0x7F)
    return c.astype(np.int64)


def check_bars(res: Result, kind: str, fmt: str, forced: bool) -> None:
    """Assert the tolerances for the mode that ran: every key present must
    meet its bar, and the keys of the state kind and param format must be
    there (so a comparison that did not run cannot pass)."""
    w = res.forced if forced else res.free
    bars = {"theta_excess": 1.0, "theta16_excess": 1.0, "m_excess": 1.0, "v_excess": 1.0,
            "m_ulp": 1, "v_ulp": 1, "m_code": 1, "v_code": 1, "m_scale_rel": 1e-6,
            "v_scale_rel": 1e-6, "copy_mismatch": 0}
    need = {"f32": ["m_excess", "v_excess"], "bf16": ["m_ulp", "v_ulp"]}.get(
        kind, ["m_code", "v_code", "m_scale_rel", "v_scale_rel"])
    need = need + (["theta_excess"] if fmt == "f32" else ["theta16_excess"])
    for k in need:
        assert k in w, (k, w)
    for k, bar in bars.items():
        assert w.get(k, 0) <= bar, (k, w)
