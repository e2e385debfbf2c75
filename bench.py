#!/usr/bin/env python3
"""Benchmark of the fused multi-tensor AdamW step on GB300.

Default workload: the parameter list of an 8B Llama-3-shaped model (291
tensors, 8,030,261,248 elements) with bf16 params and grads and fp32 moments,
22 bytes of algorithmic traffic per element and step; two groups (matrices
with weight decay, norms without). ``--workload few_large`` runs eight
4096x4096 fp32 tensors (28 bytes per element) instead.
One step is one ``adamw_step`` call (one kernel launch) over every tensor:
overflow predicate, per-tensor step count and bias-correction scalars, the
descriptor walk, load/decode, moment and parameter update, encode/store.

Prints ONE JSON line (rank 0):
  value      parameter-elements per second, whole job (all ranks), inputs resident
  roofline   achieved algorithmic GB/s of the step kernel vs the measured HBM peak
  e2e        the same metric through the C ABI with HOST buffers: every step
             copies the grads in from pinned host memory and the updated params
             back out; the optimizer state stays resident in HBM
             (``--e2e-offload`` adds a fully offloaded variant: params, grads
             and moments cross the host link every step)
  cpu_baseline  the CPU oracle on a bounded sample of the workload (rank 0)
  clocks     SM clocks sampled by nvidia-smi during the timed region

``--impl reference`` times the CPU oracle instead, on the same metric.
``--impl torch_fused`` / ``torch_foreach`` time PyTorch's own AdamW
(``torch.optim.AdamW(fused=True)`` / ``foreach=True``) on the same workload
and GPU, for context: it keeps its moments in the param dtype, so its line
compares with this step's ``--state f32`` line for fp32 params and
``--state bf16`` for 16-bit ones.
Under torchrun each rank runs an independent replica ("replicas only": the step
has no exchange); value = elements of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

BYTES_PER_ELEM = {  # (param dtype, state kind) -> read + write bytes per element
    ("f32", "f32"): 28, ("bf16", "f32"): 22, ("f16", "f32"): 22,
    ("f32", "bf16"): 20, ("bf16", "bf16"): 14, ("f16", "bf16"): 14,
    ("f32", "int8"): 16.0625, ("bf16", "int8"): 10.0625, ("f16", "int8"): 10.0625,
}
for _p in ("f32", "bf16", "f16"):       # the other 8-bit codecs move the same bytes
    for _k in ("int8uv", "dyn8"):
        BYTES_PER_ELEM[(_p, _k)] = BYTES_PER_ELEM[(_p, "int8")]
FALLBACK_HBM_GBS = 6800.0


def bytes_per_elem(param_dtype: str, state: str, master: bool = False) -> float:
    """Algorithmic bytes per element of one step. With fp32 master weights
    theta is read from the master (4 B instead of the 16-bit param's 2) and
    written to both (4 + 2 B instead of 2): 6 B more."""
    return BYTES_PER_ELEM[(param_dtype, state)] + (6 if master else 0)
KERNEL_SRCS = [os.path.join(ROOT, "compact_state_gb300", "csrc", f)
               for f in ("step_kernel.cuh", "adamw_internal.h")]


def kernel_hash() -> str:
    """Hash of the step kernel's code, comments and layout whitespace left
    out (a committed traffic figure is only reported while it matches)."""
    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        with open(path, encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def load_workload(name: str):
    import workloads
    return {"few_large": workloads.few_large, "llama3_8b": workloads.llama3_8b,
            "llama3_8b_layer": workloads.llama3_8b_layer,
            "many_small_only": workloads.many_small_only,
            "many_small": workloads.many_small, "lora": workloads.lora,
            "tiny": workloads.tiny}[name]()


def describe(wl, state: str) -> str:
    shapes = {}
    for t in wl.tensors:
        shapes[t.shape] = shapes.get(t.shape, 0) + 1
    if len(shapes) <= 4:
        lst = ", ".join(f"{c} x {'x'.join(map(str, s))}" for s, c in shapes.items())
    else:
        lst = f"{len(wl.tensors)} tensors"
    return (f"{wl.name}: {lst}; {wl.param_dtype} params/grads, {state} m/v, "
            f"{len(wl.groups)} group(s)")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (every 100 ms)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((t, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.15 <= r[0] <= (self.t1 or 1e30) + 0.15]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in use for k, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use), "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": len(inside)}


# ------------------------------------------------------------------ peaks
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def committed_traffic(workload: str, state: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            j = json.load(f)
        e = j.get(f"{workload}/{state}")
        if e and e.get("kernel_sha") == kernel_hash():
            return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError):
        pass
    return None


# ------------------------------------------------------------------ oracle
def _oracle_setup(wl, state, n, master=False):
    import numpy as np
    from oracle.adamw import new_state
    big = max(range(len(wl.tensors)), key=lambda i: wl.tensors[i].numel)
    n = min(wl.tensors[big].numel, n)
    rng = np.random.default_rng(0)
    st = [new_state(rng.normal(0, wl.param_std, n), wl.param_dtype, state,
                    group=wl.tensors[big].group, master=master)]
    groups = [dict(lr=x.lr, beta1=x.beta1, beta2=x.beta2, eps=x.eps,
                   weight_decay=x.weight_decay) for x in wl.groups]
    grads = [rng.normal(0, wl.grad_std, n) * wl.grad_prescale for _ in range(2)]
    return st, groups, grads, n, wl.tensors[big].name


def cpu_baseline(wl, state: str, budget_s: float = 12.0, n_max: int = 1 << 21,
                 master: bool = False) -> dict:
    """The oracle, as it is, on a bounded sample: a contiguous slice of the
    workload's largest tensor, stepped repeatedly for about ``budget_s``."""
    from oracle.adamw import oracle_step
    st, groups, grads, n, name = _oracle_setup(wl, state, n_max, master)
    steps = 0
    t0 = time.perf_counter()
    while True:
        oracle_step(st, groups, [grads[steps % 2]], inv_scale=wl.inv_scale)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": steps * n / el, "unit": "param-elements/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{n} elements of tensor '{name}' ({wl.param_dtype} params"
                      f"{' with fp32 master' if master else ''}, {state} state), {steps} steps in {el:.1f} s, numpy float64, "
                      f"one thread"}


def reference_arm(wl, state: str, steps: int, warmup: int, n: int = 1 << 20,
                  master: bool = False) -> dict:
    """W untimed + K timed oracle steps, each over a bounded sample of n elements."""
    from oracle.adamw import oracle_step
    st, groups, grads, n, name = _oracle_setup(wl, state, n, master)
    for k in range(warmup):
        oracle_step(st, groups, [grads[k % 2]], inv_scale=wl.inv_scale)
    t0 = time.perf_counter()
    for k in range(steps):
        oracle_step(st, groups, [grads[k % 2]], inv_scale=wl.inv_scale)
    el = time.perf_counter() - t0
    return {"value": steps * n / el, "unit": "param-elements/s", "cores": 1,
            "kind": "oracle", "elapsed_s": el, "step_elements": n,
            "ms_per_sample_step": el / max(steps, 1) * 1e3,
            "sample": f"each step: {n} elements of tensor '{name}' ({wl.param_dtype} "
                      f"params{' with fp32 master' if master else ''}, {state} state), numpy float64, one thread"}


# ------------------------------------------------------------------ GPU arm
def alloc_state(wl, state, dev, master=False, min_8bit_size=0, unit_elems=0):
    import torch
    import workloads
    from compact_state_gb300.torch_adapter import AdamWState
    pdt = workloads.torch_dtype(wl.param_dtype)
    params = []
    for i, t in enumerate(wl.tensors):
        p = torch.empty(t.numel, dtype=pdt, device=dev)
        p.copy_(workloads.init_param(wl, i, device=dev).reshape(-1))
        params.append(p)
    grads = [torch.empty_like(p) for p in params]
    st = AdamWState(params, grads, state, [t.group for t in wl.tensors], unit_elems,
                    master=master, min_8bit_size=min_8bit_size)
    return st


def grad_sets(wl, st, n_sets, dev):
    """Pre-generated grad buffers (seeded, fresh per step up to n_sets)."""
    import torch
    import workloads
    big = max(t.numel for t in wl.tensors)
    scratch = torch.empty(big, dtype=torch.float32, device=dev)
    sets = [st.grads]
    for _ in range(n_sets - 1):
        sets.append([torch.empty_like(g) for g in st.grads])
    for k, gs in enumerate(sets):
        for i, g in enumerate(gs):
            workloads.fill_grad(wl, i, k + 1, g.view(wl.tensors[i].shape), scratch=scratch)
    del scratch
    return sets


def run_torch_adamw(args, wl, dev, impl):
    """PyTorch's AdamW (``fused=True`` or ``foreach=True``, by ``impl``) over
    the workload's tensors: one optimizer step
    per timed step, every gradient present, the workload's groups as param
    groups. Moments in the param dtype (PyTorch's rule): 28 B/element with
    fp32 params, 14 with 16-bit ones."""
    import torch
    import workloads
    pdt = workloads.torch_dtype(wl.param_dtype)
    params = []
    for i, t in enumerate(wl.tensors):
        p = torch.empty(t.numel, dtype=pdt, device=dev)
        p.copy_(workloads.init_param(wl, i, device=dev).reshape(-1))
        p.grad = torch.empty_like(p)
        workloads.fill_grad(wl, i, 1, p.grad.view(t.shape))
        params.append(p)
    pgroups = [dict(params=[p for p, t in zip(params, wl.tensors) if t.group == k],
                    lr=g.lr, betas=(g.beta1, g.beta2), eps=g.eps, weight_decay=g.weight_decay)
               for k, g in enumerate(wl.groups)]
    mode = {"fused": True} if impl == "torch_fused" else {"foreach": True}
    opt = torch.optim.AdamW([g for g in pgroups if g["params"]], **mode)
    for _ in range(args.warmup):
        opt.step()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(dev.index if dev.index is not None else 0)
    clk.start()
    time.sleep(0.3)
    clk.mark(True)
    e0.record(stream)
    for _ in range(args.steps):
        opt.step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk.mark(False)
    ms = e0.elapsed_time(e1) / args.steps
    bpe = 28 if wl.param_dtype == "f32" else 14
    peak, peak_src = hbm_peak()
    achieved = wl.total_numel * bpe / (ms / 1e3) / 1e9
    return {"value": wl.total_numel / (ms / 1e3), "ms_per_step": ms, "clocks": clk.stop(),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None,
                         "peak_source": f"hbm_gbs of {peak_src}", "bytes_per_elem": bpe}}


def run_native(args, wl, rank, world, dev):
    import torch
    import compact_state_gb300 as cs
    from compact_state_gb300 import tensor_desc
    state = args.state
    st = alloc_state(wl, state, dev, args.master, args.min_8bit_size, args.unit_elems)
    plan_info = cs.adamw_plan_info(st.plan)
    # grad buffers: fresh seeded grads per step, cycling through a pool
    per_set = sum(g.numel() * g.element_size() for g in st.grads)
    free, _ = torch.cuda.mem_get_info()
    n_sets = int(max(1, min(args.grad_sets, (free * 0.5) // max(per_set, 1))))
    sets = grad_sets(wl, st, n_sets, dev)
    # one plan per grad set (descriptors hold grad pointers)
    plans = [st.plan]
    for gs in sets[1:]:
        descs = [tensor_desc(p, g, m, v, ms, vs, group=t.group, master=mw, flags=int(f32))
                 for p, g, m, v, ms, vs, mw, f32, t in zip(
                     st.params, gs, st.m, st.v, st.m_scale, st.v_scale, st.master,
                     st.fp32_state, wl.tensors)]
        plans.append(cs.adamw_plan_create(descs, state, args.unit_elems))
    groups = cs.groups_array([dict(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                                   weight_decay=g.weight_decay) for g in wl.groups])
    ng = len(wl.groups)
    inv = torch.tensor([wl.inv_scale], dtype=torch.float32, device=dev)
    fi = torch.zeros(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    L = cs.lib()
    hs = stream.cuda_stream

    pro = torch.zeros(3, dtype=torch.float32, device=dev)   # found_inf, norm, scale
    fi_one = torch.ones(1, dtype=torch.float32, device=dev)

    # The workload's own schedule: tensors without a gradient in a step (the
    # seeded grad-presence mask) and overflowing steps (found_inf = 1) are
    # timed as configured; a step updates only its present tensors.
    n_t = len(wl.tensors)
    schedule = []
    for s_ in range(1, wl.steps + 1):
        pres = wl.present(s_)
        bits = None if pres.all() else cs.pack_present(pres, n_t)
        upd = int(sum(t.numel for t, p in zip(wl.tensors, pres) if p))
        schedule.append((bits, bool(wl.found_inf(s_)), upd))

    def sched(k):
        return schedule[k % len(schedule)]

    def one(k):
        plan = plans[k % len(plans)].handle
        bits, skip, _ = sched(k)
        fi_k = fi_one if skip else fi
        if args.prologue is not None:
            # unscale, non-finite check and clip first; the step takes their result
            rc = L.adamw_grad_prologue(plan, bits, inv.data_ptr(), float(args.prologue),
                                       pro.data_ptr(), pro.data_ptr() + 4,
                                       pro.data_ptr() + 8, hs)
            if rc:
                raise cs.CompactStateError(rc, "adamw_grad_prologue")
            rc = L.adamw_step(plan, groups, ng, bits, st.step.data_ptr(), pro.data_ptr() + 8,
                              fi_k.data_ptr() if skip else pro.data_ptr(), hs)
        else:
            rc = L.adamw_step(plan, groups, ng, bits, st.step.data_ptr(), inv.data_ptr(),
                              fi_k.data_ptr(), hs)
        if rc:
            raise cs.CompactStateError(rc, "adamw_step")

    for k in range(args.warmup):
        one(k)
    torch.cuda.synchronize(dev)
    K = args.steps
    clk = ClockSampler(dev.index if dev.index is not None else 0)
    if rank == 0:
        clk.start()
        time.sleep(0.3)
    # the timed region: K steps back to back between one start and one end
    # event (an event pair around every launch would add its own records
    # between the launches)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    clk.mark(True)
    t0 = time.perf_counter()
    e_start.record(stream)
    for k in range(K):
        one(args.warmup + k)
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    clk.mark(False)
    barrier(world)
    total_ms = e_start.elapsed_time(e_end)
    clocks = clk.stop() if rank == 0 else None
    max_ms = allreduce_max(total_ms, world, dev)
    # diagnostics, outside the timed region: the same K steps again with an
    # event pair around each launch (per-step medians, the skipped step)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for k in range(K):
        starts[k].record(stream)
        one(args.warmup + k)
        ends[k].record(stream)
    torch.cuda.synchronize(dev)
    per = [starts[k].elapsed_time(ends[k]) for k in range(K)]
    elems = wl.total_numel
    # per tensor: tensors an 8-bit plan keeps in fp32 move fp32-state bytes
    tbytes = [t.numel * bytes_per_elem(wl.param_dtype, "f32" if f32 else state, args.master)
              + (t.numel * (4 if wl.param_dtype == "f32" else 2) if args.prologue is not None
                 else 0)        # the prologue reads the grads once more
              for t, f32 in zip(wl.tensors, st.fp32_state)]
    bpe = sum(tbytes) / max(elems, 1)
    # elements and bytes each timed step updates (its present tensors; none
    # when the step is skipped for overflow)
    upd, ubytes, run_ms, skip_ms = [], [], [], []
    for k in range(K):
        bits, skip, n_upd = sched(args.warmup + k)
        if skip:
            skip_ms.append(per[k])
            continue
        pres = wl.present(((args.warmup + k) % len(schedule)) + 1)
        upd.append(n_upd)
        ubytes.append(sum(b for b, p in zip(tbytes, pres) if p))
        run_ms.append(per[k])
    # value: updated elements of all ranks per second of the timed region;
    # achieved: the bytes the timed steps moved per second of this rank's
    # timed region (skipped steps included in the time)
    value = world * sum(upd) / (max_ms / 1e3)
    avg_kernel_ms = sum(run_ms) / len(run_ms)
    alg_bytes = sum(ubytes) / len(ubytes)
    peak, peak_src = hbm_peak()
    achieved = sum(ubytes) / (total_ms / 1e3) / 1e9
    key = (args.workload + (f"_{args.param_dtype}" if args.param_dtype else "")
           + ("_master" if args.master else "")
           + (f"_min8bit{args.min_8bit_size}" if args.min_8bit_size else ""))
    traffic = committed_traffic(key, state)
    result = dict(
        value=value, ms_per_step=max_ms / K, kernel_ms_avg=avg_kernel_ms,
        kernel_ms_median=statistics.median(run_ms), wall_s=wall, clocks=clocks,
        timing="K steps back to back between two CUDA events on the launching stream; "
               "kernel_ms_avg/median from a second pass with an event pair per launch",
        roofline={"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                  "unit": "GB/s", "frac": round(achieved / peak, 4),
                  "traffic": traffic, "peak_source": f"hbm_gbs of {peak_src}",
                  "algorithmic_bytes_per_launch": alg_bytes,
                  "bytes_per_elem": bpe},
        plan=plan_info, grad_sets=len(plans),
        schedule={"elements_updated_per_step": sum(upd) / len(upd),
                  "steps_skipped_for_overflow": len(skip_ms),
                  "skipped_step_ms": (sum(skip_ms) / len(skip_ms)) if skip_ms else None,
                  "grad_none_fraction": wl.none_fraction})
    for p in plans[1:]:
        cs.adamw_plan_destroy(p)
    del sets
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, wl, st, groups, ng, dev, world, offload=False)
        if args.e2e_offload:
            result["e2e_offload"] = run_e2e(args, wl, st, groups, ng, dev, world,
                                            offload=True)
    return result


def link_bandwidth(dev, nbytes=1 << 30, reps=3):
    """Host-link copy bandwidth of this GPU (GB/s): pinned host -> device,
    device -> pinned host, and both directions at once on two streams."""
    import torch
    n = nbytes // 2
    h = [torch.empty(n, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    d = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    s = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]

    def run(h2d, d2h):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(reps):
            if h2d:
                with torch.cuda.stream(s[0]):
                    d[0].copy_(h[0], non_blocking=True)
            if d2h:
                with torch.cuda.stream(s[1]):
                    h[1].copy_(d[1], non_blocking=True)
        torch.cuda.synchronize(dev)
        return reps * nbytes * (int(h2d) + int(d2h)) / (time.perf_counter() - t0) / 1e9

    run(True, True)   # warm-up
    return {"h2d": round(run(True, False), 1), "d2h": round(run(False, True), 1),
            "both": round(run(True, True), 1)}


def run_e2e(args, wl, st, groups, ng, dev, world, offload=False):
    """End to end through the public API with host buffers.

    Default: the step's inputs are the gradients and its result the updated
    params, while the optimizer state (moments, scales, step counts, fp32
    masters) stays resident in HBM as in training. Every step copies the grads
    in from pinned host memory and the params back out.
    offload=True: params, grads and moments all live in pinned host memory;
    every step copies them in and params and moments back (a fully offloaded
    optimizer).
    The parameter set is cut into chunks with one plan each, so the copy-in of
    chunk i+1, the step of chunk i and the copy-out of chunk i-1 overlap on
    three streams (both copy directions run at once)."""
    import torch
    import compact_state_gb300 as cs
    from compact_state_gb300 import tensor_desc
    # chunks of at least 4 Mi elements, and at most about 64 per step for
    # large parameter sets (one plan per chunk)
    want = args.e2e_chunk or max(1 << 22, wl.total_numel // 64)
    chunk = max(256, (want // 256) * 256)
    chunks = []        # (tensor, device views: param, grad, m, v, m_scale, v_scale, master)
    for i in range(len(st.params)):
        n = st.params[i].numel()
        for c0 in range(0, max(n, 1), chunk):
            c1 = min(n, c0 + chunk)
            b0, b1 = c0 // 256, -(-c1 // 256)
            sl = lambda x, a, b: None if x is None else x[a:b]
            dv = [st.params[i][c0:c1], st.grads[i][c0:c1], st.m[i][c0:c1], st.v[i][c0:c1],
                  sl(st.m_scale[i], b0, b1), sl(st.v_scale[i], b0, b1),
                  sl(st.master[i], c0, c1)]
            chunks.append((i, dv))
    plans = []
    for (i, dv) in chunks:
        plans.append(cs.adamw_plan_create(
            [tensor_desc(dv[0], dv[1], dv[2], dv[3], dv[4], dv[5], group=wl.tensors[i].group,
                         master=dv[6], flags=int(st.fp32_state[i]))], args.state, 0))
    steps = torch.zeros(len(chunks), dtype=torch.int32, device=dev)
    inv = torch.tensor([wl.inv_scale], dtype=torch.float32, device=dev)
    # in: what the step reads (theta from the master when there is one); out:
    # what it writes. Without offload only the grads go in and the params out.
    if offload:
        in_idx = lambda dv: [j for j in ([1, 2, 3, 4, 5, 6] if dv[6] is not None
                                         else [0, 1, 2, 3, 4, 5]) if dv[j] is not None]
        out_idx = lambda dv: [j for j in (0, 2, 3, 4, 5, 6) if dv[j] is not None]
    else:
        in_idx = lambda dv: [1]
        out_idx = lambda dv: [0]
    # pinned host copies of the buffers that cross the link, and only those
    host = [[dv[j].detach().to("cpu").pin_memory()
             if dv[j] is not None and (j in in_idx(dv) or j in out_idx(dv)) else None
             for j in range(len(dv))] for _, dv in chunks]
    nbytes = lambda h: h.numel() * h.element_size()
    h2d = sum(nbytes(host[c][j]) for c, (_, dv) in enumerate(chunks) for j in in_idx(dv))
    d2h = sum(nbytes(host[c][j]) for c, (_, dv) in enumerate(chunks) for j in out_idx(dv))
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in chunks]
    ev_cmp = [torch.cuda.Event() for _ in chunks]
    ev_out = [torch.cuda.Event() for _ in chunks]
    L = cs.lib()
    first = [True]

    def one():
        for c, (_, dv) in enumerate(chunks):
            if not first[0]:
                s_in.wait_event(ev_out[c])
            with torch.cuda.stream(s_in):
                for j in in_idx(dv):
                    dv[j].copy_(host[c][j], non_blocking=True)
                ev_in[c].record(s_in)
            s_cmp.wait_event(ev_in[c])
            rc = L.adamw_step(plans[c].handle, groups, ng, None, steps[c:c + 1].data_ptr(),
                              inv.data_ptr(), None, s_cmp.cuda_stream)
            if rc:
                raise cs.CompactStateError(rc, "adamw_step")
            ev_cmp[c].record(s_cmp)
            s_out.wait_event(ev_cmp[c])
            with torch.cuda.stream(s_out):
                for j in out_idx(dv):
                    host[c][j].copy_(dv[j], non_blocking=True)
                ev_out[c].record(s_out)
        first[0] = False

    K = max(1, min(args.steps, args.e2e_steps))
    torch.cuda.synchronize(dev)
    for _ in range(min(2, args.warmup)):
        one()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_cmp.wait_event(e0)
    s_out.wait_event(e0)
    for _ in range(K):
        one()
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_cmp)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    ms = allreduce_max(e0.elapsed_time(e1), world, dev)
    for p in plans:
        cs.adamw_plan_destroy(p)
    # the link's own floor for these bytes: each direction alone, and both at once
    link = link_bandwidth(dev)
    floor_ms = 1e3 * max(h2d / (link["h2d"] * 1e9), d2h / (link["d2h"] * 1e9),
                         (h2d + d2h) / (link["both"] * 1e9))
    return {"value": world * wl.total_numel * K / (ms / 1e3), "unit": "param-elements/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
            "ms_per_step": ms / K, "chunks": len(chunks),
            "link_gbs": link, "link_floor_ms": round(floor_ms, 3),
            "of_link_floor": round(floor_ms / (ms / K), 4),
            "how": ("params, grads and moments in pinned host memory" if offload else
                    "grads in from pinned host memory, params out; optimizer state "
                    "resident in HBM") +
                   ", per-chunk plans, copy-in / step / copy-out overlapped on three streams"}


# ------------------------------------------------------------------ dist
def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x, world, dev):
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=dev if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def init_dist(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "native" else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="llama3_8b",
                    choices=["few_large", "llama3_8b", "llama3_8b_layer", "many_small",
                             "many_small_only", "lora", "tiny"])
    ap.add_argument("--state", default="f32", choices=["f32", "bf16", "int8", "int8uv", "dyn8"])
    ap.add_argument("--min-8bit-size", type=int, default=0,
                    help="with an 8-bit state, tensors below this size keep fp32 moments")
    ap.add_argument("--param-dtype", default=None, choices=["f32", "bf16", "f16"],
                    help="override the workload's param/grad dtype")
    ap.add_argument("--impl", default="native",
                    choices=["native", "reference", "torch_fused", "torch_foreach"])
    ap.add_argument("--prologue", type=float, default=None, metavar="MAX_NORM",
                    help="run the gradient prologue (non-finite check, norm, clip at "
                         "MAX_NORM) before every step and time both")
    ap.add_argument("--master", action="store_true",
                    help="fp32 master weights for the 16-bit params")
    ap.add_argument("--unit-elems", type=int, default=0,
                    help="elements per work unit (0: the library default)")
    ap.add_argument("--grad-sets", type=int, default=8)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-chunk", type=int, default=0,
                    help="elements per e2e chunk (0: max(4 Mi, total/64))")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-offload", action="store_true",
                    help="also time a fully offloaded step (params, grads and moments "
                         "copied over the host link every step)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)

    rank, world, local = init_dist(args)
    wl = load_workload(args.workload)
    if args.param_dtype:
        import dataclasses
        wl = dataclasses.replace(wl, param_dtype=args.param_dtype,
                                 name=f"{wl.name}_{args.param_dtype}")
    if args.master and wl.param_dtype == "f32":
        raise SystemExit("bench.py: --master needs 16-bit params (--param-dtype bf16 or f16)")
    metric = "AdamW step param-elements/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
    config = {"workload": describe(wl, args.state), "elements": wl.total_numel,
              "tensors": len(wl.tensors), "param_dtype": wl.param_dtype,
              "state": args.state, "groups": len(wl.groups),
              "master_weights": bool(args.master),
              "min_8bit_size": args.min_8bit_size,
              "l2": "inputs larger than L2 (no flush needed)"
                    if wl.total_numel * BYTES_PER_ELEM[(wl.param_dtype, args.state)] > 4 * 129e6
                    else "inputs smaller than L2"}

    if args.impl == "reference":
        if rank != 0:
            return 0
        cb = reference_arm(wl, args.state, args.steps, args.warmup, master=args.master)
        v = cb["value"]
        # ms_per_step is the time the oracle really spent per step: each step
        # covers the bounded sample named in cpu_baseline (step_elements), not
        # the whole parameter list, and value is elements of that sample per s
        line = {"impl": "reference", "metric": metric, "value": v, "unit": "param-elements/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": cb["ms_per_sample_step"], "step_elements": cb["step_elements"],
                "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded)", "config": config, "cpu_baseline": cb,
                "e2e": {"value": v, "unit": "param-elements/s",
                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the step has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.impl in ("torch_fused", "torch_foreach"):
        if rank != 0:
            return 0
        res = run_torch_adamw(args, wl, dev, args.impl)
        moments = "fp32" if wl.param_dtype == "f32" else wl.param_dtype
        line = {"impl": args.impl, "metric": metric, "value": res["value"],
                "unit": "param-elements/s", "n_gpus": 1, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic (seeded normal params and grads)",
                "config": dict(config, state=f"{moments} (PyTorch keeps moments in the "
                                             f"param dtype)",
                               grad_none_fraction=0.0, found_inf_steps=[]),
                "roofline": res["roofline"], "clocks": res["clocks"]}
        print(json.dumps(line), flush=True)
        return 0
    from compact_state_gb300 import build
    build.build()
    res = run_native(args, wl, rank, world, dev)
    if rank != 0:
        return 0
    cb = None if args.no_cpu_baseline or world > 1 else cpu_baseline(wl, args.state, args.cpu_budget,
                                                                    master=args.master)
    line = {"metric": metric, "value": res["value"], "unit": "param-elements/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded normal params and grads)", "config": config,
            "roofline": res["roofline"], "clocks": res["clocks"],
            "e2e": res.get("e2e"), "e2e_offload": res.get("e2e_offload"),
            "gpu_launches": args.steps * (2 if args.prologue is not None else 1),
            "kernel_ms_avg": res["kernel_ms_avg"], "kernel_ms_median": res["kernel_ms_median"],
            "timing": res["timing"],
            "grad_sets": res["grad_sets"], "schedule": res["schedule"], "cpu_baseline": cb}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
