"""The sharded step on one GPU: every rank's part run one after the other.

Each rank's ShardedAdamW is built in this one process; the reduce-scatter is
replaced by copying the rank's shard of the full gradient into its
grad_shard, and the all-gather by copying every rank's parameter shard into
every replica (the collectives themselves are exercised with gloo ranks in
test_sharded_cpu.py). The union of the ranks' updates must equal the
unsharded step of the same CUDA library bit for bit (parameters, moments,
scales and step counts), and, with fp32 moments, the oracle by the fp32 bar,
over steps with a found_inf skip and tensors without gradients.
"""
import numpy as np
import pytest
import torch

import workloads
from tests.parity_harness import _bits_equal, f32_excess

pytestmark = pytest.mark.gpu

SIZES = [5, 300, 0, 1000, 256, 70001, 1, 4096, 257, 49152 * 2 + 77]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compact_state_gb300 import build
    build.build()


def _run(world, kind, pdt, steps=6):
    from compact_state_gb300.sharded import ShardedAdamW
    from compact_state_gb300.torch_adapter import AdamWState
    wl = workloads.mixed(SIZES, param_dtype=pdt, groups=2, steps=steps, none_fraction=0.25,
                         found_inf_steps=(3,), grad_prescale=1024.0)
    grp_of = [t.group for t in wl.tensors]
    ranks = [ShardedAdamW(SIZES, pdt, kind, grp_of, world, r, "cuda") for r in range(world)]
    L0 = ranks[0].layout
    init = [workloads.init_param(wl, i).reshape(-1).cuda() for i in range(len(SIZES))]
    for sh in ranks:
        for i, x in enumerate(init):
            sh.param(i).copy_(x)
    full_p = [x.clone() for x in init]
    full_g = [torch.zeros_like(x) for x in init]
    ref = AdamWState(full_p, full_g, kind, grp_of)
    groups = [dict(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                   weight_decay=g.weight_decay) for g in wl.groups]
    inv = torch.tensor([wl.inv_scale], device="cuda")
    flat_g = torch.zeros(L0.flat_elems, dtype=full_p[0].dtype, device="cuda")
    grads_host = []
    for s in range(1, steps + 1):
        present = wl.present(s)
        fi = torch.tensor([1.0 if wl.found_inf(s) else 0.0], device="cuda")
        gs = [workloads.grad(wl, i, s).reshape(-1) for i in range(len(SIZES))]
        grads_host.append((gs, present, wl.found_inf(s)))
        for i, g in enumerate(gs):
            full_g[i].copy_(g)
            a, b = L0.flat_range(i)
            flat_g[a:b].copy_(g)
        ref.run(groups, present, inv, fi)
        for sh in ranks:       # reduce-scatter stand-in, then the local step
            s0 = sh.layout.shard_start
            sh.grad_shard.copy_(flat_g[s0:s0 + sh.layout.shard_elems])
            sh.local_step(groups, present, inv, fi)
        shards = [sh.param_shard.clone() for sh in ranks]       # all-gather stand-in
        for sh in ranks:
            for r, x in enumerate(shards):
                s0 = r * L0.shard_elems
                sh.flat_param[s0:s0 + L0.shard_elems].copy_(x)
    torch.cuda.synchronize()
    return wl, ranks, ref, init, grads_host, groups


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("kind,pdt", [("f32", "f32"), ("bf16", "bf16"), ("int8", "bf16"),
                                      ("int8uv", "f32")])
def test_union_of_shards_equals_the_unsharded_step(world, kind, pdt):
    wl, ranks, ref, _, _, _ = _run(world, kind, pdt)
    for sh in ranks:
        assert torch.equal(sh.step_counts, ref.step)
        for i in range(len(SIZES)):
            assert _bits_equal(sh.param(i), ref.params[i]), (sh.layout.rank, i)
            lo, hi = sh.layout.lo[i], sh.layout.hi[i]
            if hi > lo:
                assert _bits_equal(sh.m[i], ref.m[i][lo:hi]) and _bits_equal(sh.v[i], ref.v[i][lo:hi])
                if sh.m_scale[i] is not None:
                    b0, b1 = sh.layout.block_range(i)
                    assert _bits_equal(sh.m_scale[i][:b1 - b0], ref.m_scale[i][b0:b1])
                    assert _bits_equal(sh.v_scale[i][:b1 - b0], ref.v_scale[i][b0:b1])


def test_sharded_fp32_run_matches_the_oracle():
    from oracle.adamw import new_state, oracle_step
    wl, ranks, _, init, grads_host, groups = _run(2, "f32", "f32", steps=8)
    f = lambda x: float(np.float32(x))
    og = [{k: f(v) for k, v in g.items()} for g in groups]
    st = [new_state(x.double().cpu().numpy(), "f32", "f32", group=t.group)
          for x, t in zip(init, wl.tensors)]
    for gs, present, fi in grads_host:
        oracle_step(st, og, [g.double().numpy() if p else None for g, p in zip(gs, present)],
                    inv_scale=f(wl.inv_scale), found_inf=1.0 if fi else 0.0)
    sh = ranks[1]
    assert sh.step_counts.cpu().tolist()[:len(SIZES)] == [o.step for o in st]
    for i, o in enumerate(st):
        assert f32_excess(sh.param(i).double().cpu().numpy(), o.theta) <= 1.0, i
        # the moments of rank r's part against the oracle's slice
        for r in ranks:
            lo, hi = r.layout.lo[i], r.layout.hi[i]
            if hi > lo:
                assert f32_excess(r.m[i].double().cpu().numpy(), o.m[lo:hi],
                                  rms_floor=float(np.sqrt(np.mean(o.m ** 2)))) <= 1.0


def test_sharded_step_through_nccl_on_one_rank():
    """ShardedAdamW.step() end to end on the GPU: NCCL reduce-scatter of the
    flat gradients, all-reduce (max) of found_inf, the local fused step and
    the all-gather of parameters, with one rank (the collectives then move
    data but exchange nothing). The result must equal the unsharded step bit
    for bit, including a step whose found_inf is set."""
    import os
    import socket
    import torch.distributed as dist
    from compact_state_gb300.sharded import ShardedAdamW
    from compact_state_gb300.torch_adapter import AdamWState
    if dist.is_initialized():
        pytest.skip("a process group is already initialised")
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    try:
        wl = workloads.mixed(SIZES, param_dtype="bf16", groups=2, steps=4, found_inf_steps=(3,),
                             grad_prescale=1024.0)
        grp_of = [t.group for t in wl.tensors]
        opt = ShardedAdamW(SIZES, "bf16", "int8", grp_of, 1, 0, "cuda")
        init = [workloads.init_param(wl, i).reshape(-1).cuda() for i in range(len(SIZES))]
        for i, x in enumerate(init):
            opt.param(i).copy_(x)
        ref_p = [x.clone() for x in init]
        ref_g = [torch.zeros_like(x) for x in init]
        ref = AdamWState(ref_p, ref_g, "int8", grp_of)
        groups = [dict(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                       weight_decay=g.weight_decay) for g in wl.groups]
        inv = torch.tensor([wl.inv_scale], device="cuda")
        for s in range(1, 5):
            fi = torch.tensor([1.0 if wl.found_inf(s) else 0.0], device="cuda")
            for i in range(len(SIZES)):
                g = workloads.grad(wl, i, s).reshape(-1).cuda()
                opt.grad(i).copy_(g)
                ref_g[i].copy_(g)
            opt.step(groups, None, inv, fi)
            ref.run(groups, None, inv, fi)
        torch.cuda.synchronize()
        assert torch.equal(opt.step_counts, ref.step)
        for i in range(len(SIZES)):
            assert _bits_equal(opt.param(i), ref_p[i]), i
            if SIZES[i]:
                assert _bits_equal(opt.m[i], ref.m[i]) and _bits_equal(opt.v[i], ref.v[i]), i
    finally:
        dist.destroy_process_group()
