"""The sharded step's partition and exchange, on the CPU.

* ``adamw_shard_ranges`` (host only): over all ranks, every element of every
  tensor is owned exactly once; parts start on 256-element blocks and end on
  one or at the tensor's end, so no 8-bit scale block is split; shards are
  equal and hold whole blocks.
* ``exchange_step`` with two gloo ranks: reduce-scatter of gradients,
  all-reduce(max) of found_inf, a local update, all-gather of parameters. The
  local update here is the oracle over each rank's slices (the CUDA update of
  the same slices is compared with the unsharded CUDA step on the GPU, in
  test_sharded_gpu.py). The result must equal the unsharded oracle run on the
  summed gradients bit for bit, with a found_inf step raised on one rank only
  and tensors without gradients, and both ranks must keep identical step
  counts.
"""
import os
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SIZES = [5, 300, 0, 1000, 256, 70001, 1, 4096, 257]


@pytest.fixture(scope="module")
def cs():
    from compact_state_gb300 import build
    build.build()
    import compact_state_gb300
    return compact_state_gb300


@pytest.mark.parametrize("world", [1, 2, 3, 8])
@pytest.mark.parametrize("sizes", [SIZES, [0, 0], [1], [256] * 7, [49152 * 3 + 11, 17, 513]])
def test_partition_covers_every_element_once(cs, world, sizes):
    own = [np.zeros(n, dtype=np.int64) for n in sizes]
    shard = None
    for r in range(world):
        lo, hi, off, sh = cs.adamw_shard_ranges(sizes, world, r)
        shard = sh if shard is None else shard
        assert sh == shard and sh % 256 == 0
        for i, n in enumerate(sizes):
            assert 0 <= lo[i] <= hi[i] <= n
            if hi[i] > lo[i]:
                assert lo[i] % 256 == 0 and (hi[i] % 256 == 0 or hi[i] == n)
                # the part lies inside the rank's flat shard
                assert r * sh <= off[i] + lo[i] and off[i] + hi[i] <= (r + 1) * sh
            else:
                assert lo[i] == hi[i] == 0
            own[i][lo[i]:hi[i]] += 1
        # offsets: end to end, each tensor padded to whole blocks
        exp = np.concatenate([[0], np.cumsum([-(-n // 256) * 256 for n in sizes])[:-1]])
        assert list(off) == [int(x) for x in exp]
    for i, n in enumerate(sizes):
        assert np.all(own[i] == 1), (i, n)
    flat = sum(-(-n // 256) * 256 for n in sizes)
    assert world * shard >= flat and (world * shard - flat) < world * 256


def test_partition_rejects_bad_arguments(cs):
    with pytest.raises(cs.CompactStateError):
        cs.adamw_shard_ranges([10], 0, 0)
    with pytest.raises(cs.CompactStateError):
        cs.adamw_shard_ranges([10], 2, 2)
    with pytest.raises(cs.CompactStateError):
        cs.adamw_shard_ranges([-1], 2, 0)


def _groups():
    return [dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01),
            dict(lr=5e-4, beta1=0.8, beta2=0.99, eps=1e-6, weight_decay=0.0)]


def _schedule(step, n):
    rng = np.random.default_rng(1000 + step)
    present = rng.random(n) >= 0.25
    return present


def _grads(rank, step, sizes):
    rng = np.random.default_rng(7 * step + 100 * rank)
    return [rng.normal(0, 1e-3, n).astype(np.float32) for n in sizes]


def _init(sizes):
    rng = np.random.default_rng(3)
    return [rng.normal(0, 0.02, n).astype(np.float32) for n in sizes]


STEPS = 5
FOUND_INF = {3: 1}      # step -> the one rank that sees an overflow


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from compact_state_gb300.sharded import ShardLayout, exchange_step
    from oracle.adamw import new_state, oracle_step
    L = ShardLayout(SIZES, world, rank)
    flat_param = torch.zeros(L.flat_elems)
    flat_grad = torch.zeros(L.flat_elems)
    grad_shard = torch.zeros(L.shard_elems)
    for i, x in enumerate(_init(SIZES)):
        a, b = L.flat_range(i)
        flat_param[a:b] = torch.from_numpy(x)
    s0 = L.shard_start
    groups = _groups()
    states = [new_state(flat_param[L.offsets[i] + L.lo[i]:L.offsets[i] + L.hi[i]].double()
                        .numpy(), "f32", "f32", group=i % 2) for i in range(len(SIZES))]
    for step in range(1, STEPS + 1):
        for i, g in enumerate(_grads(rank, step, SIZES)):
            a, b = L.flat_range(i)
            flat_grad[a:b] = torch.from_numpy(g)
        present = _schedule(step, len(SIZES))
        fi = torch.tensor([1.0 if FOUND_INF.get(step) == rank else 0.0])

        def local(fi_all):
            grads = []
            for i in range(len(SIZES)):
                a, b = L.shard_range(i)
                grads.append(grad_shard[a:b].double().numpy() if present[i] else None)
            oracle_step(states, groups, grads, found_inf=float(fi_all.item()))
            for i, st in enumerate(states):
                a, b = L.shard_range(i)
                flat_param[s0 + a:s0 + b] = torch.from_numpy(st.theta).float()

        exchange_step(L, flat_grad, grad_shard, flat_param, fi, local)
    q.put((rank, flat_param.numpy().copy(), [st.step for st in states]))
    dist.destroy_process_group()


def test_two_gloo_ranks_equal_the_unsharded_oracle(cs):
    from oracle.adamw import new_state, oracle_step
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29700 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict((r, (fp, st)) for r, fp, st in (q.get(timeout=300) for _ in range(world)))
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    # the unsharded run: the oracle over whole tensors, gradients summed over ranks
    states = [new_state(x.astype(np.float64), "f32", "f32", group=i % 2)
              for i, x in enumerate(_init(SIZES))]
    for step in range(1, STEPS + 1):
        gs = [sum(_grads(r, step, SIZES)[i] for r in range(world)) for i in range(len(SIZES))]
        present = _schedule(step, len(SIZES))
        oracle_step(states, _groups(), [g.astype(np.float64) if p else None
                                        for g, p in zip(gs, present)],
                    found_inf=1.0 if step in FOUND_INF else 0.0)
    L = __import__("compact_state_gb300.sharded", fromlist=["ShardLayout"]).ShardLayout(
        SIZES, world, 0)
    for r in range(world):
        fp, steps = res[r]
        for i, st in enumerate(states):
            a, b = L.flat_range(i)
            assert np.array_equal(fp[a:b], st.theta.astype(np.float32)), (r, i)
        assert steps == [st.step for st in states], r
    assert res[0][1] == res[1][1]
