"""Host logic of the multi-rank bench path on CPU: two gloo ranks agree on the
maximum time (the slowest rank sets the job time) and pass the barriers."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    r, w, _ = bench.dist_setup()
    assert (r, w) == (rank, world)
    bench.dist_barrier(w)
    out[rank] = bench.dist_max(10.0 + 5.0 * rank, w)
    bench.dist_barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_is_identity():
    import bench
    assert bench.dist_max(3.5, 1) == 3.5


# ---------------------------------------------------------------- sharded step (host logic)

def test_assign_balances_work_deterministically():
    from tiled_newton_schulz_03_b300 import shard, synth
    shapes = synth.llama3_8b_shapes()
    for world in (1, 2, 4, 8):
        owner = shard.assign(shapes, world, 128, 5)
        assert owner == shard.assign(shapes, world, 128, 5)
        load = [0.0] * world
        for (H, W), r in zip(shapes, owner):
            load[r] += H * W
        assert max(load) <= 1.02 * (sum(load) / world)      # within 2 % of even


def _shard_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    from tiled_newton_schulz_03_b300 import shard
    dist.init_process_group("gloo", rank=rank, world_size=world)
    shapes = [(8, 8), (4, 16), (16, 4), (2, 2), (8, 4)]
    Ws = [torch.full(s, -1.0) for s in shapes]
    Gs = [torch.full(s, float(i)) for i, s in enumerate(shapes)]
    Ms = [torch.zeros(s) for s in shapes]
    calls = []

    def fake_step(W, G, M):            # stands in for the GPU step: W <- 10 * G + owner
        calls.append(len(W))
        for w, g, m in zip(W, G, M):
            w.copy_(10 * g + rank)
            m.add_(g)

    st = shard.ShardedStep(shapes, 4, 5, fake_step)
    st(Ws, Gs, Ms)
    out[rank] = ([w.flatten()[0].item() for w in Ws], st.owner, sum(calls),
                 [m.flatten()[0].item() for m in Ms])
    dist.destroy_process_group()


def test_sharded_step_two_gloo_ranks_get_the_owners_weights():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    w0, owner, n0, m0 = out[0]
    w1, _, n1, m1 = out[1]
    assert w0 == w1                                           # every rank holds the same W
    assert w0 == [10.0 * i + owner[i] for i in range(5)]      # each from its owner
    assert n0 + n1 == 5 and n0 > 0 and n1 > 0                 # each matrix stepped once
    for i in range(5):                                        # momentum only at the owner
        assert (m0[i], m1[i]) == ((float(i), 0.0) if owner[i] == 0 else (0.0, float(i)))
