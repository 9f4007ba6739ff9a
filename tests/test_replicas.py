"""Host logic of the N>1 path (replicas, no data-path collective), run as two gloo ranks
on the CPU: environment parsing, per-rank sharding of the sequences, the barrier and the
max-over-ranks time from which the job's aggregate throughput is computed."""
import socket

import pytest
import torch.multiprocessing as mp

from block_diffusion_drafter_concat_gb300 import replicas
from workload import configs, inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import os

    import torch.distributed as dist
    env = {"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)}
    os.environ.update(env, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    rep = replicas.from_env(env)
    dist.init_process_group("gloo", rank=rep.rank, world_size=rep.world)
    try:
        replicas.barrier(rep)
        mine = 0.5 + rep.rank          # rank r "took" 0.5 + r seconds
        slowest = replicas.max_over_ranks(rep, mine)
        value = replicas.aggregate(100, rep, slowest)
        w = replicas.shard(configs.QWEN3_8B_B1, rep.rank)
        ws = replicas.shard(configs.small_bf16(), rep.rank)
        wt = inputs.weights(ws)
        digest = float(sum(t.float().sum() for t in wt.values()))
        lens = inputs.ctx_lens(ws).tolist()
        x0 = float(inputs.ctx_hidden(ws, 0, 0, 4).float().sum())
        replicas.barrier(rep)
        out.put((rep.rank, slowest, value, w.seed, w.rows, digest, lens, x0))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(out.get(timeout=10) for _ in range(world))
    slowest = 0.5 + (world - 1)
    for rank, t, value, seed, rows, _, _, _ in res:
        assert t == pytest.approx(slowest)          # every rank sees the max, not its own
        assert value == pytest.approx(100 * world / slowest)
        assert rows == configs.QWEN3_8B_B1.rows
        assert seed == configs.QWEN3_8B_B1.seed     # one weight seed on every rank
    # replicas share the weights but draft different sequences
    assert res[0][5] == res[1][5]
    assert res[0][6] != res[1][6] and res[0][7] != res[1][7]
    assert res[0][6] == inputs.ctx_lens(configs.small_bf16()).tolist()


def test_single_process_needs_no_process_group():
    rep = replicas.from_env({})
    assert rep == replicas.Replica(0, 1, 0) and not rep.distributed
    replicas.barrier(rep)
    assert replicas.max_over_ranks(rep, 1.25) == 1.25
    assert replicas.aggregate(10, rep, 2.0) == 5.0


@pytest.mark.parametrize("env", [{"RANK": "2", "WORLD_SIZE": "2"},
                                 {"RANK": "-1", "WORLD_SIZE": "2"},
                                 {"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "-3"}])
def test_bad_coordinates_are_rejected(env):
    with pytest.raises(ValueError):
        replicas.from_env(env)


def test_aggregate_rejects_a_nonpositive_time():
    with pytest.raises(ValueError):
        replicas.aggregate(1, replicas.Replica(0, 2, 0), 0.0)
