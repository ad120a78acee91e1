"""The N > 1 path of bench.py on two CPU ranks (gloo): disjoint token shards,
the slowest rank's time taken by every rank, and the whole-job rate."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = 10.0 + 5.0 * rank  # rank 1 is the slow one
    slowest = bench.max_over_ranks(mine, world, torch.device("cpu"))
    first = bench.rank_first_token(rank, 1024)
    dist.barrier()
    q.put((rank, slowest, first))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_shard_tokens():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [15.0, 15.0]
    firsts = [g[2] for g in got]
    assert firsts == [0, 1024]  # shards [0, 1024) and [1024, 2048) do not overlap


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_job_rate_counts_every_rank():
    # 2 ranks x 100 steps in 50 ms (the slowest rank) -> 4000 steps/s
    assert bench.job_rate(100, 2, 50.0) == pytest.approx(4000.0)


@pytest.mark.parametrize("steps,n_inputs,chunk_max", [(20, 1024, 32), (32, 1024, 32), (1000, 1024, 32),
                                                     (1, 1, 32), (37, 896, 32), (64, 16, 8), (7, 4, 8)])
def test_graph_plan_replays_exactly_the_requested_steps(steps, n_inputs, chunk_max):
    """A timed region replays full * chunk + rem graph steps == --steps, and
    the graph variants start at distinct input offsets within n_inputs."""
    p = bench.graph_plan(steps, n_inputs, chunk_max)
    assert p["full"] * p["chunk"] + p["rem"] == steps
    assert 1 <= p["chunk"] <= chunk_max and p["rem"] < p["chunk"]
    if p["full"]:
        assert p["variants"] >= 1
        offsets = [v * p["chunk"] for v in range(p["variants"])]
        assert len(set(o % n_inputs for o in offsets)) == len(offsets) or p["variants"] == 1


def test_spread_reports_median_min_max_per_step():
    s = bench.spread([4.0, 2.0, 3.0, 10.0, 3.0], 2)
    assert s == {"repeats": 5, "ms_per_step_median": 1.5, "ms_per_step_min": 1.0, "ms_per_step_max": 5.0}
