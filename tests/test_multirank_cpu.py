"""The N>1 path on CPU: two gloo ranks shard the batch by request with no
data-path collective, and the benchmark's timing reduction takes the max
over ranks (its only collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, num_requests, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist
    import bench
    from linear_attention_recurrent_gdn_gb300.sharding import shard_requests, slots_of_requests
    r, w, d = bench.dist_setup("cpu")
    assert (r, w) == (rank, world)
    mine = list(shard_requests(num_requests, world, rank))
    gathered = [None] * world
    dist.all_gather_object(gathered, mine)
    t = bench.reduce_max(d, 10.0 + rank, torch.device("cpu"))
    r_slots, b_slots = slots_of_requests(mine, 8)
    out[rank] = (gathered, t, len(r_slots), sum(len(b) for b in b_slots))
    bench.barrier(d)
    dist.destroy_process_group()


@pytest.mark.parametrize("num_requests", [64, 7])
def test_two_gloo_ranks_shard_and_reduce(num_requests):
    world = 2
    ctx = mp.get_context("spawn")     # no fork after threads (the manager too)
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, num_requests, out))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    shards = out[0][0]
    flat = [x for s in shards for x in s]
    assert sorted(flat) == list(range(num_requests))          # complete and disjoint
    assert all(out[r][1] == 11.0 for r in range(world))       # max over ranks
    for r in range(world):
        assert out[r][3] == 8 * out[r][2]                     # branches stay with requests
