"""Host logic of the multi-rank benchmark on CPU: two gloo ranks.

Every rank decodes its own layers (weak scaling: the units are independent
(sequence, layer) decode steps, no collective on the data path); the only
exchange is the max over ranks of the timed region."""
import os
import socket

import pytest


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import json
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        layers = bench.rank_layers(rank, world, 4)
        plan = bench.step_plan(rank, 10, 4)
        bench.barrier(world)
        # every rank times something different; the reported time is the max
        t = bench.max_over_ranks(1.5 + rank, world, None)
        gathered = [None] * world
        dist.all_gather_object(gathered, layers)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"layers": layers, "plan": plan, "t": t,
                       "all_layers": gathered}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    import json
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r in res:
        assert r["t"] == pytest.approx(2.5)           # max over ranks
        assert len(r["plan"]) == 10
        assert sorted({s for (_, s) in r["plan"]}) == list(range(10))
        assert {L for (L, _) in r["plan"]} == {0, 1, 2, 3}
    l0, l1 = res[0]["all_layers"]
    assert l0 == res[0]["layers"] and l1 == res[1]["layers"]
    assert not set(l0) & set(l1)                       # disjoint work units
    assert len(set(l0)) == 4 and len(set(l1)) == 4


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)
    assert bench.rank_layers(0, 1, 3) == [0, 1, 2]
