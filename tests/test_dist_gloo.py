"""The multi-GPU (owner-sharded) path's host logic on CPU: two gloo ranks each
take their share of the owner plan through the C ABI; the shares are disjoint,
cover the set, and the timing reductions bench.py uses give max / sum."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    import matrix_optimizers_gb300 as mo
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        shapes, idx, _ = bench.workload_shapes("llama7b_owner0", rank, world, mo.plan_owners)
        gathered = [None] * world
        dist.all_gather_object(gathered, idx)
        mx = bench._max_over_ranks(float(rank + 1), dist)
        sm = bench._sum_over_ranks(float(len(idx)), dist)
        out_q.put((rank, gathered, mx, sm, len(shapes)))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_owner_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, gathered, mx, sm, n in results:
        a, b = set(gathered[0]), set(gathered[1])
        assert not (a & b)
        assert len(gathered[0]) == len(gathered[1]) == 28     # shares of the 8-rank plan
        assert mx == 2.0 and sm == 56.0 and n == 224
