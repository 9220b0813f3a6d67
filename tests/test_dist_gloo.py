"""bench.py's multi-rank plumbing on CPU: world size 2 over gloo.

With N GPUs each rank runs an independent replica of the layer (no data
exchange); the bench brackets the timed region with barriers and takes the
slowest rank's time.  This test runs that reduction and barrier on two CPU
processes.
"""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        bench.barrier(w)
        slowest = bench.max_over_ranks(1.5 + r, w)
        # weak scaling: every rank processes its own batch; value uses the slowest rank
        flops = bench.step_flops(64, 256, 256, 8)
        value = w * flops / slowest
        q.put((r, w, lr, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [x[0] for x in res] == [0, 1]
    assert all(x[1] == 2 for x in res)
    assert all(x[3] == 2.5 for x in res)         # max over ranks of 1.5 + rank
    flops = 4 * 64 * 256 * 256 + 6 * 64 * 8 * 512
    assert all(abs(x[4] - 2 * flops / 2.5) < 1e-6 for x in res)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.step_flops(4096, 4096, 4096, 16) == 278_099_132_416
