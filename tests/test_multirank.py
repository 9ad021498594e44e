"""The bench's multi-rank plumbing on CPU: two gloo ranks, each with its own
batch, time reduced as the max over ranks and tokens as the sum (weak scaling)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, local, w = bench.dist_env()
    bench.init_group(w, "gloo")
    bench.barrier(w)
    t = bench.max_over_ranks(10.0 + 5.0 * r, w)
    n = bench.sum_over_ranks(256.0, w)
    # each rank draws its own batch: seed + rank
    import moe_synth as S
    x = S.gen_x(4, 128, seed=0 + r)
    xs = [torch.zeros_like(x) for _ in range(w)]
    dist.all_gather(xs, x)
    q.put((r, local, w, t, n, not torch.equal(xs[0], xs[1])))
    dist.destroy_process_group()


def test_two_ranks_weak_scaling_reductions():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, local, world, t, n, distinct) in enumerate(out):
        assert (rank, local, world) == (r, r, 2)
        assert t == 15.0          # the slowest rank's time
        assert n == 512.0         # tokens of all ranks
        assert distinct           # ranks hold different batches
