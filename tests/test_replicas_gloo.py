"""Multi-GPU runs are replicas: each rank decodes its own requests with no
data-path collective; the bench takes the max time over ranks and sums the
tokens.  The host-side aggregation is checked here with two gloo ranks on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = [4.0, 6.5][rank]
    ms = bench.max_over_ranks(ms_local, torch.device("cpu"))
    tok = bench.replica_tokens_per_s(batch=16, world=world, ms=ms)
    lens = bench.replica_lengths(8, rank)
    q.put((rank, ms, tok, lens))
    dist.destroy_process_group()


def test_two_rank_aggregation():
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
    (r0, ms0, tok0, l0), (r1, ms1, tok1, l1) = out
    assert ms0 == ms1 == 6.5                 # the slowest replica sets the time
    assert tok0 == tok1 == pytest.approx(2 * 16 / 6.5e-3)
    assert l0 != l1 and all(16 <= x <= 4096 for x in l0 + l1)   # each replica has its own requests
