"""The N > 1 path of bench.py on CPU: world_size 2 over gloo (no GPU).  Each
rank is a replica of the batch; the job's step time is the slowest rank's
and the throughput counts every rank's units."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from paged_kv_cache_125_gb300 import workloads as W
    r, w, local = bench.dist_info()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(world)
    ms = 1.0 + rank  # rank 1 is the slow one
    value, ms_job = bench.aggregate(1000.0, ms, world, device="cpu")
    # every replica builds the identical seeded batch
    m = W.config2_decode().steps[0].attn.meta
    digest = int(m.context_lens.sum()) * 1_000_003 + int(m.block_tables[:, 0].sum())
    dg = torch.tensor([digest], dtype=torch.int64)
    gathered = [torch.zeros_like(dg) for _ in range(world)]
    dist.all_gather(gathered, dg)
    out[rank] = (value, ms_job, len({int(g) for g in gathered}))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    for r in range(world):
        value, ms_job, distinct = out[r]
        assert ms_job == pytest.approx(2.0)
        assert value == pytest.approx(1000.0 * 2 / 2e-3)
        assert distinct == 1
