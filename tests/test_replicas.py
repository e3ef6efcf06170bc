"""Replica bookkeeping of the multi-GPU launch, on CPU with two gloo processes: every rank
decodes its own sequence (distinct seeds, no data exchange), the timed region is bracketed
by barriers and the step time is the maximum over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from query_aware_kv_gb300 import replicas
from query_aware_kv_gb300 import workloads as wl


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        ri = replicas.rank_info()
        assert (ri.rank, ri.world, ri.local) == (rank, world, rank)
        w = wl.tiny(seed=replicas.workload_seed(ri.rank))
        replicas.barrier(ri.world)
        step_us = 10.0 + 7.0 * rank            # rank 1 is the slow one
        m = replicas.max_over_ranks(step_us, ri.world)
        fingerprint = float(w.k_pool.float().sum())
        fps = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(fps, torch.tensor([fingerprint], dtype=torch.float64))
        out.put((rank, m, [float(f) for f in fps]))
    finally:
        dist.destroy_process_group()


def test_two_replicas_on_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, fps in res:
        assert m == pytest.approx(17.0)        # max over ranks, seen by every rank
        assert fps[0] != fps[1]                 # replicas decode different sequences


def test_single_process_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    ri = replicas.rank_info()
    assert (ri.rank, ri.world, ri.local) == (0, 1, 0)
    assert replicas.max_over_ranks(3.5, 1) == 3.5
    assert replicas.job_bytes_per_second(100.0, 4, 2.0) == 200.0
