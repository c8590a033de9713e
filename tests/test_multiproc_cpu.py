"""The N > 1 path of bench.py on CPU: two gloo ranks run the same helpers the GPU ranks use
(rendezvous from the environment, barrier, max over ranks).  The block itself shards as
independent replicas (weak scaling) and has no collective on its data path."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup(world)
    assert (w, r, local) == (world, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(w)
        # each rank reports a different step time; every rank must see the maximum
        t = bench.max_over_ranks(1.0 + rank, w, torch.device("cpu"))
        out[rank] = t
        bench.barrier(w)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_step_time():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.0, 1: 2.0}


def test_gpus_flag_without_launcher_is_rejected(monkeypatch):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "1")
    with pytest.raises(SystemExit):
        bench.dist_setup(2)
