"""Head-sharded tensor parallelism on the CPU: the partition of the kv groups over ranks, the
weight shards, and the sum all-reduce over two gloo ranks, each computing its shard's partial
Delta_attn with the fp64 oracle.  The sum of the partials must be the block's Delta_attn (the
row-parallel output projection's reduction), which pins the partition independently of any
GPU code."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import gqa_oracle as orc
from transformer_gqa_attention_gb300 import inputs as gin
from transformer_gqa_attention_gb300 import tp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [1, 2, 4, 8])
def test_kv_group_ranges_partition_the_groups(world):
    owned = []
    for rank in range(world):
        g0, n = tp.kv_group_range(rank, world)
        assert n == 8 // world
        owned += list(range(g0, g0 + n))
    assert owned == list(range(8))


@pytest.mark.parametrize("world,rank", [(3, 0), (16, 0), (2, 2), (0, 0)])
def test_kv_group_range_rejects_uneven_or_bad_worlds(world, rank):
    with pytest.raises(ValueError):
        tp.kv_group_range(rank, world)


def test_shards_reassemble_the_weights():
    gen = torch.Generator().manual_seed(3)
    wq, wk, wv, wo = gin.make_weights(gen)
    parts = [tp.shard_weights(wq, wk, wv, wo, *tp.kv_group_range(r, 4)) for r in range(4)]
    assert parts[1][0].shape == (1024, 4096) and parts[1][1].shape == (256, 4096)
    assert parts[1][3].shape == (4096, 1024) and parts[1][3].is_contiguous()
    assert torch.equal(torch.cat([p[0] for p in parts], 0), wq)
    assert torch.equal(torch.cat([p[1] for p in parts], 0), wk)
    assert torch.equal(torch.cat([p[2] for p in parts], 0), wv)
    assert torch.equal(torch.cat([p[3] for p in parts], 1), wo)


def _partial_delta(inp, g0, n, **kw):
    """The oracle's Delta_attn of kv groups g0 .. g0+n-1 alone (their 4 n query heads)."""
    wq, wk, wv, wo = (gin.to_f64(t) for t in tp.shard_weights(inp.wq, inp.wk, inp.wv, inp.wo, g0, n))
    delta, _ = orc.attention_block(gin.to_f64(inp.x), wq, wk, wv, wo, gin.to_f64(inp.R), n_heads=4 * n, **kw)
    return delta


def test_partials_of_every_split_sum_to_the_block():
    inp = gin.make_custom(seed=31, B=2, T=9)
    w64 = [gin.to_f64(t) for t in (inp.wq, inp.wk, inp.wv, inp.wo)]
    ref, _ = orc.attention_block(gin.to_f64(inp.x), *w64, gin.to_f64(inp.R))
    for split in ([8], [4, 4], [2, 2, 2, 2], [1] * 8, [3, 5]):
        total = np.zeros_like(ref)
        g0 = 0
        for n in split:
            total += _partial_delta(inp, g0, n)
            g0 += n
        np.testing.assert_allclose(total, ref, rtol=0, atol=1e-12 * np.abs(ref).max())
    # one shard alone is not the block
    assert np.abs(_partial_delta(inp, 0, 4) - ref).max() > 1e-3 * np.abs(ref).max()


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.set_num_threads(2)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = gin.make_custom(seed=32, B=1, T=7)
        g0, n = tp.kv_group_range(rank, world)
        delta = torch.from_numpy(_partial_delta(inp, g0, n))
        tp.all_reduce_delta(delta)
        w64 = [gin.to_f64(t) for t in (inp.wq, inp.wk, inp.wv, inp.wo)]
        ref, _ = orc.attention_block(gin.to_f64(inp.x), *w64, gin.to_f64(inp.R))
        out[rank] = float(np.abs(delta.numpy() - ref).max() / np.abs(ref).max())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_all_reduce_their_partials_into_the_block():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    assert sorted(out.keys()) == [0, 1]
    assert max(out.values()) < 1e-12
