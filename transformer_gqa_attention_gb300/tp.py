"""Head-sharded tensor parallelism of the block: partition bookkeeping and the sum all-reduce.

The quoted Llama code splits the attention block over model-parallel ranks by heads (page
"Llama 3.1 8B · Grouped-query attention", Query projection: n_local_heads = n_heads /
model_parallel_size, n_local_kv_heads = n_kv_heads / model_parallel_size; W_Q, W_K, W_V are
ColumnParallelLinear(gather_output=False) layers), and the output projection is a
RowParallelLinear(input_is_parallel=True) (page "Llama 3.1 8B · Merge and project"): each
rank multiplies its own heads' H by its own columns of W_O, and the ranks' partial results
are summed across ranks.  The sum itself is not printed on the pages; a RowParallelLinear
reduces its output over the model-parallel group, which is read here as a sum all-reduce.

This module holds no arithmetic of the block: it only decides which kv groups a rank owns,
cuts the weights accordingly (the shards the library's attn_create_shard takes) and calls
the collective that sums the partial Delta_attn.
"""
from __future__ import annotations

import torch

N_KV_HEADS = 8
N_REP = 4  # query heads per kv group
HEAD_DIM = 128


def kv_group_range(rank: int, world: int, n_kv: int = N_KV_HEADS) -> tuple[int, int]:
    """(first kv group, number of kv groups) of `rank` among `world` ranks: contiguous,
    balanced ranges (world must divide n_kv, as n_kv_heads // model_parallel_size needs)."""
    if world < 1 or n_kv % world != 0 or not 0 <= rank < world:
        raise ValueError(f"cannot split {n_kv} kv groups over {world} ranks (rank {rank})")
    n = n_kv // world
    return rank * n, n


def shard_weights(wq, wk, wv, wo, g0: int, n: int):
    """The weights of kv groups g0 .. g0+n-1 in the layouts attn_create_shard takes:
    W_Q rows of query heads 4 g0 .. 4 (g0+n) - 1 ([512 n, dim], the column-parallel shard),
    W_K / W_V rows of kv heads g0 .. g0+n-1 ([128 n, dim]), and W_O columns of those query
    heads ([dim, 512 n], the row-parallel shard), each made contiguous."""
    q0, q1 = g0 * N_REP * HEAD_DIM, (g0 + n) * N_REP * HEAD_DIM
    k0, k1 = g0 * HEAD_DIM, (g0 + n) * HEAD_DIM
    return (wq[q0:q1].contiguous(), wk[k0:k1].contiguous(), wv[k0:k1].contiguous(),
            wo[:, q0:q1].contiguous())


def all_reduce_delta(delta_partial: torch.Tensor, group=None) -> torch.Tensor:
    """Sum the ranks' partial Delta_attn in place (the row-parallel projection's reduction)
    and return it."""
    torch.distributed.all_reduce(delta_partial, op=torch.distributed.ReduceOp.SUM, group=group)
    return delta_partial
