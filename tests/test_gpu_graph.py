"""The block's calls captured in a CUDA graph and replayed (GPU).

A decode loop or a fixed-shape prefill can be recorded once and replayed to take the host's
launch work off the critical path.  The library's calls are asynchronous on the caller's
stream and allocate nothing once the context's workspace has reached the call's size, so
after one warm-up call at that size they can be captured; their kernels are launched with
programmatic dependent launch, which the graph keeps as programmatic edges.  Each replay is
checked against the fp64 oracle."""
import numpy as np
import pytest
import torch

from oracle import gqa_oracle as orc
from tests import gpu_util as gu
from transformer_gqa_attention_gb300 import abi
from transformer_gqa_attention_gb300 import inputs as gin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from transformer_gqa_attention_gb300 import _build
    _build.build()


def test_decode_step_replayed_from_a_cuda_graph():
    B, pos, S_max = 8, 700, 768
    inp = gin.make_custom(seed=81, B=B, T=1, start_pos=pos, S_max=S_max, fill_cache=True)
    blk = gu.Block(inp)
    try:
        x, R = inp.x.to(gu.DEV), inp.R.to(gu.DEV)
        ck, cv = inp.cache_k.to(gu.DEV), inp.cache_v.to(gu.DEV)
        delta = torch.empty(B, 1, 4096, dtype=torch.float32, device=gu.DEV)
        abi.attn_decode(blk.ctx, x, B, pos, R, ck, cv, S_max, delta)  # sizes the workspace
        abi.attn_sync_status(blk.ctx)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            abi.attn_decode(blk.ctx, x, B, pos, R, ck, cv, S_max, delta)
        wq, wk, wv, wo = blk.w64
        ref, _ = orc.attention_decode(gin.to_f64(inp.x), wq, wk, wv, wo, gin.to_f64(inp.R),
                                      gin.to_f64(inp.cache_k), gin.to_f64(inp.cache_v), pos)
        for _ in range(3):
            delta.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            abi.attn_sync_status(blk.ctx)
            gu.assert_close(gu.np64(delta), ref, what="graph replay of a decode step")
    finally:
        blk.close()


def test_prefill_replayed_from_a_cuda_graph():
    B, T = 2, 300
    inp = gin.make_custom(seed=82, B=B, T=T)
    blk = gu.Block(inp)
    try:
        x, R = inp.x.to(gu.DEV), inp.R.to(gu.DEV)
        ck, cv = gu.empty_cache(B, T)
        delta = torch.empty(B, T, 4096, dtype=torch.float32, device=gu.DEV)
        abi.attn_prefill(blk.ctx, x, B, T, R, True, ck, cv, T, 0, delta)  # sizes the workspace
        abi.attn_sync_status(blk.ctx)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            abi.attn_prefill(blk.ctx, x, B, T, R, True, ck, cv, T, 0, delta)
        ref, _ = gu.oracle_prefill(blk, inp)
        for _ in range(2):
            delta.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            abi.attn_sync_status(blk.ctx)
            gu.assert_close(gu.np64(delta), ref, what="graph replay of a prefill")
    finally:
        blk.close()
