"""Seeded sweeps over the prefill and decode parameter spaces through the C ABI against the
fp64 oracle.

Each case draws (B, T, start_pos, causal, kv-group shard) at random from one seeded
generator: a context over kv groups g0 .. g0+n-1 (the whole block when n = 8) fills its cache
with a first prefill of start_pos positions, then prefills T more positions continuing it
(causal or not); the second call's Delta (the shard's partial for n < 8) is compared with the
oracle run on the same weights and the whole sequence, on that call's rows.  T spans the
short-prefill kernel (T <= 16), one ragged flash tile and several tiles; start_pos spans
zero, values inside the first key tile and across tiles."""
import numpy as np
import pytest
import torch

from oracle import gqa_oracle as orc
from tests import gpu_util as gu
from transformer_gqa_attention_gb300 import abi
from transformer_gqa_attention_gb300 import inputs as gin
from transformer_gqa_attention_gb300 import tp

pytestmark = pytest.mark.gpu

N_CASES = 24


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from transformer_gqa_attention_gb300 import _build
    _build.build()


def _cases():
    rng = np.random.default_rng(2024)
    out = []
    for i in range(N_CASES):
        n = int(rng.choice([8, 8, 4, 2, 1]))
        g0 = int(rng.integers(0, 8 // n)) * n
        T = int(rng.choice([1, 3, 8, 16, 17, 64, 130, 257]))
        start_pos = int(rng.choice([0, 0, 5, 63, 64, 200]))
        B = int(rng.integers(1, 4))
        causal = bool(rng.random() < 0.75)
        out.append((i, B, T, start_pos, causal, g0, n))
    return out


@pytest.mark.parametrize("i,B,T,start_pos,causal,g0,n", _cases())
def test_prefill_sweep(i, B, T, start_pos, causal, g0, n):
    full = gin.make_custom(seed=500 + i, B=B, T=start_pos + T)
    ws = tp.shard_weights(full.wq, full.wk, full.wv, full.wo, g0, n)
    wd = [t.to(gu.DEV) for t in ws]
    ctx = abi.attn_create(*wd) if n == 8 else abi.attn_create_shard(*wd, n)
    try:
        S_max = start_pos + T
        shape = (B, S_max, n, 128)
        ck = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=gu.DEV)
        cv = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=gu.DEV)
        x, R = full.x.to(gu.DEV), full.R.to(gu.DEV)
        if start_pos:
            d0 = torch.empty(B, start_pos, 4096, dtype=torch.float32, device=gu.DEV)
            abi.attn_prefill(ctx, x[:, :start_pos].contiguous(), B, start_pos, R[:start_pos].contiguous(), True,
                             ck, cv, S_max, 0, d0)
        d = torch.empty(B, T, 4096, dtype=torch.float32, device=gu.DEV)
        abi.attn_prefill(ctx, x[:, start_pos:].contiguous(), B, T, R[start_pos:].contiguous(), causal, ck, cv,
                         S_max, start_pos, d)
        abi.attn_sync_status(ctx)
        w64 = [gin.to_f64(t) for t in ws]
        rows = np.arange(start_pos, start_pos + T)
        if causal:
            ref, _ = orc.attention_block(gin.to_f64(full.x), *w64, gin.to_f64(full.R), rows=rows, n_heads=4 * n)
        else:
            # a non-causal chunk sees every cached key and all of its own positions: the
            # causal prefix fill leaves the same keys and values, so the oracle's non-causal
            # block over the whole sequence gives the chunk's rows
            ref, _ = orc.attention_block(gin.to_f64(full.x), *w64, gin.to_f64(full.R), rows=rows, causal=False,
                                         n_heads=4 * n)
        gu.assert_close(gu.np64(d), ref,
                        what=f"case {i}: B={B} T={T} start_pos={start_pos} causal={causal} groups {g0}+{n}")
    finally:
        abi.attn_destroy(ctx)


def _decode_cases():
    rng = np.random.default_rng(2025)
    out = []
    for i in range(12):
        n = int(rng.choice([8, 8, 4, 1]))
        g0 = int(rng.integers(0, 8 // n)) * n
        B = int(rng.choice([1, 5, 32, 33, 64, 80]))
        pos = int(rng.choice([0, 1, 63, 64, 500, 2100]))
        out.append((i, B, pos, g0, n))
    return out


@pytest.mark.parametrize("i,B,pos,g0,n", _decode_cases())
def test_decode_sweep(i, B, pos, g0, n):
    # one decode step at position pos against a cache holding positions < pos (drawn): the
    # batch crosses the 32-token and 64-token projection kernels and the many-token path
    # (B = 80), the cache length crosses the 64-key tile and several key splits
    S_max = pos + 1
    inp = gin.make_custom(seed=600 + i, B=B, T=1, start_pos=pos, S_max=S_max, fill_cache=True)
    ws = tp.shard_weights(inp.wq, inp.wk, inp.wv, inp.wo, g0, n)
    wd = [t.to(gu.DEV) for t in ws]
    ctx = abi.attn_create(*wd) if n == 8 else abi.attn_create_shard(*wd, n)
    try:
        ck = inp.cache_k[:, :, g0:g0 + n].contiguous().to(gu.DEV)
        cv = inp.cache_v[:, :, g0:g0 + n].contiguous().to(gu.DEV)
        d = torch.empty(B, 1, 4096, dtype=torch.float32, device=gu.DEV)
        abi.attn_decode(ctx, inp.x.to(gu.DEV), B, pos, inp.R.to(gu.DEV), ck, cv, S_max, d)
        abi.attn_sync_status(ctx)
        w64 = [gin.to_f64(t) for t in ws]
        ref, _ = orc.attention_decode(gin.to_f64(inp.x), *w64, gin.to_f64(inp.R),
                                      gin.to_f64(inp.cache_k[:, :, g0:g0 + n]),
                                      gin.to_f64(inp.cache_v[:, :, g0:g0 + n]), pos, n_heads=4 * n)
        gu.assert_close(gu.np64(d), ref, what=f"decode case {i}: B={B} pos={pos} groups {g0}+{n}")
    finally:
        abi.attn_destroy(ctx)
