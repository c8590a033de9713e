"""Head-sharded tensor parallelism through the C ABI on one GPU (attn_create_shard).

The shards of a 2-, 4- and 8-way split (and an uneven 3 + 5 split) run one after another on
the same GPU, each with its own weight shards and its own kv cache; their partial Delta_attn
are summed in fp64 on the host (standing in for the row-parallel projection's all-reduce) and
compared element by element with the fp64 oracle of the whole block at the block's tolerance.
Each shard's cache entries, rotated queries and head outputs are checked against the
oracle's for its heads."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import gqa_oracle as orc
from tests import gpu_util as gu
from transformer_gqa_attention_gb300 import abi
from transformer_gqa_attention_gb300 import inputs as gin
from transformer_gqa_attention_gb300 import tp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from transformer_gqa_attention_gb300 import _build
    _build.build()


def _splits(world):
    return [tp.kv_group_range(r, world) for r in range(world)]


class Shard:
    def __init__(self, inp, g0, n):
        self.g0, self.n = g0, n
        self.w = [t.to(gu.DEV) for t in tp.shard_weights(inp.wq, inp.wk, inp.wv, inp.wo, g0, n)]
        self.ctx = abi.attn_create_shard(*self.w, n)
        abi.attn_sync_status(self.ctx)

    def close(self):
        abi.attn_destroy(self.ctx)


def _shard_cache(B, S_max, n):
    shape = (B, S_max, n, 128)
    return (torch.full(shape, float("nan"), dtype=torch.bfloat16, device=gu.DEV),
            torch.full(shape, float("nan"), dtype=torch.bfloat16, device=gu.DEV))


def _run_prefill_and_decode(inp, splits, decode=True):
    B, T = inp.x.shape[:2]
    S_max = T + 1
    x, R = inp.x.to(gu.DEV), inp.R.to(gu.DEV)
    w64 = [gin.to_f64(t) for t in (inp.wq, inp.wk, inp.wv, inp.wo)]
    ref, ex = orc.attention_block(gin.to_f64(inp.x), *w64, gin.to_f64(inp.R), keep=True)
    # the next token of each sequence, decoded against the caches the prefill filled
    x1 = torch.randn(B, 1, 4096, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    R1 = gin.rope_table([T])
    cache_k = np.zeros((B, S_max, 8, 128))
    cache_v = np.zeros((B, S_max, 8, 128))
    cache_k[:, :T] = ex["K_r"]
    cache_v[:, :T] = ex["V"]
    ref1, _ = orc.attention_decode(gin.to_f64(x1), *w64, gin.to_f64(R1), cache_k, cache_v, T)

    total = np.zeros(ref.shape)
    total1 = np.zeros(ref1.shape)
    for g0, n in splits:
        sh = Shard(inp, g0, n)
        try:
            ck, cv = _shard_cache(B, S_max, n)
            delta = torch.empty(B, T, 4096, dtype=torch.float32, device=gu.DEV)
            abi.attn_prefill(sh.ctx, x, B, T, R, True, ck, cv, S_max, 0, delta)
            abi.attn_sync_status(sh.ctx)
            total += gu.np64(delta)
            what = f"shard g{g0}+{n}"
            gu.assert_close(gu.np64(ck[:, :T]), ex["K_r"][:, :, g0:g0 + n], gu.TOL_BF16_REL_L1, gu.TOL_BF16_MAX,
                            what + " K_r")
            gu.assert_close(gu.np64(cv[:, :T]), ex["V"][:, :, g0:g0 + n], gu.TOL_BF16_REL_L1, gu.TOL_BF16_MAX,
                            what + " V")
            q_ptr, h_ptr = abi.attn_debug_buffers(sh.ctx)
            q_r = gu.np64(gu.device_view(q_ptr, (B * T, 512 * n))).reshape(B, T, 4 * n, 128)
            h = gu.np64(gu.device_view(h_ptr, (B * T, 512 * n))).reshape(B, T, 512 * n)
            gu.assert_close(q_r, ex["Q_r"][:, :, 4 * g0:4 * (g0 + n)], gu.TOL_BF16_REL_L1, gu.TOL_BF16_MAX,
                            what + " Q_r")
            gu.assert_close(h, ex["H"][:, :, 512 * g0:512 * (g0 + n)], gu.TOL_REL_L1, gu.TOL_MAX, what + " H")
            if decode:
                d1 = torch.empty(B, 1, 4096, dtype=torch.float32, device=gu.DEV)
                abi.attn_decode(sh.ctx, x1.to(gu.DEV), B, T, R1.to(gu.DEV), ck, cv, S_max, d1)
                abi.attn_sync_status(sh.ctx)
                total1 += gu.np64(d1)
        finally:
            sh.close()
    gu.assert_close(total, ref, what=f"sum of {len(splits)} shard partials (prefill)")
    if decode:
        gu.assert_close(total1, ref1, what=f"sum of {len(splits)} shard partials (decode)")


@pytest.mark.parametrize("world", [2, 4, 8])
def test_shard_partials_sum_to_the_block(world):
    _run_prefill_and_decode(gin.make_custom(seed=90 + world, B=2, T=300), _splits(world))


def test_uneven_shards_sum_to_the_block():
    _run_prefill_and_decode(gin.make_custom(seed=95, B=1, T=200), [(0, 3), (3, 5)])


def test_few_token_shards_sum_to_the_block():
    # 16 tokens: the split-K projection kernels, with the shards' narrower weights
    _run_prefill_and_decode(gin.make_custom(seed=96, B=1, T=16), _splits(2))


def test_whole_shard_equals_the_block_context():
    inp = gin.make_custom(seed=97, B=1, T=130)
    _run_prefill_and_decode(inp, [(0, 8)], decode=False)


def test_residual_form_is_rejected_on_a_shard():
    inp = gin.make_custom(seed=98, B=1, T=4)
    sh = Shard(inp, 0, 4)
    try:
        w = torch.ones(4096, dtype=torch.bfloat16, device=gu.DEV)
        assert abi.raw_status("attn_set_norm", sh.ctx, w.data_ptr(), ctypes.c_float(1e-5), None) == 1
    finally:
        sh.close()


def test_shard_chunked_prefill_and_large_decode_batch():
    # a 2-way split: each shard prefills 150 positions, then continues with 100 more at
    # start_pos = 150 against its own cache; then a decode of 80 sequences (more than 64
    # tokens: the many-token projection kernels) on a filled cache
    B, T1, T2 = 2, 150, 100
    inp = gin.make_custom(seed=99, B=B, T=T1 + T2)
    w64 = [gin.to_f64(t) for t in (inp.wq, inp.wk, inp.wv, inp.wo)]
    ref, _ = orc.attention_block(gin.to_f64(inp.x), *w64, gin.to_f64(inp.R))
    Bd, pos, S_d = 80, 300, 320
    dec = gin.make_custom(seed=100, B=Bd, T=1, start_pos=pos, S_max=S_d, fill_cache=True)
    wd64 = [gin.to_f64(t) for t in (dec.wq, dec.wk, dec.wv, dec.wo)]
    ref_d, _ = orc.attention_decode(gin.to_f64(dec.x), *wd64, gin.to_f64(dec.R), gin.to_f64(dec.cache_k),
                                    gin.to_f64(dec.cache_v), pos)
    total = np.zeros(ref.shape)
    total_d = np.zeros(ref_d.shape)
    for g0, n in _splits(2):
        sh = Shard(inp, g0, n)
        try:
            ck, cv = _shard_cache(B, T1 + T2, n)
            for t0, t1 in ((0, T1), (T1, T1 + T2)):
                d = torch.empty(B, t1 - t0, 4096, dtype=torch.float32, device=gu.DEV)
                abi.attn_prefill(sh.ctx, inp.x[:, t0:t1].contiguous().to(gu.DEV), B, t1 - t0,
                                 inp.R[t0:t1].contiguous().to(gu.DEV), True, ck, cv, T1 + T2, t0, d)
                abi.attn_sync_status(sh.ctx)
                total[:, t0:t1] += gu.np64(d)
        finally:
            sh.close()
        shd = Shard(dec, g0, n)
        try:
            ck = dec.cache_k[:, :, g0:g0 + n].contiguous().to(gu.DEV)
            cv = dec.cache_v[:, :, g0:g0 + n].contiguous().to(gu.DEV)
            d = torch.empty(Bd, 1, 4096, dtype=torch.float32, device=gu.DEV)
            abi.attn_decode(shd.ctx, dec.x.to(gu.DEV), Bd, pos, dec.R.to(gu.DEV), ck, cv, S_d, d)
            abi.attn_sync_status(shd.ctx)
            total_d += gu.np64(d)
        finally:
            shd.close()
    gu.assert_close(total, ref, what="chunked prefill, sum of 2 shard partials")
    gu.assert_close(total_d, ref_d, what="decode B=80, sum of 2 shard partials")


@pytest.mark.parametrize("name", ["prefill_b1_t32768_tp8", "prefill_b1_t32768_tp2", "prefill_b1_t2048_tp8"])
def test_shard_prefill_workloads_full_size_sampled_rows(name):
    # one rank of the split as bench.py times it: kv groups 0 .. n-1 of the workload's
    # weights, a cache of n groups; its partial Delta on sampled query rows against the
    # oracle run with the same shard (4 n query heads, n kv heads)
    w = gin.WORKLOADS[name]
    inp = gin.make_inputs(name)
    n = w.n_kv
    sh = Shard(inp, 0, n)
    try:
        B, T = inp.x.shape[:2]
        ck, cv = _shard_cache(B, T, n)
        delta = torch.empty(B, T, 4096, dtype=torch.float32, device=gu.DEV)
        abi.attn_prefill(sh.ctx, inp.x.to(gu.DEV), B, T, inp.R.to(gu.DEV), True, ck, cv, T, 0, delta)
        abi.attn_sync_status(sh.ctx)
        rows = gu.sample_rows(T)
        w64 = [gin.to_f64(t) for t in tp.shard_weights(inp.wq, inp.wk, inp.wv, inp.wo, 0, n)]
        ref, _ = orc.attention_block(gin.to_f64(inp.x), *w64, gin.to_f64(inp.R), rows=rows, n_heads=4 * n)
        gu.assert_close(gu.np64(delta[:, rows]), ref, what=f"{name} partial delta rows")
    finally:
        sh.close()


def test_shard_decode_workload_full_size_sampled_sequences():
    name = "decode_b64_pos4095_tp8"
    w = gin.WORKLOADS[name]
    inp = gin.make_inputs(name)
    n, pos = w.n_kv, w.start_pos
    sh = Shard(inp, 0, n)
    try:
        ck = inp.cache_k[:, :, :n].contiguous().to(gu.DEV)
        cv = inp.cache_v[:, :, :n].contiguous().to(gu.DEV)
        d = torch.empty(w.B, 1, 4096, dtype=torch.float32, device=gu.DEV)
        abi.attn_decode(sh.ctx, inp.x.to(gu.DEV), w.B, pos, inp.R.to(gu.DEV), ck, cv, w.s_max, d)
        abi.attn_sync_status(sh.ctx)
        w64 = [gin.to_f64(t) for t in tp.shard_weights(inp.wq, inp.wk, inp.wv, inp.wo, 0, n)]
        for b in (0, 31, 63):
            ref, _ = orc.attention_decode(gin.to_f64(inp.x[b:b + 1]), *w64, gin.to_f64(inp.R),
                                          gin.to_f64(inp.cache_k[b:b + 1, :, :n]),
                                          gin.to_f64(inp.cache_v[b:b + 1, :, :n]), pos, n_heads=4 * n)
            gu.assert_close(gu.np64(d[b:b + 1]), ref, what=f"{name} partial delta, sequence {b}")
    finally:
        sh.close()
