"""Failure path on the GPU without a fault: a one-shot host-armed hook makes one work unit of
a kernel issue no loads, its consumers' bounded waits run out, the kernel records
GQA_ERR_TIMEOUT and returns.  The test checks that attn_sync_status reports it and that the
same context then computes correct results again (nothing traps, faults or hangs)."""
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


def _prefill_call(blk, inp, ck, cv, delta):
    B, T = inp.x.shape[:2]
    abi.attn_prefill(blk.ctx, inp.x.to(gu.DEV), B, T, inp.R.to(gu.DEV), True, ck, cv, T, 0, delta)


@pytest.mark.parametrize("kind", ["qkv_gemm", "flash_prefill", "out_gemm"])
def test_prefill_timeout_reported_and_context_recovers(kind):
    inp = gin.make_custom(seed=71, B=1, T=300)
    blk = gu.Block(inp)
    try:
        ck, cv = gu.empty_cache(1, 300)
        delta = torch.empty(1, 300, 4096, dtype=torch.float32, device=gu.DEV)
        abi.attn_debug_inject_timeout(blk.ctx, kind)
        _prefill_call(blk, inp, ck, cv, delta)
        with pytest.raises(abi.GQAError) as err:
            abi.attn_sync_status(blk.ctx)
        assert err.value.status == 5  # GQA_ERR_TIMEOUT
        # the same context works again
        _prefill_call(blk, inp, ck, cv, delta)
        abi.attn_sync_status(blk.ctx)
        ref, _ = gu.oracle_prefill(blk, inp)
        gu.assert_close(gu.np64(delta), ref, what=f"after {kind} timeout")
    finally:
        blk.close()


@pytest.mark.parametrize("kind", ["qkv_splitk", "decode_attn", "out_splitk"])
def test_decode_timeout_reported_and_context_recovers(kind):
    B, S_max, pos = 4, 512, 500
    inp = gin.make_custom(seed=72, B=B, T=1, start_pos=pos, S_max=S_max, fill_cache=True)
    blk = gu.Block(inp)
    try:
        x, R = inp.x.to(gu.DEV), inp.R.to(gu.DEV)
        delta = torch.empty(B, 1, 4096, dtype=torch.float32, device=gu.DEV)
        ck, cv = inp.cache_k.to(gu.DEV), inp.cache_v.to(gu.DEV)
        abi.attn_debug_inject_timeout(blk.ctx, kind)
        abi.attn_decode(blk.ctx, x, B, pos, R, ck, cv, S_max, delta)
        with pytest.raises(abi.GQAError) as err:
            abi.attn_sync_status(blk.ctx)
        assert err.value.status == 5
        ck, cv = inp.cache_k.to(gu.DEV), inp.cache_v.to(gu.DEV)
        abi.attn_decode(blk.ctx, x, B, pos, R, ck, cv, S_max, delta)
        abi.attn_sync_status(blk.ctx)
        wq, wk, wv, wo = blk.w64
        ref, _ = orc.attention_decode(gin.to_f64(inp.x), wq, wk, wv, wo, gin.to_f64(inp.R),
                                      gin.to_f64(inp.cache_k), gin.to_f64(inp.cache_v), pos)
        gu.assert_close(gu.np64(delta), ref, what=f"after {kind} timeout")
    finally:
        blk.close()


@pytest.mark.parametrize("start_pos", [0, 1265])
def test_short_prefill_timeout_reported_and_context_recovers(start_pos):
    # T = 16 runs the four-position attention kernel: with one key split (start_pos 0) an
    # aborted CTA writes no H; with five splits (a 1281-key cache) its split never arrives, so
    # its group's arrival counter stays short until attn_sync_status resets the counters
    B, T = 1, 16
    full = gin.make_custom(seed=73 + start_pos, B=B, T=start_pos + T)
    blk = gu.Block(full)
    try:
        S_max = start_pos + T
        ck, cv = gu.empty_cache(B, S_max)
        x, R = full.x.to(gu.DEV), full.R.to(gu.DEV)
        if start_pos:
            blk.prefill(x[:, :start_pos].contiguous(), R[:start_pos].contiguous(), ck, cv)
        xs, Rs = x[:, start_pos:].contiguous(), R[start_pos:].contiguous()
        delta = torch.empty(B, T, 4096, dtype=torch.float32, device=gu.DEV)
        abi.attn_debug_inject_timeout(blk.ctx, "decode_attn")
        abi.attn_prefill(blk.ctx, xs, B, T, Rs, True, ck, cv, S_max, start_pos, delta)
        with pytest.raises(abi.GQAError) as err:
            abi.attn_sync_status(blk.ctx)
        assert err.value.status == 5
        d = blk.prefill(xs, Rs, ck, cv, start_pos=start_pos)
        ref, _ = gu.oracle_prefill(blk, full, rows=list(range(start_pos, start_pos + T)))
        gu.assert_close(gu.np64(d), ref, what=f"short prefill after a timeout (start_pos {start_pos})")
    finally:
        blk.close()
