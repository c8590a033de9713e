"""GPU parity of short prefills (T <= 16 positions per sequence), which run the attention
through the decode kernel with four positions per CTA, each masked causally, against the
fp64 oracle through the C ABI.

Cases: every position-group shape (T = 1 .. 16, ragged groups of 1-3 positions), chunks
continuing caches across the 64-key tile and over several key splits (including a split that
holds no visible key for the first position group), the non-causal form, the largest batch
the arrival counters serve (256 sequences x 16 positions) and the first batch past it (257,
which falls back to the flash kernel), and which kernel a call runs: the four-position kernel
while the cache is at most 256 keys or the flash grid would have fewer than 32 CTAs, else the
flash kernel (its tcgen05 tiles cost less per key once its grid fills the GPU)."""
import numpy as np
import pytest
import torch

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


def _prefill_from_zero(inp, causal=True):
    blk = gu.Block(inp)
    try:
        B, T = inp.x.shape[:2]
        ck, cv = gu.empty_cache(B, T)
        delta = blk.prefill(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv, causal=causal)
        ref, ex = gu.oracle_prefill(blk, inp, causal=causal, keep=True)
        _, h = blk.intermediates(B * T)
        gu.assert_close(gu.np64(h).reshape(B, T, 4096), ex["H"], what=f"H (B={B}, T={T})")
        gu.assert_close(gu.np64(delta), ref, what=f"delta (B={B}, T={T})")
    finally:
        blk.close()


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 7, 8, 11, 13, 15, 16])
def test_every_position_group_shape(T):
    _prefill_from_zero(gin.make_custom(seed=300 + T, B=2, T=T))


def test_non_causal_short_prefill():
    _prefill_from_zero(gin.make_custom(seed=320, B=2, T=16), causal=False)


def _continue_cache(B, T, start_pos, seed, causal=True):
    full = gin.make_custom(seed=seed, B=B, T=start_pos + T)
    blk = gu.Block(full)
    try:
        S_max = start_pos + T
        ck, cv = gu.empty_cache(B, S_max)
        x, R = full.x.to(gu.DEV), full.R.to(gu.DEV)
        blk.prefill(x[:, :start_pos].contiguous(), R[:start_pos].contiguous(), ck, cv)
        d = blk.prefill(x[:, start_pos:].contiguous(), R[start_pos:].contiguous(), ck, cv, start_pos=start_pos,
                        causal=causal)
        rows = np.arange(start_pos, start_pos + T)
        if causal:
            ref, _ = gu.oracle_prefill(blk, full, rows=rows)
        else:
            # a non-causal chunk sees every cached key and all of its own positions: the
            # oracle's non-causal block over the cache plus the chunk, the chunk's rows
            ref, _ = gu.oracle_prefill(blk, full, rows=rows, causal=False)
        gu.assert_close(gu.np64(d), ref, what=f"{T} positions after {start_pos} (B={B}, causal={causal})")
    finally:
        blk.close()


@pytest.mark.parametrize("B,T,start_pos", [(2, 16, 48), (2, 5, 60), (1, 16, 1000), (1, 13, 4090),
                                           (1, 16, 1265), (2, 9, 127), (3, 16, 1000)])
def test_short_prefill_continuing_a_cache(B, T, start_pos):
    # (16, 48): the chunk ends on the 64-key tile; (5, 60): it straddles it; (13, 4090):
    # several key splits; (16, 1265): the first position group sees no key of the last split;
    # (3, 16, 1000): a long cache with a batch whose flash grid fills the GPU: the flash kernel
    _continue_cache(B, T, start_pos, seed=330 + T + start_pos)


@pytest.mark.parametrize("B,T,start_pos,kernel", [(1, 16, 0, "decode_attn"), (4, 16, 0, "decode_attn"),
                                                  (4, 16, 240, "decode_attn"), (1, 16, 4080, "decode_attn"),
                                                  (2, 16, 4080, "flash_prefill"), (4, 16, 496, "flash_prefill"),
                                                  (1, 17, 0, "flash_prefill")])
def test_kernel_choice_for_short_prefills(B, T, start_pos, kernel):
    # which attention kernel a call runs (the library's per-kernel profile): the four-position
    # kernel up to 16 positions while the cache is short or the flash grid would be small
    inp = gin.make_custom(seed=360, B=B, T=start_pos + T)
    blk = gu.Block(inp)
    try:
        S_max = start_pos + T
        ck, cv = gu.empty_cache(B, S_max)
        x, R = inp.x.to(gu.DEV), inp.R.to(gu.DEV)
        if start_pos:
            blk.prefill(x[:, :start_pos].contiguous(), R[:start_pos].contiguous(), ck, cv)
        abi.attn_profile_begin(blk.ctx)
        blk.prefill(x[:, start_pos:].contiguous(), R[start_pos:].contiguous(), ck, cv, start_pos=start_pos)
        prof = abi.attn_profile_end(blk.ctx)
        ran = {k for k, (_, n) in prof.items() if n > 0 and k in ("decode_attn", "flash_prefill")}
        assert ran == {kernel}, prof
    finally:
        blk.close()


def test_non_causal_chunk_sees_the_whole_cache():
    _continue_cache(2, 7, 100, seed=340, causal=False)


@pytest.mark.parametrize("B", [256, 257])
def test_counter_capacity_boundary(B):
    # 256 x 8 groups x 4 position groups = 8192 arrival counters: the short kernel; one more
    # sequence: the flash kernel.  Checked on a sample of sequences (each is independent).
    T = 16
    inp = gin.make_custom(seed=350 + B, B=B, T=T)
    blk = gu.Block(inp)
    try:
        ck, cv = gu.empty_cache(B, T)
        d = gu.np64(blk.prefill(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv))
        seqs = [0, 1, 127, B - 2, B - 1]
        sub = gin.BlockInputs(x=inp.x[seqs].contiguous(), R=inp.R, wq=inp.wq, wk=inp.wk, wv=inp.wv, wo=inp.wo)
        ref, _ = gu.oracle_prefill(blk, sub)
        gu.assert_close(d[seqs], ref, what=f"B={B} x T=16, sequences {seqs}")
    finally:
        blk.close()
