"""The allocation-free decode attention entry point (GPU), against the fp64 oracle.

attn_decode_attention_noalloc serves callers that cannot let the library allocate device
memory (an engine that keeps all of HBM in its own pool, a decode loop that cannot afford
cudaMalloc's device-wide synchronisation).  Its scratch is a fixed device array inside the
library, so this test checks that two calls in a row, of different sizes, both reproduce the
oracle's merged head outputs H (and the context-based attn_decode's), that a call at the
largest batch the array holds (where the key splits are cut down to fit it) is right too,
that the calls allocate nothing on the device, and that a device-side time-out is reported
and leaves NaN rather than stale partial results.

This file is collected last (tests/test_zz_*), so a run that stops at its first failure has
already run every other test.
"""
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


def _decode_case(seed, B, pos, S_max):
    """Run attn_decode (context path) on a filled cache; return the inputs, its rotated
    queries and merged head outputs, and the cache it left behind (new token written)."""
    inp = gin.make_custom(seed=seed, B=B, T=1, start_pos=pos, S_max=S_max, fill_cache=True)
    blk = gu.Block(inp)
    try:
        ck = inp.cache_k.to(gu.DEV)
        cv = inp.cache_v.to(gu.DEV)
        blk.decode(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv, pos)
        q_r, h = blk.intermediates(B)
        w64 = blk.w64
    finally:
        blk.close()
    return inp, w64, q_r, h, ck, cv


def _oracle_h(inp, w64, pos, seqs):
    """The oracle's H (after the head merge) of the listed sequences ([len(seqs), 4096]);
    each sequence's decode depends on its own token and cache rows only."""
    wq, wk, wv, wo = w64
    s = np.asarray(seqs)
    _, ex = orc.attention_decode(gin.to_f64(inp.x[s]), wq, wk, wv, wo, gin.to_f64(inp.R),
                                 gin.to_f64(inp.cache_k[s, :pos + 1]), gin.to_f64(inp.cache_v[s, :pos + 1]), pos,
                                 keep=True)
    return ex["H"].reshape(len(s), 4096)


def _free_bytes():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def test_noalloc_decode_attention_matches_oracle_on_two_calls():
    cases = [(61, 4, 700, 1024), (62, 2, 299, 300)]
    runs = [_decode_case(*c) for c in cases]
    outs = [torch.full((c[1], 4096), float("nan"), dtype=torch.bfloat16, device=gu.DEV) for c in cases]
    torch.cuda.synchronize()

    # The first call in a process sets the device up, and CUDA loads the library module that
    # holds the fixed scratch array then (lazy module loading): that one-time footprint is the
    # array itself.  Free device memory is then sampled around each of the calls under test.
    # This assumes no other process allocates on the GPU meanwhile (the GPU tests run alone);
    # a cudaMalloc by the library would show up as a drop.
    _, B0, pos0, S0 = cases[0]
    _, _, q0, _, ck0, cv0 = runs[0]
    abi.attn_decode_attention_noalloc(q0, ck0, cv0, B0, pos0 + 1, S0, outs[0])
    abi.attn_decode_attention_noalloc_status()
    around = []
    for (seed, B, pos, S_max), (_, _, q_r, _, ck, cv), h in zip(cases, runs, outs):
        before = _free_bytes()
        abi.attn_decode_attention_noalloc(q_r, ck, cv, B, pos + 1, S_max, h)
        around.append((before, _free_bytes()))
    abi.attn_decode_attention_noalloc_status()

    for (seed, B, pos, S_max), (inp, w64, _, h_ctx, _, _), h in zip(cases, runs, outs):
        ref = _oracle_h(inp, w64, pos, range(B))
        gu.assert_close(gu.np64(h), ref, gu.TOL_REL_L1, gu.TOL_MAX, f"no-alloc H vs oracle (B={B}, kv_len={pos + 1})")
        gu.assert_close(gu.np64(h), gu.np64(h_ctx), gu.TOL_REL_L1, gu.TOL_MAX,
                        f"no-alloc H vs attn_decode (B={B}, kv_len={pos + 1})")
    for before, after in around:
        assert after >= before, "the allocation-free call reduced free device memory"


def test_noalloc_at_its_largest_batch_where_splits_are_cut_to_fit():
    # B = 256 sequences x 8 kv heads fill the array's 2048 units: the two key splits the
    # kernel would otherwise use for 600 keys are cut down to one.
    B, pos, S_max = 256, 599, 640
    inp, w64, q_r, h_ctx, ck, cv = _decode_case(63, B, pos, S_max)
    h = torch.full((B, 4096), float("nan"), dtype=torch.bfloat16, device=gu.DEV)
    abi.attn_decode_attention_noalloc(q_r, ck, cv, B, pos + 1, S_max, h)
    abi.attn_decode_attention_noalloc_status()
    seqs = [0, 1, 77, 128, 200, 255]
    ref = _oracle_h(inp, w64, pos, seqs)
    gu.assert_close(gu.np64(h)[seqs], ref, gu.TOL_REL_L1, gu.TOL_MAX, "no-alloc H vs oracle at B=256")
    gu.assert_close(gu.np64(h), gu.np64(h_ctx), gu.TOL_REL_L1, gu.TOL_MAX, "no-alloc H vs attn_decode at B=256")


def test_noalloc_timeout_is_reported_and_leaves_nan():
    seed, B, pos, S_max = 64, 3, 400, 512
    inp, w64, q_r, _, ck, cv = _decode_case(seed, B, pos, S_max)
    h = torch.zeros((B, 4096), dtype=torch.bfloat16, device=gu.DEV)
    abi.attn_decode_attention_noalloc_debug_inject_timeout()
    abi.attn_decode_attention_noalloc(q_r, ck, cv, B, pos + 1, S_max, h)
    with pytest.raises(abi.GQAError) as err:
        abi.attn_decode_attention_noalloc_status()
    assert err.value.status == 5  # GQA_ERR_TIMEOUT
    assert torch.isnan(h.float()).all()
    abi.attn_decode_attention_noalloc_status()  # read and cleared
    # the next call is correct again
    abi.attn_decode_attention_noalloc(q_r, ck, cv, B, pos + 1, S_max, h)
    abi.attn_decode_attention_noalloc_status()
    gu.assert_close(gu.np64(h), _oracle_h(inp, w64, pos, range(B)), gu.TOL_REL_L1, gu.TOL_MAX,
                    "no-alloc H after a time-out")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    ok = torch.zeros(16, dtype=torch.bfloat16, device=gu.DEV)
    st = abi.raw_status("attn_decode_attention_noalloc", ok.data_ptr(), ok.data_ptr(), ok.data_ptr(),
                        257, 16, 16, ok.data_ptr(), None)
    assert st == 2  # GQA_ERR_SHAPE: more than 256 sequences
    st = abi.raw_status("attn_decode_attention_noalloc", ok.data_ptr(), ok.data_ptr(), ok.data_ptr(),
                        4, 17, 16, ok.data_ptr(), None)
    assert st == 2  # kv_len > S_max
