"""The allocation-free decode attention entry point against attn_decode (GPU).

attn_decode_attention_noalloc serves callers that cannot let the library allocate device
memory (an engine that keeps all of HBM in its own pool, a decode loop that cannot afford
cudaMalloc's device-wide synchronisation).  Its scratch is a fixed device array inside
the library, so this test also checks that two calls in a row, of different sizes, both
reproduce what the context-based attn_decode computed, and that the second call leaves
the device's free memory unchanged.
"""
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


def _decode_reference(seed, B, pos, S_max):
    """Run attn_decode (context path) and return its rotated queries, merged head outputs
    and the cache it left behind (with the new token written)."""
    inp = gin.make_custom(seed=seed, B=B, T=1, start_pos=pos, S_max=S_max, fill_cache=True)
    blk = gu.Block(inp)
    try:
        ck = inp.cache_k.to(gu.DEV)
        cv = inp.cache_v.to(gu.DEV)
        blk.decode(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv, pos)
        q_r, h = blk.intermediates(B)
    finally:
        blk.close()
    return q_r, h, ck, cv


def test_noalloc_decode_attention_matches_attn_decode_on_two_calls():
    cases = [(61, 4, 700, 1024), (62, 2, 299, 300)]
    refs = [_decode_reference(*c) for c in cases]
    outs = [torch.full((c[1], 4096), float("nan"), dtype=torch.bfloat16, device=gu.DEV) for c in cases]
    torch.cuda.synchronize()

    free_after = []
    for (seed, B, pos, S_max), (q_r, _, ck, cv), h in zip(cases, refs, outs):
        abi.attn_decode_attention_noalloc(q_r, ck, cv, B, pos + 1, S_max, h)
        torch.cuda.synchronize()
        free_after.append(torch.cuda.mem_get_info()[0])

    for (seed, B, pos, S_max), (_, h_ref, _, _), h in zip(cases, refs, outs):
        gu.assert_close(gu.np64(h), gu.np64(h_ref), gu.TOL_REL_L1, gu.TOL_MAX,
                        f"no-alloc H (B={B}, kv_len={pos + 1})")
    # the second call allocated nothing on the device
    assert free_after[1] == free_after[0]


def test_noalloc_rejects_sizes_beyond_its_scratch():
    ok = torch.zeros(16, dtype=torch.bfloat16, device=gu.DEV)
    st = abi.raw_status("attn_decode_attention_noalloc", ok.data_ptr(), ok.data_ptr(), ok.data_ptr(),
                        257, 16, 16, ok.data_ptr(), None)
    assert st == 2  # GQA_ERR_SHAPE: more than 256 sequences
    st = abi.raw_status("attn_decode_attention_noalloc", ok.data_ptr(), ok.data_ptr(), ok.data_ptr(),
                        4, 17, 16, ok.data_ptr(), None)
    assert st == 2  # kv_len > S_max
