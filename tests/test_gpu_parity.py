"""GPU parity of the C-ABI path against the fp64 oracle (element by element, seeded inputs).

Sizes span several 128-row tiles with ragged tails; the full-size workloads are checked on
sampled query rows / sequences that the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

from oracle import gqa_oracle as orc
from tests import gpu_util as gu
from transformer_gqa_attention_gb300 import inputs as gin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from transformer_gqa_attention_gb300 import _build
    _build.build()


def _run_prefill_case(inp, causal=True, check_intermediates=True):
    blk = gu.Block(inp)
    try:
        B, T = inp.x.shape[:2]
        x = inp.x.to(gu.DEV)
        R = inp.R.to(gu.DEV)
        ck, cv = gu.empty_cache(B, T)
        delta = blk.prefill(x, R, ck, cv, causal=causal)
        ref, ex = gu.oracle_prefill(blk, inp, causal=causal, keep=check_intermediates)
        out = {}
        if check_intermediates:
            q_r, h = blk.intermediates(B * T)
            out["K_r"] = gu.assert_close(gu.np64(ck), ex["K_r"], gu.TOL_BF16_REL_L1, gu.TOL_BF16_MAX, "K_r")
            out["V"] = gu.assert_close(gu.np64(cv), ex["V"], gu.TOL_BF16_REL_L1, gu.TOL_BF16_MAX, "V")
            out["Q_r"] = gu.assert_close(gu.np64(q_r).reshape(B, T, 32, 128), ex["Q_r"],
                                         gu.TOL_BF16_REL_L1, gu.TOL_BF16_MAX, "Q_r")
            out["H"] = gu.assert_close(gu.np64(h).reshape(B, T, 4096), ex["H"], gu.TOL_REL_L1,
                                       gu.TOL_MAX, "H")
        out["delta"] = gu.assert_close(gu.np64(delta), ref, what="delta")
        return out
    finally:
        blk.close()


def test_prefill_b1_t16_workload():
    _run_prefill_case(gin.make_inputs("prefill_b1_t16"))


@pytest.mark.parametrize("B,T", [(1, 1), (2, 3), (1, 64), (3, 17), (1, 129), (2, 200), (1, 1000)])
def test_prefill_ragged_shapes(B, T):
    _run_prefill_case(gin.make_custom(seed=100 + T, B=B, T=T))


def test_prefill_with_scaled_rope_table():
    # the Llama 3.1 scaled table is just another R input: same kernels, same oracle
    inp = gin.make_custom(seed=9, B=2, T=1000)
    inp.R = gin.rope_table(np.arange(1000), scaled=True)
    _run_prefill_case(inp)


def test_prefill_non_causal():
    _run_prefill_case(gin.make_custom(seed=7, B=2, T=300), causal=False)


def test_prefill_b1_t2048_workload_full():
    _run_prefill_case(gin.make_inputs("prefill_b1_t2048"), check_intermediates=False)


def test_prefill_narrow_last_round_pieces():
    # 4096 tokens: the Q/K/V projection's 384 tiles of 256 x 256 leave 4 (the V columns of the
    # last 256 rows) for a partial last round, cut into 32-column pieces (N = 32 UMMAs, 16-row
    # weight boxes); W_O's 256 tiles leave 28 (rows 3584..4095), cut into 96-column pieces.
    # K_r and V are checked in full, Q_r, H and Delta on sampled rows that include those rows.
    B, T = 1, 4096
    inp = gin.make_custom(seed=41, B=B, T=T)
    blk = gu.Block(inp)
    try:
        ck, cv = gu.empty_cache(B, T)
        delta = blk.prefill(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv)
        rows = np.union1d(gu.sample_rows(T), np.arange(3584, T, 9))
        ref, ex = gu.oracle_prefill(blk, inp, rows=rows, keep=True)
        q_r, h = blk.intermediates(B * T)
        gu.assert_close(gu.np64(ck), ex["K_r"], gu.TOL_BF16_REL_L1, gu.TOL_BF16_MAX, "K_r")
        gu.assert_close(gu.np64(cv), ex["V"], gu.TOL_BF16_REL_L1, gu.TOL_BF16_MAX, "V")
        gu.assert_close(gu.np64(q_r).reshape(B, T, 32, 128)[:, rows], ex["Q_r"], gu.TOL_BF16_REL_L1,
                        gu.TOL_BF16_MAX, "Q_r rows")
        gu.assert_close(gu.np64(h).reshape(B, T, 4096)[:, rows], ex["H"], gu.TOL_REL_L1, gu.TOL_MAX, "H rows")
        gu.assert_close(gu.np64(delta[:, rows]), ref, what="delta rows")
    finally:
        blk.close()


@pytest.mark.parametrize("name", ["prefill_b4_t8192", "prefill_b1_t32768"])
def test_prefill_large_workloads_sampled_rows(name):
    inp = gin.make_inputs(name)
    blk = gu.Block(inp)
    try:
        B, T = inp.x.shape[:2]
        ck, cv = gu.empty_cache(B, T)
        delta = blk.prefill(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv)
        rows = gu.sample_rows(T)
        ref, _ = gu.oracle_prefill(blk, inp, rows=rows)
        gu.assert_close(gu.np64(delta[:, rows]), ref, what=f"{name} delta rows")
        # keys / values of a few positions land in the cache
        wq, wk, wv, wo = blk.w64
        pos = rows[:8]
        x64 = gin.to_f64(inp.x[:, pos])
        K = orc.rope(orc.linear(x64, wk).reshape(B, len(pos), 8, 128), gin.to_f64(inp.R[pos]))
        gu.assert_close(gu.np64(ck[:, pos]), K, gu.TOL_BF16_REL_L1, gu.TOL_BF16_MAX, "cache K rows")
    finally:
        blk.close()


def test_chunked_prefill_continues_from_cache():
    B, T1, T2 = 2, 100, 77
    inp = gin.make_custom(seed=21, B=B, T=T1 + T2)
    blk = gu.Block(inp)
    try:
        x = inp.x.to(gu.DEV)
        R = inp.R.to(gu.DEV)
        ck, cv = gu.empty_cache(B, T1 + T2 + 5)
        blk.prefill(x[:, :T1].contiguous(), R[:T1].contiguous(), ck, cv)
        d2 = blk.prefill(x[:, T1:].contiguous(), R[T1:].contiguous(), ck, cv, start_pos=T1)
        ref, _ = gu.oracle_prefill(blk, inp)
        gu.assert_close(gu.np64(d2), ref[:, T1:], what="second chunk")
    finally:
        blk.close()


def test_decode_small():
    B, S_max, pos = 3, 300, 257
    inp = gin.make_custom(seed=31, B=B, T=1, start_pos=pos, S_max=S_max, fill_cache=True)
    blk = gu.Block(inp)
    try:
        ck = inp.cache_k.to(gu.DEV)
        cv = inp.cache_v.to(gu.DEV)
        delta = blk.decode(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv, pos)
        wq, wk, wv, wo = blk.w64
        ref, ex = orc.attention_decode(gin.to_f64(inp.x), wq, wk, wv, wo, gin.to_f64(inp.R),
                                       gin.to_f64(inp.cache_k), gin.to_f64(inp.cache_v), pos)
        gu.assert_close(gu.np64(delta), ref, what="decode delta")
        gu.assert_close(gu.np64(ck[:, pos]), ex["cache_k"][:, pos], gu.TOL_BF16_REL_L1, gu.TOL_BF16_MAX,
                        "new cache K")
        # untouched cache entries stay bit-identical
        assert torch.equal(ck[:, :pos].cpu(), inp.cache_k[:, :pos])
        assert torch.equal(cv[:, pos + 1:].cpu(), inp.cache_v[:, pos + 1:])
    finally:
        blk.close()


@pytest.mark.parametrize("pos", [0, 63, 64, 65, 1000])
def test_decode_at_tile_boundaries_and_first_position(pos):
    # kv_len = pos + 1 around the 64-key tile of the split-KV kernel; pos = 0 attends over the
    # new token alone, so H of head h is exactly the new V of its kv head h // 4 (rounded once)
    B = 2
    inp = gin.make_custom(seed=200 + pos, B=B, T=1, start_pos=pos, S_max=pos + 1, fill_cache=True)
    blk = gu.Block(inp)
    try:
        ck, cv = inp.cache_k.to(gu.DEV), inp.cache_v.to(gu.DEV)
        delta = blk.decode(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv, pos)
        wq, wk, wv, wo = blk.w64
        ref, ex = orc.attention_decode(gin.to_f64(inp.x), wq, wk, wv, wo, gin.to_f64(inp.R),
                                       gin.to_f64(inp.cache_k), gin.to_f64(inp.cache_v), pos, keep=True)
        gu.assert_close(gu.np64(delta), ref, what=f"decode at position {pos}")
        if pos == 0:
            _, h = blk.intermediates(B)
            v_new = gu.np64(cv[:, 0])  # [B, 8, 128] as stored by the kernel (bf16)
            expect = np.repeat(v_new, 4, axis=1).reshape(B, 4096)
            np.testing.assert_array_equal(gu.np64(h), expect)
    finally:
        blk.close()


@pytest.mark.parametrize("T,start_pos", [(1, 5), (1, 300), (3, 129), (17, 1000)])
def test_short_prefill_continuing_a_long_cache(T, start_pos):
    B = 2
    full = gin.make_custom(seed=210 + T, B=B, T=start_pos + T)
    blk = gu.Block(full)
    try:
        S_max = start_pos + T
        ck, cv = gu.empty_cache(B, S_max)
        x, R = full.x.to(gu.DEV), full.R.to(gu.DEV)
        blk.prefill(x[:, :start_pos].contiguous(), R[:start_pos].contiguous(), ck, cv)
        d = blk.prefill(x[:, start_pos:].contiguous(), R[start_pos:].contiguous(), ck, cv, start_pos=start_pos)
        rows = np.arange(start_pos, start_pos + T)
        ref, _ = gu.oracle_prefill(blk, full, rows=rows)
        gu.assert_close(gu.np64(d), ref, what=f"prefill of {T} positions after {start_pos}")
    finally:
        blk.close()


def test_decode_b64_pos4095_workload_sampled_sequences():
    inp = gin.make_inputs("decode_b64_pos4095")
    pos = 4095
    blk = gu.Block(inp)
    try:
        ck = inp.cache_k.to(gu.DEV)
        cv = inp.cache_v.to(gu.DEV)
        delta = blk.decode(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv, pos)
        wq, wk, wv, wo = blk.w64
        for b in (0, 17, 63):
            ref, _ = orc.attention_decode(gin.to_f64(inp.x[b:b + 1]), wq, wk, wv, wo, gin.to_f64(inp.R),
                                          gin.to_f64(inp.cache_k[b:b + 1]), gin.to_f64(inp.cache_v[b:b + 1]),
                                          pos)
            gu.assert_close(gu.np64(delta[b:b + 1]), ref, what=f"decode seq {b}")
    finally:
        blk.close()


def test_decode_equals_last_prefill_row_on_gpu():
    B, T = 2, 150
    inp = gin.make_custom(seed=41, B=B, T=T)
    blk = gu.Block(inp)
    try:
        x = inp.x.to(gu.DEV)
        R = inp.R.to(gu.DEV)
        ck, cv = gu.empty_cache(B, T)
        dp = blk.prefill(x, R, ck, cv)
        dd = blk.decode(x[:, T - 1:].contiguous(), R[T - 1:].contiguous(), ck, cv, T - 1)
        l1, mx = gu.metrics(gu.np64(dd[:, 0]), gu.np64(dp[:, T - 1]))
        assert l1 < 5e-3 and mx < 2e-2, (l1, mx)
    finally:
        blk.close()


def test_prefill_then_three_decode_steps_against_oracle():
    # prefill 300 positions of 3 sequences, then decode positions 300, 301, 302 one at a time
    # through the same caches; every step's Delta against the oracle fed the oracle's own
    # caches (rotated keys and values of all earlier positions)
    B, T, steps = 3, 300, 3
    inp = gin.make_custom(seed=77, B=B, T=T)
    blk = gu.Block(inp)
    try:
        S_max = T + steps
        ck, cv = gu.empty_cache(B, S_max)
        blk.prefill(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv)
        wq, wk, wv, wo = blk.w64
        _, ex = orc.attention_block(gin.to_f64(inp.x), wq, wk, wv, wo, gin.to_f64(inp.R), keep=True)
        ok = np.zeros((B, S_max, 8, 128))
        ov = np.zeros((B, S_max, 8, 128))
        ok[:, :T], ov[:, :T] = ex["K_r"], ex["V"]
        gen = torch.Generator().manual_seed(78)
        for i in range(steps):
            pos = T + i
            x1 = torch.randn(B, 1, 4096, generator=gen).to(torch.bfloat16)
            R1 = gin.rope_table([pos])
            d = blk.decode(x1.to(gu.DEV), R1.to(gu.DEV), ck, cv, pos)
            ref, ex1 = orc.attention_decode(gin.to_f64(x1), wq, wk, wv, wo, gin.to_f64(R1), ok, ov, pos, keep=True)
            gu.assert_close(gu.np64(d), ref, what=f"decode step at position {pos}")
            ok, ov = ex1["cache_k"], ex1["cache_v"]
    finally:
        blk.close()


def test_prefill_maximum_token_count():
    # B*T at the documented limit (262144): GEMM M = 262144, 32768 attention CTAs, a 4 GB
    # workspace; a few sequences checked against the oracle
    B, T = 2048, 128
    inp = gin.make_custom(seed=71, B=B, T=T)
    blk = gu.Block(inp)
    try:
        ck, cv = gu.empty_cache(B, T)
        delta = blk.prefill(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv)
        wq, wk, wv, wo = blk.w64
        for b in (0, 1023, 2047):
            ref, _ = orc.attention_block(gin.to_f64(inp.x[b:b + 1]), wq, wk, wv, wo, gin.to_f64(inp.R))
            gu.assert_close(gu.np64(delta[b:b + 1]), ref, what=f"max-token prefill seq {b}")
    finally:
        blk.close()


def test_decode_maximum_s_max():
    # S_max at the documented limit (2^20 positions per sequence, 2 GB between sequences);
    # positions past the 131072 seeded keys hold NaN, so any read beyond kv_len shows
    B, S_max, pos = 2, 1 << 20, 131071
    inp = gin.make_custom(seed=72, B=B, T=1, start_pos=pos, S_max=pos + 1, fill_cache=True)
    blk = gu.Block(inp)
    try:
        ck, cv = gu.empty_cache(B, S_max)
        ck[:, :pos + 1] = inp.cache_k.to(gu.DEV)
        cv[:, :pos + 1] = inp.cache_v.to(gu.DEV)
        delta = blk.decode(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv, pos)
        assert torch.isnan(ck[:, pos + 1:pos + 65].float()).all()  # nothing written past the slot
        wq, wk, wv, wo = blk.w64
        ref, _ = orc.attention_decode(gin.to_f64(inp.x), wq, wk, wv, wo, gin.to_f64(inp.R),
                                      gin.to_f64(inp.cache_k), gin.to_f64(inp.cache_v), pos)
        gu.assert_close(gu.np64(delta), ref, what="decode at S_max = 2^20")
    finally:
        blk.close()


def test_decode_maximum_batch():
    # B at the decode limit (1024): the projections take the many-token path
    B, pos = 1024, 199
    inp = gin.make_custom(seed=73, B=B, T=1, start_pos=pos, S_max=pos + 1, fill_cache=True)
    blk = gu.Block(inp)
    try:
        delta = blk.decode(inp.x.to(gu.DEV), inp.R.to(gu.DEV), inp.cache_k.to(gu.DEV), inp.cache_v.to(gu.DEV), pos)
        wq, wk, wv, wo = blk.w64
        for b in (0, 511, 1023):
            ref, _ = orc.attention_decode(gin.to_f64(inp.x[b:b + 1]), wq, wk, wv, wo, gin.to_f64(inp.R),
                                          gin.to_f64(inp.cache_k[b:b + 1]), gin.to_f64(inp.cache_v[b:b + 1]), pos)
            gu.assert_close(gu.np64(delta[b:b + 1]), ref, what=f"max-batch decode seq {b}")
    finally:
        blk.close()


def test_causality_and_determinism_bit_exact():
    B, T, t0 = 1, 300, 130
    inp = gin.make_custom(seed=51, B=B, T=T)
    blk = gu.Block(inp)
    try:
        x = inp.x.to(gu.DEV)
        R = inp.R.to(gu.DEV)
        ck, cv = gu.empty_cache(B, T)
        d0 = blk.prefill(x, R, ck, cv).clone()
        d1 = blk.prefill(x, R, ck, cv).clone()
        assert torch.equal(d0, d1)
        xp = x.clone()
        xp[:, t0 + 1:] = -xp[:, t0 + 1:] * 3
        d2 = blk.prefill(xp, R, ck, cv)
        assert torch.equal(d2[:, :t0 + 1], d0[:, :t0 + 1])
        assert not torch.equal(d2[:, t0 + 1:], d0[:, t0 + 1:])
    finally:
        blk.close()


@pytest.mark.parametrize("name", ["prefill_b1_t2048_pos30720", "prefill_b4_t16_pos4080"])
def test_prefill_continuing_a_drawn_cache_workloads(name):
    # the chunked-prefill workloads as bench.py times them: a drawn cache of start_pos
    # positions, the chunk's rows (sampled for the long chunk) against the oracle with that cache
    w = gin.WORKLOADS[name]
    inp = gin.make_inputs(name)
    blk = gu.Block(inp)
    try:
        B, T = inp.x.shape[:2]
        ck, cv = inp.cache_k.to(gu.DEV), inp.cache_v.to(gu.DEV)
        delta = blk.prefill(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv, start_pos=w.start_pos)
        rows = gu.sample_rows(T) if T > 64 else np.arange(T)
        wq, wk, wv, wo = blk.w64
        ref, ex = orc.attention_block(gin.to_f64(inp.x), wq, wk, wv, wo, gin.to_f64(inp.R), start_pos=w.start_pos,
                                      cache_k=gin.to_f64(inp.cache_k), cache_v=gin.to_f64(inp.cache_v), rows=rows)
        gu.assert_close(gu.np64(delta[:, rows]), ref, what=f"{name} delta rows")
        # the chunk's keys and values landed after the cached positions, the cache before is intact
        n_keys = w.start_pos + T
        gu.assert_close(gu.np64(ck[:, w.start_pos:n_keys]), ex["cache_k"][:, w.start_pos:n_keys],
                        gu.TOL_BF16_REL_L1, gu.TOL_BF16_MAX, "chunk K_r in the cache")
        np.testing.assert_array_equal(gu.np64(ck[:, :w.start_pos]), gin.to_f64(inp.cache_k[:, :w.start_pos]))
    finally:
        blk.close()
