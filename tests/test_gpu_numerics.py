"""Numerical stress of the attention kernels' online softmax through the C ABI.

Scaling W_Q changes only how peaked the softmax is: x3 makes the scores ~3 times larger (std
~7 in log2 units), so each row is dominated by a few keys; W_Q = 0 makes every visible key
equally likely, so H is the running mean of V (a closed form).  Each case runs the flash
kernel (several tiles, a ragged tail), the four-position short-prefill kernel or the decode
kernel, and compares with the fp64 oracle.  Spikes (one token's x, or one cached key and
value, scaled 20x) make row maxima jump past the lazy-rescale threshold in a later key tile and
make one key split dominate the split merge.

Peaked scores amplify the rounding of the bf16 intermediates (Q_r, K_r, V, P, H): a score
error of |S| 2^-9 becomes a relative error of P.  The bound for these cases is therefore
derived from the same rounding applied to the oracle's own fp64 intermediates (Q_r, K_r, V
rounded to bf16, P = exp(S - max) rounded to bf16, l the sum of the rounded P, H rounded to
bf16): the kernels may add at most a quarter of that floor (and never less than the block's
usual tolerance)."""
import math

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


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()


def _with_wq(inp, factor):
    inp.wq = (inp.wq.float() * factor).to(torch.bfloat16)
    return inp


def _floor_delta(Q_r, keys, vals, wo, first_pos):
    """Delta with the bf16 roundings applied to fp64 intermediates.  Q_r [B, R, 32, 128] for
    query rows at absolute positions first_pos .. first_pos + R - 1 (causal), keys / vals
    [B, n_keys, 8, 128]."""
    B, R = Q_r.shape[:2]
    Q, K, V = _bf16(Q_r), _bf16(keys), _bf16(vals)
    n_keys = K.shape[1]
    pos = first_pos + np.arange(R)
    mask = np.where(np.arange(n_keys)[None, :] > pos[:, None], -np.inf, 0.0)
    H = np.empty((B, R, 32, 128))
    for b in range(B):
        for h in range(32):
            g = h // 4
            S = Q[b, :, h, :] @ K[b, :, g, :].T / math.sqrt(128) + mask
            P = _bf16(np.exp(S - S.max(axis=1, keepdims=True)))
            H[b, :, h, :] = (P @ V[b, :, g, :]) / P.sum(axis=1, keepdims=True)
    return _bf16(H.reshape(B, R, 4096)) @ wo.T


def _bound(floor, ref):
    l1, mx = gu.metrics(floor, ref)
    return max(gu.TOL_REL_L1, 1.25 * l1), max(gu.TOL_MAX, 1.25 * mx)


@pytest.mark.parametrize("T", [16, 300, 2048])
def test_peaked_softmax_prefill(T):
    inp = _with_wq(gin.make_custom(seed=700 + T, B=1, T=T), 3.0)
    blk = gu.Block(inp)
    try:
        ck, cv = gu.empty_cache(1, T)
        delta = blk.prefill(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv)
        ref, ex = gu.oracle_prefill(blk, inp, keep=T <= 512)
        if T > 512:  # intermediates without the attention matrices
            wq, wk, wv, wo = blk.w64
            x64, R64 = gin.to_f64(inp.x), gin.to_f64(inp.R)
            ex = {"Q_r": orc.rope(orc.linear(x64, wq).reshape(1, T, 32, 128), R64),
                  "K_r": orc.rope(orc.linear(x64, wk).reshape(1, T, 8, 128), R64),
                  "V": orc.linear(x64, wv).reshape(1, T, 8, 128)}
        rl1, rmx = _bound(_floor_delta(ex["Q_r"], ex["K_r"], ex["V"], blk.w64[3], 0), ref)
        gu.assert_close(gu.np64(delta), ref, rl1, rmx, what=f"W_Q x3, T={T} (bound {rl1:.2e} / {rmx:.2e})")
    finally:
        blk.close()


@pytest.mark.parametrize("T", [13, 300])
def test_uniform_softmax_prefill(T):
    inp = _with_wq(gin.make_custom(seed=710 + T, B=2, T=T), 0.0)
    blk = gu.Block(inp)
    try:
        ck, cv = gu.empty_cache(2, T)
        delta = blk.prefill(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv)
        ref, ex = gu.oracle_prefill(blk, inp, keep=True)
        # with Q = 0 every visible key has the same weight: H is the running mean of V
        mean = np.cumsum(ex["V"], axis=1) / np.arange(1, T + 1)[None, :, None, None]
        np.testing.assert_allclose(ex["H"].reshape(2, T, 32, 128), np.repeat(mean, 4, axis=2), rtol=1e-9, atol=1e-12)
        _, h = blk.intermediates(2 * T)
        gu.assert_close(gu.np64(h).reshape(2, T, 4096), ex["H"], what=f"W_Q = 0, T={T} H")
        gu.assert_close(gu.np64(delta), ref, what=f"W_Q = 0, T={T} delta")
    finally:
        blk.close()


@pytest.mark.parametrize("factor", [3.0, 0.0])
def test_decode_softmax_extremes(factor):
    B, pos = 3, 1000
    inp = _with_wq(gin.make_custom(seed=720, B=B, T=1, start_pos=pos, S_max=pos + 1, fill_cache=True), factor)
    blk = gu.Block(inp)
    try:
        d = blk.decode(inp.x.to(gu.DEV), inp.R.to(gu.DEV), inp.cache_k.to(gu.DEV), inp.cache_v.to(gu.DEV), pos)
        wq, wk, wv, wo = blk.w64
        ref, ex = orc.attention_decode(gin.to_f64(inp.x), wq, wk, wv, wo, gin.to_f64(inp.R),
                                       gin.to_f64(inp.cache_k), gin.to_f64(inp.cache_v), pos, keep=True)
        rl1, rmx = _bound(_floor_delta(ex["Q_r"], ex["cache_k"][:, :pos + 1], ex["cache_v"][:, :pos + 1], wo, pos),
                          ref)
        gu.assert_close(gu.np64(d), ref, rl1, rmx, what=f"decode, W_Q x{factor} (bound {rl1:.2e} / {rmx:.2e})")
    finally:
        blk.close()


def _spike(t, index, factor=20.0):
    t = t.clone()
    t[index] = (t[index].float() * factor).to(torch.bfloat16)
    return t


def test_spike_key_forces_rescale_prefill():
    # token 200's x scaled 20x: its key dominates (or vanishes from) every later row, so the
    # running max of many rows jumps far past the lazy-rescale threshold in the second 128-key
    # tile, and its value dominates those rows' H
    T = 600
    inp = gin.make_custom(seed=730, B=1, T=T)
    inp.x = _spike(inp.x, (0, 200))
    blk = gu.Block(inp)
    try:
        ck, cv = gu.empty_cache(1, T)
        delta = blk.prefill(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv)
        ref, ex = gu.oracle_prefill(blk, inp, keep=True)
        rl1, rmx = _bound(_floor_delta(ex["Q_r"], ex["K_r"], ex["V"], blk.w64[3], 0), ref)
        gu.assert_close(gu.np64(delta), ref, rl1, rmx, what=f"spike key, T={T} (bound {rl1:.2e} / {rmx:.2e})")
    finally:
        blk.close()


@pytest.mark.parametrize("T", [1, 16])
def test_spike_key_across_key_splits(T):
    # a cache of 1281 positions (several key splits) whose position 700 has a 20x key and
    # value: the split holding it has a running max far above the others', so the split merge
    # (log-sum-exp) must weight the other splits by ~0; T = 1 is the decode kernel, T = 16 the
    # four-position kernel (a prefill continuing the cache)
    B, start_pos = (2, 1280) if T == 1 else (1, 1265)  # B = 1: the 16 positions take the four-position kernel
    S_max = start_pos + T
    inp = gin.make_custom(seed=740 + T, B=B, T=T, start_pos=start_pos, S_max=S_max, fill_cache=True)
    inp.cache_k = _spike(inp.cache_k, (slice(None), 700))
    inp.cache_v = _spike(inp.cache_v, (slice(None), 700))
    blk = gu.Block(inp)
    try:
        ck, cv = inp.cache_k.to(gu.DEV), inp.cache_v.to(gu.DEV)
        if T == 1:
            d = blk.decode(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv, start_pos)
        else:
            d = blk.prefill(inp.x.to(gu.DEV), inp.R.to(gu.DEV), ck, cv, start_pos=start_pos)
        wq, wk, wv, wo = blk.w64
        ref, ex = orc.attention_block(gin.to_f64(inp.x), wq, wk, wv, wo, gin.to_f64(inp.R), start_pos=start_pos,
                                      cache_k=gin.to_f64(inp.cache_k), cache_v=gin.to_f64(inp.cache_v), keep=True)
        rl1, rmx = _bound(_floor_delta(ex["Q_r"], ex["cache_k"][:, :S_max], ex["cache_v"][:, :S_max], wo, start_pos),
                          ref)
        gu.assert_close(gu.np64(d), ref, rl1, rmx, what=f"spike in a long cache, T={T} (bound {rl1:.2e} / {rmx:.2e})")
    finally:
        blk.close()
