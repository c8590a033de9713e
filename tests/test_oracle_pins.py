"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test ties one step of the oracle to something other than the oracle itself:
the counts the pages print, a library routine that computes the same thing by another
route (numpy / torch complex products, numpy.repeat / torch.repeat_interleave, torch's
scaled_dot_product_attention in fp64), closed forms, invariants, or an element-by-element
brute force with the head sharing materialised.  A plausible slip (dropped term, wrong
sign or index, transposed operand, missing scale, off-by-one mask) fails at least one,
as the planted-mistake tests at the end show.
"""
import math

import numpy as np
import pytest
import torch

from oracle import gqa_oracle as orc
from tests.conftest import read_golden
from transformer_gqa_attention_gb300 import inputs as gin


def tiny(seed=0, B=2, T=6, dim=32, n_heads=8, n_kv=2, x_std=1.0, w_std=0.3):
    """Small fp64 block with the real head ratio 4 (n_heads / n_kv)."""
    rng = np.random.default_rng(seed)
    d = dim // n_heads
    x = rng.standard_normal((B, T, dim)) * x_std
    wq = rng.standard_normal((n_heads * d, dim)) * w_std
    wk = rng.standard_normal((n_kv * d, dim)) * w_std
    wv = rng.standard_normal((n_kv * d, dim)) * w_std
    wo = rng.standard_normal((dim, n_heads * d)) * w_std
    R = gin.rope_table(np.arange(T), head_dim=d, theta=10000.0).numpy().astype(np.float64)
    return x, wq, wk, wv, wo, R


# ---------------------------------------------------------------- printed figures
def test_param_accounting_matches_pages():
    g = read_golden("param_accounting.txt")
    gen = torch.Generator("cpu").manual_seed(0)
    wq, wk, wv, wo = gin.make_weights(gen)
    assert wq.numel() == g["query_projection"] == g["query_projection_total"]
    assert wk.numel() == g["key_projection"]
    assert wv.numel() == g["value_projection"]
    assert wo.numel() == g["output_projection"] == g["merge_and_project_total"]
    total = orc.param_count(wq, wk, wv, wo)
    assert total == g["per_instance_total"] == 41_943_040
    assert total * g["blocks"] == g["across_blocks"]
    assert wo.numel() * g["blocks"] == g["merge_and_project_across_blocks"]
    assert wq.numel() * g["blocks"] == g["query_projection_across_blocks"]
    # dimensions the oracle assumes are the catalogue's
    assert orc.DIM == g["dim"] and orc.N_HEADS == g["n_heads"] and orc.N_KV_HEADS == g["n_kv_heads"]
    assert gin.ROPE_THETA == g["rope_theta"]
    assert g["dim"] // g["n_heads"] == g["head_dim"] == 2 * g["rope_pairs"]
    assert tuple(wk.shape) == (g["n_kv_heads"] * g["head_dim"], g["dim"])  # [out, in]


# ---------------------------------------------------------------- RoPE (steps 4-5)
def test_rope_equals_complex_product_numpy_and_torch():
    rng = np.random.default_rng(1)
    z = rng.standard_normal((2, 7, 3, 16))
    R = gin.rope_table(np.arange(7), head_dim=16, theta=500000.0).numpy().astype(np.float64)
    got = orc.rope(z, R)
    # numpy complex product of adjacent pairs
    zc = z[..., 0::2] + 1j * z[..., 1::2]
    f = R[..., 0] + 1j * R[..., 1]
    prod = zc * f[None, :, None, :]
    ref = np.empty_like(z)
    ref[..., 0::2] = prod.real
    ref[..., 1::2] = prod.imag
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-14)
    # torch view_as_complex route (the quoted apply_rotary_emb's construction)
    zt = torch.from_numpy(z)
    zct = torch.view_as_complex(zt.reshape(*zt.shape[:-1], -1, 2).contiguous())
    ft = torch.complex(torch.from_numpy(R[..., 0]), torch.from_numpy(R[..., 1]))[None, :, None, :]
    reft = torch.view_as_real(zct * ft).flatten(3).numpy()
    np.testing.assert_allclose(got, reft, rtol=0, atol=1e-14)


def test_rope_preserves_pair_norm_and_is_identity_at_zero():
    rng = np.random.default_rng(2)
    z = rng.standard_normal((1, 9, 4, 128))
    R = gin.rope_table(np.arange(9)).numpy().astype(np.float64)
    out = orc.rope(z, R)
    n_in = z[..., 0::2] ** 2 + z[..., 1::2] ** 2
    n_out = out[..., 0::2] ** 2 + out[..., 1::2] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-6)  # table is fp32-rounded
    np.testing.assert_array_equal(out[:, 0], z[:, 0])  # R[0] = (1, 0) exactly


def test_rope_dot_depends_only_on_relative_position():
    rng = np.random.default_rng(3)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    # exact fp64 table so the property holds to rounding
    def table(p):
        j = np.arange(64)
        a = p * 500000.0 ** (-(2.0 * j) / 128)
        return np.stack([np.cos(a), np.sin(a)], -1)[None]
    def rot(v, p):
        return orc.rope(v.reshape(1, 1, 1, 128), table(p)).ravel()
    base = rot(q, 11) @ rot(k, 4)
    for shift in (1, 17, 300):
        np.testing.assert_allclose(rot(q, 11 + shift) @ rot(k, 4 + shift), base, rtol=1e-9, atol=1e-9)


# ---------------------------------------------------------------- head sharing (6-7)
def test_kv_head_map_is_repeat_interleave():
    idx = np.array([orc.kv_head(h, 4) for h in range(32)])
    np.testing.assert_array_equal(idx, np.repeat(np.arange(8), 4))
    np.testing.assert_array_equal(
        idx, torch.repeat_interleave(torch.arange(8), 4).numpy())
    # the quoted expand + reshape construction gives the same order
    kv = torch.arange(8).reshape(1, 1, 8, 1)
    expanded = kv[:, :, :, None, :].expand(1, 1, 8, 4, 1).reshape(1, 1, 32, 1)
    np.testing.assert_array_equal(idx, expanded.ravel().numpy())


# ---------------------------------------------------------------- mask (10)
def test_mask_is_triu_with_cached_zero_columns():
    T, sp = 5, 3
    M = orc.mask(T, T, 0, True)
    np.testing.assert_array_equal(M, np.triu(np.full((T, T), -np.inf), 1))
    M2 = orc.mask(T, sp + T, sp, True)
    ref = np.hstack([np.zeros((T, sp)), np.triu(np.full((T, T), -np.inf), 1)])
    np.testing.assert_array_equal(M2, ref)
    assert orc.mask(1, 9, 8, True) is None
    np.testing.assert_array_equal(orc.mask(T, T, 0, False), np.zeros((T, T)))


# ---------------------------------------------------------------- softmax (11)
def test_softmax_rows_sum_to_one_and_masked_entries_are_zero():
    x, wq, wk, wv, wo, R = tiny()
    _, ex = orc.attention_block(x, wq, wk, wv, wo, R, n_heads=8, keep=True)
    A = ex["A"]
    np.testing.assert_allclose(A.sum(-1), 1.0, rtol=0, atol=1e-14)
    T = x.shape[1]
    upper = np.triu(np.ones((T, T), dtype=bool), 1)
    assert np.all(A[..., upper] == 0.0)
    assert np.all(A[..., ~upper] > 0.0)


# ---------------------------------------------------------------- steps 6-12 as a library routine
@pytest.mark.parametrize("causal", [True, False])
def test_attention_core_equals_torch_sdpa_fp64(causal):
    x, wq, wk, wv, wo, R = tiny(seed=4, T=9)
    _, ex = orc.attention_block(x, wq, wk, wv, wo, R, causal=causal, n_heads=8, keep=True)
    q = torch.from_numpy(ex["Q_r"]).transpose(1, 2)
    k = torch.from_numpy(ex["K_r"]).transpose(1, 2)
    v = torch.from_numpy(ex["V"]).transpose(1, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, enable_gqa=True)
    ref = ref.transpose(1, 2).reshape(x.shape[0], x.shape[1], -1).numpy()
    np.testing.assert_allclose(ex["H"], ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- closed forms
def test_causal_row0_and_single_position_give_shared_value_head():
    x, wq, wk, wv, wo, R = tiny(seed=5, T=1)
    delta, ex = orc.attention_block(x, wq, wk, wv, wo, R, n_heads=8, keep=True)
    V, H = ex["V"], ex["H"].reshape(x.shape[0], 1, 8, -1)
    for h in range(8):
        np.testing.assert_array_equal(H[:, :, h], V[:, :, h // 4])
    VG = np.repeat(V, 4, axis=2).reshape(x.shape[0], 1, -1)
    np.testing.assert_allclose(delta, VG @ wo.T, rtol=1e-13, atol=1e-13)
    # row 0 of a causal prefill sees only itself
    x, wq, wk, wv, wo, R = tiny(seed=6, T=5)
    _, ex = orc.attention_block(x, wq, wk, wv, wo, R, n_heads=8, keep=True)
    H = ex["H"].reshape(2, 5, 8, -1)
    for h in range(8):
        np.testing.assert_allclose(H[:, 0, h], ex["V"][:, 0, h // 4], rtol=0, atol=1e-15)


def test_zero_query_weights_give_running_mean_of_values():
    x, wq, wk, wv, wo, R = tiny(seed=7, T=6)
    wq = np.zeros_like(wq)
    _, ex = orc.attention_block(x, wq, wk, wv, wo, R, n_heads=8, keep=True)
    V = ex["V"]
    H = ex["H"].reshape(2, 6, 8, -1)
    for t in range(6):
        for h in range(8):
            np.testing.assert_allclose(H[:, t, h], V[:, : t + 1, h // 4].mean(axis=1),
                                       rtol=1e-13, atol=1e-14)


def test_causality_is_bit_exact():
    x, wq, wk, wv, wo, R = tiny(seed=8, T=8)
    d0, _ = orc.attention_block(x, wq, wk, wv, wo, R, n_heads=8)
    for t in (0, 3, 6):
        xp = x.copy()
        xp[:, t + 1:] += np.random.default_rng(t).standard_normal(xp[:, t + 1:].shape) * 5
        d1, _ = orc.attention_block(xp, wq, wk, wv, wo, R, n_heads=8)
        np.testing.assert_array_equal(d1[:, : t + 1], d0[:, : t + 1])
        assert not np.array_equal(d1[:, t + 1:], d0[:, t + 1:])


def test_linear_in_output_weights():
    x, wq, wk, wv, wo, R = tiny(seed=9)
    wo2 = np.random.default_rng(99).standard_normal(wo.shape)
    a, _ = orc.attention_block(x, wq, wk, wv, wo, R, n_heads=8)
    b, _ = orc.attention_block(x, wq, wk, wv, wo2, R, n_heads=8)
    c, _ = orc.attention_block(x, wq, wk, wv, wo + 2.5 * wo2, R, n_heads=8)
    np.testing.assert_allclose(c, a + 2.5 * b, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- brute force
def brute_force(x, wq, wk, wv, wo, R, causal=True, start_pos=0, cache_k=None, cache_v=None,
                n_heads=8):
    """Element-by-element loops; head sharing materialised with numpy.repeat."""
    B, T, dim = x.shape
    d = wq.shape[0] // n_heads
    n_kv = wk.shape[0] // d

    def lin(v, w):  # y[o] = sum_i w[o, i] v[i]
        return [sum(w[o][i] * v[i] for i in range(len(v))) for o in range(len(w))]

    def rot(vec, t):
        out = list(vec)
        for j in range(d // 2):
            c, s = R[t][j][0], R[t][j][1]
            a, b = vec[2 * j], vec[2 * j + 1]
            out[2 * j] = c * a - s * b
            out[2 * j + 1] = s * a + c * b
        return out

    n_keys = start_pos + T
    Kc = np.zeros((B, n_keys, n_kv, d))
    Vc = np.zeros((B, n_keys, n_kv, d))
    if cache_k is not None:
        Kc[:, :start_pos] = cache_k[:, :start_pos]
        Vc[:, :start_pos] = cache_v[:, :start_pos]
    Q = np.zeros((B, T, n_heads, d))
    for b in range(B):
        for t in range(T):
            q = lin(list(x[b, t]), wq.tolist())
            k = lin(list(x[b, t]), wk.tolist())
            v = lin(list(x[b, t]), wv.tolist())
            for h in range(n_heads):
                Q[b, t, h] = rot(q[h * d:(h + 1) * d], t)
            for g in range(n_kv):
                Kc[b, start_pos + t, g] = rot(k[g * d:(g + 1) * d], t)
                Vc[b, start_pos + t, g] = v[g * d:(g + 1) * d]
    KG = np.repeat(Kc, n_heads // n_kv, axis=2)  # materialised repeat_kv
    VG = np.repeat(Vc, n_heads // n_kv, axis=2)
    out = np.zeros((B, T, dim))
    for b in range(B):
        Hrow = np.zeros((T, n_heads * d))
        for h in range(n_heads):
            for t in range(T):
                scores = []
                for s in range(n_keys):
                    val = sum(Q[b, t, h, i] * KG[b, s, h, i] for i in range(d)) / math.sqrt(d)
                    if causal and T > 1 and s > start_pos + t:
                        val = -math.inf
                    scores.append(val)
                mx = max(scores)
                e = [math.exp(v - mx) for v in scores]
                z = sum(e)
                for i in range(d):
                    Hrow[t, h * d + i] = sum(e[s] / z * VG[b, s, h, i] for s in range(n_keys))
        for t in range(T):
            out[b, t] = lin(list(Hrow[t]), wo.tolist())
    return out


@pytest.mark.parametrize("causal", [True, False])
def test_oracle_equals_brute_force(causal):
    x, wq, wk, wv, wo, R = tiny(seed=10, B=2, T=5, dim=16, n_heads=8, n_kv=2)
    got, _ = orc.attention_block(x, wq, wk, wv, wo, R, causal=causal, n_heads=8)
    ref = brute_force(x, wq, wk, wv, wo, R, causal=causal, n_heads=8)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_oracle_with_cache_equals_brute_force():
    x, wq, wk, wv, wo, R_all = tiny(seed=11, B=2, T=7, dim=16, n_heads=8, n_kv=2)
    rng = np.random.default_rng(12)
    sp, T = 4, 3
    ck = rng.standard_normal((2, 9, 2, 2))
    cv = rng.standard_normal((2, 9, 2, 2))
    xs, R = x[:, :T], R_all[sp:sp + T]
    got, ex = orc.attention_block(xs, wq, wk, wv, wo, R, start_pos=sp, cache_k=ck, cache_v=cv,
                                  n_heads=8)
    ref = brute_force(xs, wq, wk, wv, wo, R, start_pos=sp, cache_k=ck, cache_v=cv, n_heads=8)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)
    # cache writes landed at start_pos .. start_pos+T-1 and left the rest alone
    np.testing.assert_array_equal(ex["cache_k"][:, :sp], ck[:, :sp])
    np.testing.assert_array_equal(ex["cache_k"][:, sp + T:], ck[:, sp + T:])


# ---------------------------------------------------------------- consistency
def test_decode_equals_last_prefill_row():
    x, wq, wk, wv, wo, R = tiny(seed=13, B=2, T=7)
    full, ex = orc.attention_block(x, wq, wk, wv, wo, R, n_heads=8, keep=True)
    T = x.shape[1]
    S_max = T + 2
    ck = np.zeros((2, S_max, 2, 4))
    cv = np.zeros((2, S_max, 2, 4))
    ck[:, :T - 1] = ex["K_r"][:, :T - 1]
    cv[:, :T - 1] = ex["V"][:, :T - 1]
    dec, ex2 = orc.attention_decode(x[:, T - 1:T], wq, wk, wv, wo, R[T - 1:T], ck, cv, T - 1,
                                    n_heads=8)
    np.testing.assert_allclose(dec[:, 0], full[:, T - 1], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ex2["cache_k"][:, T - 1], ex["K_r"][:, T - 1], rtol=1e-13, atol=1e-14)


def test_chunked_prefill_equals_full_prefill():
    x, wq, wk, wv, wo, R = tiny(seed=14, B=2, T=9)
    full, _ = orc.attention_block(x, wq, wk, wv, wo, R, n_heads=8)
    T1 = 4
    ck = np.zeros((2, 9, 2, 4))
    cv = np.zeros((2, 9, 2, 4))
    _, e1 = orc.attention_block(x[:, :T1], wq, wk, wv, wo, R[:T1], cache_k=ck, cache_v=cv,
                                n_heads=8)
    d2, _ = orc.attention_block(x[:, T1:], wq, wk, wv, wo, R[T1:], start_pos=T1,
                                cache_k=e1["cache_k"], cache_v=e1["cache_v"], n_heads=8)
    np.testing.assert_allclose(d2, full[:, T1:], rtol=1e-12, atol=1e-13)


def test_row_subset_equals_full():
    x, wq, wk, wv, wo, R = tiny(seed=15, B=2, T=10)
    full, _ = orc.attention_block(x, wq, wk, wv, wo, R, n_heads=8)
    rows = [0, 3, 9]
    part, _ = orc.attention_block(x, wq, wk, wv, wo, R, rows=rows, n_heads=8)
    np.testing.assert_allclose(part, full[:, rows], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- planted mistakes
def _planted(monkeypatch, name, fn):
    monkeypatch.setattr(orc, name, fn)


def test_planted_rope_sign_error_is_caught(monkeypatch):
    good = orc.rope

    def bad(z, R):
        R = np.array(R, dtype=np.float64, copy=True)
        R[..., 1] *= -1.0
        return good(z, R)
    _planted(monkeypatch, "rope", bad)
    with pytest.raises(AssertionError):
        test_rope_equals_complex_product_numpy_and_torch()


def test_planted_head_map_error_is_caught(monkeypatch):
    # interleaved sharing (h mod n_kv) instead of blocks of n_rep consecutive heads
    _planted(monkeypatch, "kv_head", lambda h, n_rep: h % 8)
    with pytest.raises(AssertionError):
        test_kv_head_map_is_repeat_interleave()
    _planted(monkeypatch, "kv_head", lambda h, n_rep: h % 2)  # tiny block: 8 heads, 2 kv heads
    with pytest.raises(AssertionError):
        test_attention_core_equals_torch_sdpa_fp64(True)


def test_planted_mask_off_by_one_is_caught(monkeypatch):
    def bad(T, n_keys, start_pos, causal):
        if T == 1:
            return None
        M = np.zeros((T, n_keys))
        t = np.arange(T).reshape(-1, 1)
        s = np.arange(n_keys).reshape(1, -1)
        M[s >= start_pos + t] = -np.inf
        M[:, 0] = 0.0
        return M
    _planted(monkeypatch, "mask", bad)
    with pytest.raises(AssertionError):
        test_attention_core_equals_torch_sdpa_fp64(True)


def test_planted_transposed_projection_is_caught(monkeypatch):
    _planted(monkeypatch, "linear", lambda x, w: np.asarray(x, np.float64) @ np.asarray(w, np.float64))
    with pytest.raises((AssertionError, ValueError)):
        x, wq, wk, wv, wo, R = tiny(seed=10, B=1, T=3, dim=16, n_heads=8, n_kv=2)
        wq = wq[:, :16] if wq.shape[1] != 16 else wq
        got, _ = orc.attention_block(x, wq, wk, wv, wo, R, n_heads=8)
        ref = brute_force(x, wq, wk, wv, wo, R, n_heads=8)
        np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_planted_missing_scale_is_caught(monkeypatch):
    orig_softmax = orc.softmax_rows
    _planted(monkeypatch, "softmax_rows", lambda Sm: orig_softmax(Sm * math.sqrt(2.0)))
    with pytest.raises(AssertionError):
        test_attention_core_equals_torch_sdpa_fp64(False)


# ---------------------------------------------------------------- around the block
def test_rms_norm_constant_row_closed_form():
    # x = c * 1: mean x^2 = c^2, so y = w * c / sqrt(c^2 + eps) (a dropped eps, a sum instead
    # of a mean or a missing weight all change this value)
    c, eps = 0.003, 1e-5
    w = np.linspace(0.5, 1.5, 64)
    y = orc.rms_norm(np.full((1, 2, 64), c), w, eps)
    np.testing.assert_allclose(y, np.broadcast_to(w * c / math.sqrt(c * c + eps), (1, 2, 64)), rtol=1e-14)


def test_rms_norm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 4, 128)) * 7.0
    y = orc.rms_norm(x, np.ones(128), eps=0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-13)  # per row
    np.testing.assert_allclose(orc.rms_norm(2.5 * x, np.ones(128), eps=0.0), y, rtol=1e-13)
    # rows are normalised independently
    x2 = x.copy()
    x2[0, 0] *= 100.0
    y2 = orc.rms_norm(x2, np.ones(128), eps=0.0)
    np.testing.assert_allclose(y2[0, 1:], y[0, 1:], rtol=1e-14)
    np.testing.assert_allclose(y2[1:], y[1:], rtol=1e-14)


def test_rms_norm_equals_loops_and_torch():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((2, 3, 16))
    w = rng.standard_normal(16)
    eps = 1e-5
    ref = np.empty_like(x)
    for b in range(2):
        for t in range(3):
            ms = sum(v * v for v in x[b, t]) / 16
            ref[b, t] = [x[b, t, j] / math.sqrt(ms + eps) * w[j] for j in range(16)]
    np.testing.assert_allclose(orc.rms_norm(x, w, eps), ref, rtol=1e-13)
    xt = torch.from_numpy(x)
    tref = torch.nn.functional.rms_norm(xt, (16,), torch.from_numpy(w), eps) if hasattr(torch.nn.functional, "rms_norm") else None
    if tref is not None:
        np.testing.assert_allclose(orc.rms_norm(x, w, eps), tref.numpy(), rtol=1e-12)


def test_residual_block_adds_update_to_unnormalised_input():
    x, wq, wk, wv, wo, R = tiny(seed=21)
    w_norm = np.random.default_rng(3).standard_normal(x.shape[-1]) * 0.2 + 1.0
    h, _ = orc.attention_block_residual(x, w_norm, wq, wk, wv, wo, R, n_heads=8)
    delta, _ = orc.attention_block(orc.rms_norm(x, w_norm), wq, wk, wv, wo, R, n_heads=8)
    np.testing.assert_allclose(h, x + delta, rtol=1e-13, atol=1e-13)
    # W_O = 0: the block is the identity on the residual stream
    h0, _ = orc.attention_block_residual(x, w_norm, wq, wk, wv, np.zeros_like(wo), R, n_heads=8)
    np.testing.assert_array_equal(h0, x)
    # the update sees the normalised input: scaling a token row leaves its own update unchanged
    # (eps aside) while the residual scales, i.e. h(c x)[t] - c x[t] == h(x)[t] - x[t] for T = 1
    x1 = x[:, :1]
    a, _ = orc.attention_block_residual(x1, w_norm, wq, wk, wv, wo, R[:1], eps=0.0, n_heads=8)
    b, _ = orc.attention_block_residual(3.0 * x1, w_norm, wq, wk, wv, wo, R[:1], eps=0.0, n_heads=8)
    np.testing.assert_allclose(b - 3.0 * x1, a - x1, rtol=1e-11, atol=1e-12)


def test_residual_decode_equals_last_prefill_row():
    x, wq, wk, wv, wo, R = tiny(seed=22, T=5)
    w_norm = np.linspace(0.8, 1.2, x.shape[-1])
    full, _ = orc.attention_block_residual(x, w_norm, wq, wk, wv, wo, R, n_heads=8)
    ck = np.zeros((x.shape[0], 5, 2, 4))
    cv = np.zeros_like(ck)
    pre, ex = orc.attention_block_residual(x[:, :4], w_norm, wq, wk, wv, wo, R[:4], n_heads=8, cache_k=ck, cache_v=cv)
    dec, _ = orc.attention_decode_residual(x[:, 4:], w_norm, wq, wk, wv, wo, R[4:5], ex["cache_k"], ex["cache_v"], 4, n_heads=8)
    np.testing.assert_allclose(dec[:, 0], full[:, 4], rtol=1e-11, atol=1e-12)


def test_planted_norm_mistakes_are_caught(monkeypatch):
    c, eps = 0.003, 1e-5
    w = np.linspace(0.5, 1.5, 64)
    want = w * c / math.sqrt(c * c + eps)
    good = orc.rms_norm

    def no_eps(x, w, eps=orc.NORM_EPS):
        x = np.asarray(x, dtype=np.float64)
        return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) * w

    def sum_not_mean(x, w, eps=orc.NORM_EPS):
        x = np.asarray(x, dtype=np.float64)
        return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps) * w

    for bad in (no_eps, sum_not_mean):
        monkeypatch.setattr(orc, "rms_norm", bad)
        y = orc.rms_norm(np.full((1, 2, 64), c), w, eps)
        assert not np.allclose(y, want, rtol=1e-6)
    monkeypatch.setattr(orc, "rms_norm", good)


# ---------------------------------------------------------------- scaled RoPE table (Llama 3.1)
def test_scaled_frequencies_keep_fast_pairs_and_slow_down_slow_pairs():
    w = 500000.0 ** (-(2.0 * np.arange(64)) / 128)
    ws = gin.scaled_frequencies(w)
    wavelen = 2 * np.pi / w
    fast = wavelen < 8192 / 4
    slow = wavelen > 8192 / 1
    assert fast.any() and slow.any() and (~fast & ~slow).any()
    np.testing.assert_array_equal(ws[fast], w[fast])
    np.testing.assert_allclose(ws[slow], w[slow] / 8, rtol=1e-15)
    mid = ~fast & ~slow
    assert np.all(ws[mid] < w[mid]) and np.all(ws[mid] > w[mid] / 8)
    # never faster than the base frequency; the interpolation meets both ends continuously
    assert np.all(ws <= w)
    lo = gin.scaled_frequencies(np.array([2 * np.pi / (8192 / 4 + 1e-9), 2 * np.pi / (8192 - 1e-9)]))
    np.testing.assert_allclose(lo, [2 * np.pi / (8192 / 4), 2 * np.pi / 8192 / 8], rtol=1e-9)


def test_scaled_table_rows_are_rotations_and_identity_at_zero():
    R = gin.rope_table(np.arange(0, 40000, 997), scaled=True).numpy().astype(np.float64)
    np.testing.assert_allclose(R[..., 0] ** 2 + R[..., 1] ** 2, 1.0, atol=1e-6)
    np.testing.assert_array_equal(R[0, :, 0], 1.0)
    np.testing.assert_array_equal(R[0, :, 1], 0.0)
    # the fastest pair is unscaled, the slowest is 8x slower than unscaled
    Ru = gin.rope_table(np.arange(0, 40000, 997)).numpy().astype(np.float64)
    np.testing.assert_array_equal(R[:, 0], Ru[:, 0])
    assert not np.allclose(R[5:, 63], Ru[5:, 63])
