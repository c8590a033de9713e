"""fp64 CPU oracle for the Llama-3 8B grouped-query attention block forward.

TEST INFRASTRUCTURE ONLY.  This module is the slow, obviously-correct statement of what
the block computes.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
may import it; the CUDA library never calls it and shares no code with it.

Every step follows the step list "All 13 steps" on the page "Llama 3.1 8B ·
Grouped-query attention" (atlas.klimoza.dev/models/llama-3.1/block?inspect=attention),
in the page's order and notation, and its in/out contract (x [B,T,4096], R [T,64 pairs],
M [T queries, T keys] -> Delta_attn [B,T,4096]).  The quoted code on that page
(llama/model.py ``Attention.forward``, ``apply_rotary_emb``, ``repeat_kv``, the mask built
in ``Transformer.forward``) fixes the details the equations leave open: the [out, in]
weight storage of ``F.linear``, the adjacent-pair complex view used by RoPE, the
``repeat_interleave`` head sharing, and the key axis growing to ``cache_len + seqlen``
with a KV cache.

Everything is float64.  Inputs (bf16 / fp32 arrays) widen exactly; nothing is rounded
back to a narrower type, so the oracle is the exact result up to fp64 rounding order.
Library primitives used as single steps: ``numpy.matmul`` for the projections, the
score product and the value product.  No blocking, fusion or reordering beyond that.

Readings taken where the page is silent (each also listed in the design notes):
  * The softmax is evaluated with the row maximum subtracted first; this is the same
    value as the page's exp(S_m)/sum exp(S_m) and avoids overflow.
  * With a KV cache of ``start_pos`` earlier positions, the key axis holds positions
    0 .. start_pos+T-1; query row t sits at absolute position start_pos+t and is masked
    (-inf) for keys s > start_pos+t when causal.  With T == 1 there is no mask (the quoted
    ``Transformer.forward`` builds one only when seqlen > 1).
  * The cache holds rotated keys and unrotated values; this call's keys/values are
    written at positions start_pos .. start_pos+T-1 before attention reads them.
  * R rows are the rotation for this call's positions: R[t] belongs to position
    start_pos+t.
"""
from __future__ import annotations

import math

import numpy as np

# Catalogue dimensions quoted on the page (sku_list.py arch_args for Llama 3.1 8B).
DIM = 4096
N_HEADS = 32
N_KV_HEADS = 8


def f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------------------
# Steps 1-3: Q = x W_Q, K = x W_K, V = x W_V.
# The quoted fairscale layers store each weight as [out, in] and apply F.linear, i.e.
# y = x A^T ("we allocate the transpose").
# --------------------------------------------------------------------------------------
def linear(x: np.ndarray, w_out_in: np.ndarray) -> np.ndarray:
    return f64(x) @ f64(w_out_in).T


# --------------------------------------------------------------------------------------
# Steps 4-5: RoPE, the 2x2 pair rotation
#   [z'_2j; z'_2j+1] = [[cos, -sin], [sin, cos]] [z_2j; z_2j+1]
# applied to every head slice of Q and of K (not V).  Pairs are adjacent elements
# (apply_rotary_emb reshapes the last axis to (-1, 2) before the complex view).
# R[t, j] = (cos(t w_j), sin(t w_j)) is an input of the block.
# --------------------------------------------------------------------------------------
def rope(z: np.ndarray, R: np.ndarray) -> np.ndarray:
    """z: [B, T, heads, d]; R: [T, d/2, 2] -> rotated z (float64)."""
    z = f64(z)
    R = f64(R)
    c = R[:, :, 0][None, :, None, :]  # [1, T, 1, d/2]
    s = R[:, :, 1][None, :, None, :]
    even = z[..., 0::2]
    odd = z[..., 1::2]
    out = np.empty_like(z)
    out[..., 0::2] = c * even - s * odd
    out[..., 1::2] = s * even + c * odd
    return out


# --------------------------------------------------------------------------------------
# Steps 6-7: K_G[h] = K_r[floor(h/4)], V_G[h] = V[floor(h/4)].  n_rep = n_heads/n_kv_heads.
# --------------------------------------------------------------------------------------
def kv_head(h: int, n_rep: int) -> int:
    return h // n_rep


# --------------------------------------------------------------------------------------
# Step 10: the mask M.  Causal: -inf where key s lies after the query's absolute position
# start_pos + t (the quoted triu(diagonal=1) hstacked after start_pos zero columns);
# otherwise 0.  None when the call has a single position.
# --------------------------------------------------------------------------------------
def mask(T: int, n_keys: int, start_pos: int, causal: bool) -> np.ndarray | None:
    if T == 1:
        return None
    M = np.zeros((T, n_keys), dtype=np.float64)
    if causal:
        t = np.arange(T).reshape(-1, 1)
        s = np.arange(n_keys).reshape(1, -1)
        M[s > start_pos + t] = -np.inf
    return M


# --------------------------------------------------------------------------------------
# Step 11: A = exp(S_m) / sum_u exp(S_m) over the key axis.
# --------------------------------------------------------------------------------------
def softmax_rows(Sm: np.ndarray) -> np.ndarray:
    m = np.max(Sm, axis=-1, keepdims=True)
    e = np.exp(Sm - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attention_block(x, wq, wk, wv, wo, R, *, causal: bool = True, start_pos: int = 0,
                    cache_k=None, cache_v=None, rows=None, n_heads: int = N_HEADS,
                    keep: bool = False):
    """Delta_attn for x [B, T, dim] (already the attention_norm output).

    wq [n_heads*d, dim], wk/wv [n_kv*d, dim], wo [dim, n_heads*d] ([out, in] storage).
    R [T, d/2, 2]: rotation for positions start_pos .. start_pos+T-1.
    cache_k / cache_v [B, S_max, n_kv, d]: earlier positions (rotated K, plain V); copies
    are updated with this call's keys/values and returned.  Without a cache, start_pos
    must be 0 and the keys are this call's tokens.
    rows: optional query rows (indices into 0..T-1) to evaluate; all rows by default.

    Returns (delta [B, len(rows), dim], extras) where extras holds the updated caches and,
    with keep=True, Q_r [B,rows,H,d], K_r and V [B,T,n_kv,d], A [B,H,rows,keys] and
    H [B,rows,H*d].
    """
    x = f64(x)
    B, T, dim = x.shape
    d = wq.shape[0] // n_heads
    n_kv = wk.shape[0] // d
    n_rep = n_heads // n_kv
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    nr = len(rows)
    R = f64(R)

    # Steps 2-3, 5: this call's keys and values (all T positions).
    K = linear(x, wk).reshape(B, T, n_kv, d)
    V = linear(x, wv).reshape(B, T, n_kv, d)
    K_r = rope(K, R)

    n_keys = start_pos + T
    if cache_k is not None:
        ck = f64(cache_k).copy()
        cv = f64(cache_v).copy()
        assert ck.shape[1] >= n_keys
        ck[:, start_pos:start_pos + T] = K_r
        cv[:, start_pos:start_pos + T] = V
        keys, vals = ck[:, :n_keys], cv[:, :n_keys]
    else:
        assert start_pos == 0, "a start_pos > 0 needs the cached keys/values"
        ck = cv = None
        keys, vals = K_r, V

    # Steps 1, 4: queries for the requested rows.
    Q = linear(x[:, rows], wq).reshape(B, nr, n_heads, d)
    Q_r = rope(Q, R[rows])

    M = mask(T, n_keys, start_pos, causal)
    Mr = None if M is None else M[rows]
    sqrt_d = math.sqrt(d)

    H = np.empty((B, nr, n_heads, d), dtype=np.float64)
    A_keep = np.empty((B, n_heads, nr, n_keys)) if keep else None
    for b in range(B):
        for h in range(n_heads):
            g = kv_head(h, n_rep)                      # steps 6-7
            S = Q_r[b, :, h, :] @ keys[b, :, g, :].T   # step 8
            Ss = S / sqrt_d                            # step 9
            Sm = Ss if Mr is None else Ss + Mr         # step 10
            A = softmax_rows(Sm)                       # step 11
            H[b, :, h, :] = A @ vals[b, :, g, :]       # step 12
            if keep:
                A_keep[b, h] = A
    Hm = H.reshape(B, nr, n_heads * d)                 # step 13 (merge heads)
    delta = linear(Hm, wo)                             # step 14: Delta = H W_O
    extras = {"cache_k": ck, "cache_v": cv}
    if keep:
        extras.update(Q_r=Q_r, K_r=K_r, V=V, A=A_keep, H=Hm)
    return delta, extras


def attention_decode(x, wq, wk, wv, wo, R_row, cache_k, cache_v, start_pos: int, *,
                     n_heads: int = N_HEADS, keep: bool = False):
    """One new token per sequence at position start_pos: x [B, 1, dim], R_row [1, d/2, 2],
    caches [B, S_max, n_kv, d] holding positions < start_pos.  Same steps with T = 1."""
    return attention_block(x, wq, wk, wv, wo, R_row, causal=True, start_pos=start_pos,
                           cache_k=cache_k, cache_v=cache_v, n_heads=n_heads, keep=keep)


# --------------------------------------------------------------------------------------
# Around the block.  The transformer block feeds the attention block attention_norm(x)
# and adds its update back: h = x + Delta_attn (page "Llama 3.1 8B · Merge and project",
# code excerpt model.py 236-248 and "Contextual evidence from Output projection").  The
# RMSNorm body is not on the pages; its plainest reading, with the catalogue's
# norm_eps = 1e-05 (sku_list.py arch_args on the same page), is
#     attention_norm(x) = x / sqrt(mean_j x_j^2 + eps) * w      (per token row, j over dim)
# --------------------------------------------------------------------------------------
NORM_EPS = 1e-5


def rms_norm(x, w, eps: float = NORM_EPS) -> np.ndarray:
    x = f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * f64(w)


def attention_block_residual(x, w_norm, wq, wk, wv, wo, R, *, eps: float = NORM_EPS, rows=None, **kw):
    """h = x + Delta_attn(attention_norm(x)) for the residual stream x [B, T, dim].

    Same keyword arguments as attention_block (causal, start_pos, caches, ...); returns
    (h [B, len(rows), dim], extras)."""
    x = f64(x)
    delta, extras = attention_block(rms_norm(x, w_norm, eps), wq, wk, wv, wo, R, rows=rows, **kw)
    xr = x if rows is None else x[:, np.asarray(rows, dtype=np.int64)]
    return xr + delta, extras


def attention_decode_residual(x, w_norm, wq, wk, wv, wo, R_row, cache_k, cache_v, start_pos: int, *,
                              eps: float = NORM_EPS, n_heads: int = N_HEADS):
    """Decode form of attention_block_residual (x [B, 1, dim])."""
    return attention_block_residual(x, w_norm, wq, wk, wv, wo, R_row, eps=eps, causal=True,
                                    start_pos=start_pos, cache_k=cache_k, cache_v=cache_v, n_heads=n_heads)


def param_count(wq, wk, wv, wo) -> int:
    """Learned parameters of one block: the four projection matrices (no biases)."""
    return sum(math.prod(tuple(w.shape)) for w in (wq, wk, wv, wo))
