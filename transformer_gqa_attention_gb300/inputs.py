"""Seeded synthetic inputs for the Llama-3 8B grouped-query attention block.

This module only draws numbers: it holds none of the block's arithmetic, so both the
CUDA path and the fp64 oracle can be fed from it without sharing any computation.

Shapes follow the "Llama 3.1 8B · Grouped-query attention" page (in/out contract:
x [B,T,4096], R [T,64 pairs]; parameter table: W_Q 4096x4096, W_K and W_V 4096x(8x128),
W_O 4096x4096) and the catalogue entry quoted there (dim 4096, n_heads 32,
n_kv_heads 8, rope_theta 500000).  Weights use the [out, in] storage of the quoted
fairscale linear layers ("we allocate the transpose").

Draw order for one workload, from one ``torch.Generator('cpu').manual_seed(seed)``:
x, W_Q, W_K, W_V, W_O, then (decode only) cache_K, cache_V.  Each draw is
``randn(float32) * std`` rounded to bf16 with round-to-nearest-even.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

DIM = 4096
N_HEADS = 32
N_KV_HEADS = 8
HEAD_DIM = DIM // N_HEADS  # 128
N_PAIRS = HEAD_DIM // 2  # 64
ROPE_THETA = 500000.0

X_STD = 1.0
W_STD = 0.02
CACHE_STD = 1.0


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: a prefill of B sequences of T tokens, or a decode step."""

    name: str
    kind: str  # "prefill" | "decode"
    B: int
    T: int
    seed: int
    causal: bool = True
    start_pos: int = 0
    S_max: int = 0  # 0 -> start_pos + T
    residual: bool = False  # attention_norm in front and the residual add behind
    n_kv: int = 8  # kv groups run: 8 = the whole block; fewer = one tensor-parallel shard

    @property
    def s_max(self) -> int:
        return self.S_max if self.S_max else self.start_pos + self.T

    @property
    def n_tok(self) -> int:
        return self.B * self.T


# The workloads the block is measured and checked on: the five shapes of the block itself,
# then two of them through the residual form, shards of a head split, and prefills that
# continue a cache.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("prefill_b1_t16", "prefill", B=1, T=16, seed=0),
        Workload("prefill_b1_t2048", "prefill", B=1, T=2048, seed=1),
        Workload("prefill_b4_t8192", "prefill", B=4, T=8192, seed=2),
        Workload("decode_b64_pos4095", "decode", B=64, T=1, seed=3, start_pos=4095, S_max=4096),
        Workload("prefill_b1_t32768", "prefill", B=1, T=32768, seed=4),
        # the same shapes through the block's residual form (attention_norm in front, the
        # residual add behind); x is then the residual stream
        Workload("prefill_b1_t2048_residual", "prefill", B=1, T=2048, seed=1, residual=True),
        Workload("decode_b64_pos4095_residual", "decode", B=64, T=1, seed=3, start_pos=4095, S_max=4096,
                 residual=True),
        # one rank's share of a head-sharded 8-way (1 kv group) or 2-way (4 kv groups) split:
        # the same inputs, the shard's weight slices and its own cache
        Workload("prefill_b1_t32768_tp8", "prefill", B=1, T=32768, seed=4, n_kv=1),
        Workload("prefill_b1_t32768_tp2", "prefill", B=1, T=32768, seed=4, n_kv=4),
        Workload("prefill_b1_t2048_tp8", "prefill", B=1, T=2048, seed=1, n_kv=1),
        Workload("decode_b64_pos4095_tp8", "decode", B=64, T=1, seed=3, start_pos=4095, S_max=4096, n_kv=1),
        # prefills continuing a cache (chunked prefill): the last 2048-token chunk of a
        # 32768-token prompt, and 16 new tokens of 4 sequences after 4080 cached positions
        # (e.g. verifying drafted tokens); the cached positions are drawn like a decode cache
        Workload("prefill_b1_t2048_pos30720", "prefill", B=1, T=2048, seed=5, start_pos=30720, S_max=32768),
        Workload("prefill_b4_t16_pos4080", "prefill", B=4, T=16, seed=6, start_pos=4080, S_max=4096),
    ]
}


def _draw(gen: torch.Generator, shape, std: float) -> torch.Tensor:
    return (torch.randn(*shape, generator=gen, dtype=torch.float32) * std).to(torch.bfloat16)


@dataclass
class BlockInputs:
    x: torch.Tensor  # [B, T, 4096] bf16
    wq: torch.Tensor  # [4096, 4096] bf16, [out, in]
    wk: torch.Tensor  # [1024, 4096] bf16
    wv: torch.Tensor  # [1024, 4096] bf16
    wo: torch.Tensor  # [4096, 4096] bf16
    R: torch.Tensor  # [T, 64, 2] fp32 (cos, sin) for positions start_pos .. start_pos+T-1
    cache_k: torch.Tensor | None = None  # [B, S_max, 8, 128] bf16 (decode: pre-filled)
    cache_v: torch.Tensor | None = None
    meta: dict = field(default_factory=dict)


# Llama 3.1 frequency scaling (the catalogue's use_scaled_rope: True).  The pages show the
# flag and the scaled frequency w' in the RoPE step but not the rule; this is the rule Meta
# published with Llama 3.1 (an external reading): wavelengths shorter than the original
# context / high_freq_factor keep their frequency, those longer than original context /
# low_freq_factor are slowed by `factor`, and the band in between is interpolated linearly
# in (original context / wavelength).
SCALE_FACTOR = 8.0
SCALE_LOW_FREQ_FACTOR = 1.0
SCALE_HIGH_FREQ_FACTOR = 4.0
SCALE_ORIGINAL_CONTEXT = 8192.0


def scaled_frequencies(w: np.ndarray) -> np.ndarray:
    """The Llama 3.1 scaled frequencies w' for base frequencies w (fp64)."""
    w = np.asarray(w, dtype=np.float64)
    wavelen = 2.0 * np.pi / w
    low_wavelen = SCALE_ORIGINAL_CONTEXT / SCALE_LOW_FREQ_FACTOR
    high_wavelen = SCALE_ORIGINAL_CONTEXT / SCALE_HIGH_FREQ_FACTOR
    smooth = (SCALE_ORIGINAL_CONTEXT / wavelen - SCALE_LOW_FREQ_FACTOR) / (SCALE_HIGH_FREQ_FACTOR - SCALE_LOW_FREQ_FACTOR)
    mid = (1.0 - smooth) * w / SCALE_FACTOR + smooth * w
    return np.where(wavelen < high_wavelen, w, np.where(wavelen > low_wavelen, w / SCALE_FACTOR, mid))


def rope_table(positions, head_dim: int = HEAD_DIM, theta: float = ROPE_THETA, scaled: bool = False) -> torch.Tensor:
    """Rotation table R[t, j] = (cos(p_t w_j), sin(p_t w_j)), w_j = theta^(-2j/head_dim)
    (with ``scaled``, the Llama 3.1 frequencies scaled_frequencies(w)).

    The pages name R as an input of the block ([T positions, 64 pairs]) but do not print
    its generator; the default is the standard unscaled form with the catalogue's theta.
    Angles are formed in fp64 and cos/sin rounded once to fp32.  Both the CUDA path and the
    oracle read this same array, so the choice of generator does not affect parity.
    """
    p = np.asarray(positions, dtype=np.float64).reshape(-1, 1)
    j = np.arange(head_dim // 2, dtype=np.float64).reshape(1, -1)
    w = theta ** (-(2.0 * j) / head_dim)
    if scaled:
        w = scaled_frequencies(w)
    ang = p * w
    out = np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)
    return torch.from_numpy(np.ascontiguousarray(out))


def make_weights(gen: torch.Generator, dim: int = DIM, n_heads: int = N_HEADS,
                 n_kv_heads: int = N_KV_HEADS):
    hd = dim // n_heads
    wq = _draw(gen, (n_heads * hd, dim), W_STD)
    wk = _draw(gen, (n_kv_heads * hd, dim), W_STD)
    wv = _draw(gen, (n_kv_heads * hd, dim), W_STD)
    wo = _draw(gen, (dim, n_heads * hd), W_STD)
    return wq, wk, wv, wo


def make_inputs(w: Workload | str, *, T: int | None = None, B: int | None = None) -> BlockInputs:
    """Draw the inputs of a workload.  ``T``/``B`` override the sizes (same seed and draw
    order) so that small parity cases keep the workload's value distributions."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    Bv = w.B if B is None else B
    Tv = w.T if T is None else T
    gen = torch.Generator("cpu").manual_seed(w.seed)
    x = _draw(gen, (Bv, Tv, DIM), X_STD)
    wq, wk, wv, wo = make_weights(gen)
    cache_k = cache_v = None
    s_max = w.S_max if w.S_max else w.start_pos + Tv
    if w.kind == "decode" or w.start_pos > 0:
        cache_k = _draw(gen, (Bv, s_max, N_KV_HEADS, HEAD_DIM), CACHE_STD)
        cache_v = _draw(gen, (Bv, s_max, N_KV_HEADS, HEAD_DIM), CACHE_STD)
    R = rope_table(np.arange(w.start_pos, w.start_pos + Tv))
    return BlockInputs(x, wq, wk, wv, wo, R, cache_k, cache_v,
                       meta=dict(name=w.name, kind=w.kind, B=Bv, T=Tv, seed=w.seed,
                                 causal=w.causal, start_pos=w.start_pos, S_max=s_max))


def make_custom(seed: int, B: int, T: int, *, start_pos: int = 0, S_max: int | None = None,
                fill_cache: bool = False) -> BlockInputs:
    """Inputs for an arbitrary (B, T, start_pos) case with the same distributions."""
    gen = torch.Generator("cpu").manual_seed(seed)
    x = _draw(gen, (B, T, DIM), X_STD)
    wq, wk, wv, wo = make_weights(gen)
    s_max = S_max if S_max else start_pos + T
    cache_k = cache_v = None
    if fill_cache:
        cache_k = _draw(gen, (B, s_max, N_KV_HEADS, HEAD_DIM), CACHE_STD)
        cache_v = _draw(gen, (B, s_max, N_KV_HEADS, HEAD_DIM), CACHE_STD)
    R = rope_table(np.arange(start_pos, start_pos + T))
    return BlockInputs(x, wq, wk, wv, wo, R, cache_k, cache_v,
                       meta=dict(name=f"custom_s{seed}_b{B}_t{T}_p{start_pos}", kind="prefill",
                                 B=B, T=T, seed=seed, causal=True, start_pos=start_pos,
                                 S_max=s_max))


NORM_W_STD = 0.1


def norm_weight(seed: int, dim: int = DIM) -> torch.Tensor:
    """attention_norm weight [dim] bf16 = 1 + 0.1 N(0, 1), from its own generator (seeded
    from the workload seed) so that the block's inputs keep their draw order."""
    gen = torch.Generator("cpu").manual_seed(seed + (1 << 20))
    return (1.0 + torch.randn(dim, generator=gen, dtype=torch.float32) * NORM_W_STD).to(torch.bfloat16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a bf16/fp32 CPU tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
