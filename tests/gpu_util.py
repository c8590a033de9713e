"""Shared helpers of the GPU parity tests: run the block through the C ABI on cuda:0 and
compare with the fp64 oracle under the block's tolerance."""
from __future__ import annotations

import numpy as np
import torch

from oracle import gqa_oracle as orc
from transformer_gqa_attention_gb300 import abi
from transformer_gqa_attention_gb300 import inputs as gin

DEV = "cuda:0"

# Acceptance bar for bf16 inputs / fp32 accumulation against the fp64 oracle:
#   max|gpu - ref| <= 2e-2 * max|ref|   and   sum|gpu - ref| / sum|ref| <= 5e-3.
TOL_MAX = 2e-2
TOL_REL_L1 = 5e-3
# Intermediates stored in bf16 (Q_r, K_r, V, H): one bf16 rounding (2^-9 relative) plus
# fp32 accumulation order.
TOL_BF16_REL_L1 = 4e-3
TOL_BF16_MAX = 1.5e-2


def metrics(gpu, ref):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    err = np.abs(g - r)
    return float(err.sum() / np.abs(r).sum()), float(err.max() / np.abs(r).max())


def assert_close(gpu, ref, rel_l1=TOL_REL_L1, max_ratio=TOL_MAX, what=""):
    g = np.asarray(gpu, dtype=np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    l1, mx = metrics(g, ref)
    assert l1 <= rel_l1 and mx <= max_ratio, f"{what}: rel-L1 {l1:.3e} (<= {rel_l1}), max {mx:.3e} (<= {max_ratio})"
    return l1, mx


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


class Block:
    """A context built on cuda:0 from the inputs' weights (copied into the library)."""

    def __init__(self, inp: gin.BlockInputs):
        self.w = [t.to(DEV) for t in (inp.wq, inp.wk, inp.wv, inp.wo)]
        self.ctx = abi.attn_create(*self.w)
        abi.attn_sync_status(self.ctx)
        self.w64 = [gin.to_f64(t) for t in (inp.wq, inp.wk, inp.wv, inp.wo)]

    def close(self):
        abi.attn_destroy(self.ctx)
        self.ctx = None

    def prefill(self, x, R, cache_k, cache_v, start_pos=0, causal=True):
        B, T = x.shape[0], x.shape[1]
        delta = torch.empty(B, T, 4096, dtype=torch.float32, device=DEV)
        abi.attn_prefill(self.ctx, x, B, T, R, causal, cache_k, cache_v, cache_k.shape[1],
                         start_pos, delta)
        abi.attn_sync_status(self.ctx)
        return delta

    def decode(self, x, R_row, cache_k, cache_v, start_pos):
        B = x.shape[0]
        delta = torch.empty(B, 1, 4096, dtype=torch.float32, device=DEV)
        abi.attn_decode(self.ctx, x, B, start_pos, R_row, cache_k, cache_v, cache_k.shape[1], delta)
        abi.attn_sync_status(self.ctx)
        return delta

    def intermediates(self, n_tok):
        """(Q_r, H) of the last call as bf16 tensors [n_tok, 4096] (copies)."""
        q_ptr, h_ptr = abi.attn_debug_buffers(self.ctx)
        return [device_view(ptr, (n_tok, 4096)).clone() for ptr in (q_ptr, h_ptr)]


class _CudaArray:
    def __init__(self, ptr, shape):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": "<i2",
                                         "data": (int(ptr), False), "version": 3, "strides": None}


def device_view(ptr, shape) -> torch.Tensor:
    """Zero-copy bf16 view of library-owned device memory."""
    return torch.as_tensor(_CudaArray(ptr, shape), device=DEV).view(torch.bfloat16)


def empty_cache(B, S_max):
    shape = (B, S_max, gin.N_KV_HEADS, gin.HEAD_DIM)
    # NaN-filled: any read of a position the call does not own poisons the result
    return (torch.full(shape, float("nan"), dtype=torch.bfloat16, device=DEV),
            torch.full(shape, float("nan"), dtype=torch.bfloat16, device=DEV))


def oracle_prefill(blk: Block, inp: gin.BlockInputs, rows=None, causal=True, keep=False):
    wq, wk, wv, wo = blk.w64
    return orc.attention_block(gin.to_f64(inp.x), wq, wk, wv, wo, gin.to_f64(inp.R), causal=causal,
                               rows=rows, keep=keep)


def sample_rows(T, n=48, seed=0):
    rng = np.random.default_rng(seed)
    fixed = {0, 1, 63, 64, 127, 128, 129, T // 2, T - 2, T - 1}
    rows = set(r for r in fixed if 0 <= r < T)
    rows |= set(rng.integers(0, T, size=n).tolist())
    return np.array(sorted(rows))
