"""The error floor of the block's residual form under bf16 storage (CPU, fp64 emulation).

The GPU stores Q_r, K_r, V, P and H in bf16 (the pages' activation dtype), and the residual
form adds one rounding more: a bf16 tensor-core GEMM needs either attention_norm(x) or the
projection weights in bf16, so either the normalised activation or the folded weight
W diag(w) is rounded once (the library folds the weight).  This test emulates exactly those
roundings in fp64 and compares the update h - x with the oracle's, which pins the floor the
GPU tolerance in tests/test_gpu_residual.py is set against:
  - block alone (five roundings): ~4.0e-3 rel-L1, under the block's 5e-3 with >= 20 % margin;
  - folded weight (the library's choice) and a single rounding of the normalised activation
    both land at ~5.3e-3 (5.75e-3 on the T = 2048 workload), above 5e-3: with bf16 GEMM
    inputs the extra rounding cannot be avoided;
  - rounding twice as the quoted model's RMSNorm does (x / rms to bf16, then times w to
    bf16) is worse, ~6.8e-3;
so the update is held to 7e-3 = about 1.2 x the largest floor, the block's own margin."""
import numpy as np
import torch

from oracle import gqa_oracle as orc
from tests.test_gpu_residual import TOL_UPDATE_REL_L1
from transformer_gqa_attention_gb300 import inputs as gin

BLOCK_TOL = 5e-3
MARGIN = 1.2


def bf(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def emulate_update(X, Wq, Wk, Wv, wo, R, row_scale=1.0):
    """Delta with the GPU's roundings: projections of X by the given weights (times the row
    scale), then Q_r, K_r, V, P and H rounded to bf16, causal softmax with an fp32-style
    unrounded row sum, fp64 elsewhere."""
    B, T, _ = X.shape
    Q = row_scale * (X @ Wq.T)
    K = row_scale * (X @ Wk.T)
    V = bf((row_scale * (X @ Wv.T)).reshape(B, T, 8, 128))
    Qr = bf(orc.rope(Q.reshape(B, T, 32, 128), R))
    Kr = bf(orc.rope(K.reshape(B, T, 8, 128), R))
    M = orc.mask(T, T, 0, True)
    H = np.empty((B, T, 32, 128))
    for b in range(B):
        for h in range(32):
            S = Qr[b, :, h] @ Kr[b, :, h // 4].T / np.sqrt(128) + M
            e = np.exp(S - S.max(-1, keepdims=True))
            H[b, :, h] = bf((bf(e) @ V[b, :, h // 4]) / e.sum(-1, keepdims=True))
    return H.reshape(B, T, 4096) @ wo.T


def rel_l1(a, r):
    return float(np.abs(a - r).sum() / np.abs(r).sum())


def test_residual_update_floor_sets_its_tolerance():
    inp = gin.make_custom(seed=600, B=1, T=300)
    x = gin.to_f64(inp.x)
    wq, wk, wv, wo = (gin.to_f64(t) for t in (inp.wq, inp.wk, inp.wv, inp.wo))
    wn = gin.to_f64(gin.norm_weight(600))
    R = gin.to_f64(inp.R)
    ref, _ = orc.attention_block_residual(x, wn, wq, wk, wv, wo, R)
    upd = ref - x
    r = 1.0 / np.sqrt(np.mean(x * x, -1, keepdims=True) + orc.NORM_EPS)
    y = x * r * wn
    five = rel_l1(emulate_update(y, wq, wk, wv, wo, R), upd)
    folded = rel_l1(emulate_update(x, bf(wq * wn), bf(wk * wn), bf(wv * wn), wo, R, row_scale=r), upd)
    act_once = rel_l1(emulate_update(bf(y), wq, wk, wv, wo, R), upd)
    act_twice = rel_l1(emulate_update(bf(bf(x * r) * wn), wq, wk, wv, wo, R), upd)
    assert 3.5e-3 < five < BLOCK_TOL / MARGIN
    # one extra rounding of either operand: the same floor, above the block's bar
    assert BLOCK_TOL < folded < 6e-3 and abs(folded - act_once) < 2e-4
    assert act_twice > folded + 1e-3
    # the GPU tolerance on the update keeps the block's margin over the largest floor seen
    # (5.75e-3 on the T = 2048 workload, where the block alone is 4.35e-3)
    assert TOL_UPDATE_REL_L1 >= MARGIN * 5.75e-3 and TOL_UPDATE_REL_L1 <= 7e-3
