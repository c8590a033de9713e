"""The FMA-pipe exponential of the prefill softmax on the GPU (attn_debug_exp2): the device
cubic agrees with its step-by-step fp32 emulation (to one rounding of the final fma), stays
within the fit's relative-error bound of exact 2^a, and agrees with the multi-function
unit's ex2.approx to that bound, over the inputs the softmax can pass it."""
import numpy as np
import pytest
import torch

from transformer_gqa_attention_gb300 import abi
from transformer_gqa_attention_gb300.csrc import fit_exp2_poly as fit

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from transformer_gqa_attention_gb300 import _build
    _build.build()


def test_fma_exp2_matches_emulation_bound_and_ex2():
    a = np.concatenate([np.linspace(-125.0, 8.0, 2_000_001, dtype=np.float32),
                        np.random.default_rng(1).uniform(-40, 8, 999_999).astype(np.float32)])
    ad = torch.from_numpy(a).to(DEV)
    out_fma = torch.empty_like(ad)
    out_mufu = torch.empty_like(ad)
    abi.attn_debug_exp2(ad, out_fma, out_mufu)
    torch.cuda.synchronize()
    got = out_fma.cpu().numpy()
    mufu = out_mufu.cpu().numpy().astype(np.float64)
    emu = fit.exp2_emulated(a)
    # the emulation's fma rounds the exact product-sum once through fp64: at most 1 ulp apart
    ulps = np.abs(got.view(np.int32).astype(np.int64) - emu.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1
    exact = np.exp2(a.astype(np.float64))
    assert np.abs(got / exact - 1).max() <= 7.6e-5
    assert np.abs(got / mufu - 1).max() <= 7.6e-5 + 2e-6  # ex2.approx is within ~2^-22 of exact
