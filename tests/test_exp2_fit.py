"""The FMA-pipe exponential of the prefill softmax (CPU): the cubic's coefficients in the
kernel source are the ones the committed Remez fit produces, and the device sequence,
emulated step by step in fp32, stays within its relative-error bound over every input the
softmax can pass it (a = s * log2(e) / sqrt(128) - m with the running maximum m at most 8
below the row's maximum, so a <= 8; finite; inputs below -125 are clamped)."""
import os
import re

import numpy as np

from transformer_gqa_attention_gb300.csrc import fit_exp2_poly as fit

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BOUND = 7.6e-5  # levelled minimax error 7.48e-5 plus the fp32 evaluation


def _source_coefficients():
    src = open(os.path.join(ROOT, "transformer_gqa_attention_gb300", "csrc", "ptx.cuh")).read()
    body = src[src.index("float2 exp2_fma2("):]
    vals = dict(re.findall(r"\b(c[0-3]) = (0x[0-9a-fp.+-]+)f", body))
    return np.array([float.fromhex(vals[f"c{i}"]) for i in range(4)], dtype=np.float32)


def test_kernel_constants_are_the_fit():
    np.testing.assert_array_equal(_source_coefficients(), fit.coefficients_f32())


def test_fit_is_minimax_levelled():
    c, E = fit.remez_relative()
    x = np.linspace(-0.5, 0.5, 100001)
    err = np.polyval(c[::-1], x) / np.exp2(x) - 1
    assert abs(np.abs(err).max() - E) < 1e-9 and 7e-5 < E < 8e-5
    # a quadratic cannot meet the bf16 budget of P; the cubic can, with ~25x margin
    assert fit.remez_relative(degree=2)[1] > 1e-3


def test_emulated_device_sequence_within_bound():
    a = np.concatenate([np.linspace(-125.0, 8.0, 4_000_001, dtype=np.float32),
                        np.random.default_rng(0).uniform(-30, 8, 1_000_000).astype(np.float32),
                        np.array([-0.5, 0.5, -1.5, 1.5, 7.5, 8.0, -124.5, -125.0], dtype=np.float32)])
    got = fit.exp2_emulated(a, _source_coefficients()).astype(np.float64)
    rel = np.abs(got / np.exp2(a.astype(np.float64)) - 1)
    assert rel.max() <= BOUND
    # exact powers of two come out exact up to the cubic's value at 0
    ints = np.arange(-125, 9, dtype=np.float32)
    got_i = fit.exp2_emulated(ints, _source_coefficients()).astype(np.float64)
    np.testing.assert_allclose(got_i / np.exp2(ints.astype(np.float64)), float(_source_coefficients()[0]), rtol=0, atol=0)


def test_clamp_below_range():
    got = fit.exp2_emulated(np.array([-126.0, -200.0, -1e30, -np.inf], dtype=np.float32), _source_coefficients())
    assert np.all(np.isfinite(got)) and np.all(got > 0) and np.all(got <= 2.0 ** -124)
