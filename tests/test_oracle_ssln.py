"""Pins for the oracle's SkipSimplifiedLayerNormalization.

Operator (com.microsoft.SkipSimplifiedLayerNormalization README, Description,
Inputs, Outputs, Attributes): S = input + skip (+ bias); output =
S / sqrt(mean(S^2) + epsilon) * gamma over the last axis; the optional second
output is S.  The pins are hand-derived closed forms on the usage example's
shape, an invariant of RMS normalization, torch's float64 rms_norm on the same
S, scale invariance, and the sign of zero when the bias is absent.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from residual_add_normalization_gb300 import synthetic

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "usage_examples.json")))["skip_simplified_layer_norm"]


def _golden_inputs(dtype):
    shape = tuple(GOLDEN["input"])
    assert shape == (2, 4)
    x = np.array([[2, 1, 0.5, -1], [-2, 0.5, 0, 3]], dtype)
    sk = np.array([[1, 3, -0.5, 1], [1, 0.5, -1, -2]], dtype)
    gamma = np.array([1, 0.5, 2, 1], dtype)
    assert x.shape == shape and gamma.shape == tuple(GOLDEN["gamma"])
    return x, sk, gamma


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
def test_golden_usage_shape_no_bias(dtype):
    x, sk, gamma = _golden_inputs(dtype)
    y, s = oracle.skip_rms(x, sk, gamma, epsilon=0.0)
    # S by hand: row 0 = [3, 4, 0, 0]; row 1 = [-1, 1, -1, 1]
    assert np.array_equal(s, np.array([[3, 4, 0, 0], [-1, 1, -1, 1]], dtype))
    # row 0: mean square (9 + 16) / 4 = 6.25, RMS 2.5 -> [1.2, 0.8, 0, 0]
    # row 1: mean square 1 -> S * gamma = [-1, 0.5, -2, 1]
    want = np.array([[3 / 2.5 * 1, 4 / 2.5 * 0.5, 0, 0], [-1, 0.5, -2, 1]], np.float64)
    assert np.array_equal(y, want.astype(dtype))


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
def test_golden_usage_shape_with_bias(dtype):
    x, sk, gamma = _golden_inputs(dtype)
    bias = np.array([1, -1, 0, 0], dtype)
    y, s = oracle.skip_rms(x, sk, gamma, bias, epsilon=0.0)
    # S by hand: row 0 = [4, 3, 0, 0]; row 1 = [0, 0, -1, 1]
    assert np.array_equal(s, np.array([[4, 3, 0, 0], [0, 0, -1, 1]], dtype))
    # row 0: RMS 2.5 -> [1.6, 0.6, 0, 0]; row 1: mean square 0.5 -> RMS 1/sqrt(2)
    r2 = math.sqrt(2.0)
    want = np.array([[4 / 2.5, 3 / 2.5 * 0.5, 0, 0], [0, 0, -r2 * 2, r2 * 1]], np.float64)
    assert np.array_equal(y, want.astype(dtype))


def test_default_epsilon_is_float32_of_1e12():
    assert np.float64(np.float32(1e-12)) == oracle.SSLN_EPS_DEFAULT


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
@pytest.mark.parametrize("eps", [0.0, 1e-12, 0.5, 3.0])
def test_rms_invariant(dtype, eps):
    """gamma = 1, no bias: each output row has RMS 1/sqrt(1 + eps/ms), where
    ms is the mean square of the row's S."""
    d = synthetic.skip_rms_inputs((37, 203), dtype, seed=11, bias=False)
    gamma = np.ones(203, dtype)
    y, s = oracle.skip_rms(d["input"], d["skip"], gamma, epsilon=eps)
    s64 = s.astype(np.float64)
    ms = (s64 ** 2).mean(axis=1)
    want = 1.0 / np.sqrt(1.0 + eps / ms)
    got = np.sqrt((y.astype(np.float64) ** 2).mean(axis=1))
    rtol = 1e-6 if dtype == np.float32 else 2e-3
    np.testing.assert_allclose(got, want, rtol=rtol)


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
@pytest.mark.parametrize("bias", [False, True])
def test_sum_is_f32_sum_rounded_once(dtype, bias):
    """S = round_T((x + skip) + bias), the adds in binary32 (numpy's IEEE
    binary32 arithmetic and its own float16 cast as the independent check)."""
    d = synthetic.skip_rms_inputs((64, 96), dtype, seed=5, bias=bias, x_std=300.0)
    _, s = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"])
    t = d["input"].astype(np.float32) + d["skip"].astype(np.float32)
    if bias:
        t = t + d["bias"].astype(np.float32)
    assert np.array_equal(s.view(np.uint8), t.astype(dtype).view(np.uint8))


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("eps", [1e-12, 1e-5, 0.25])
def test_matches_torch_rms_norm_float64(dtype, bias, eps):
    d = synthetic.skip_rms_inputs((3, 5, 257), dtype, seed=9, bias=bias)
    y, s = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"], epsilon=eps)
    s64 = torch.from_numpy(s.astype(np.float64))
    g64 = torch.from_numpy(d["gamma"].astype(np.float64))
    ref = torch.nn.functional.rms_norm(s64, (257,), weight=g64, eps=float(np.float32(eps)))
    ref = ref.numpy().astype(dtype)
    # both round a float64 value once; allow one unit in the last place for
    # values that sit on a rounding boundary after different evaluation order
    ulp = np.abs(np.spacing(ref.astype(dtype))).astype(np.float64)
    assert np.all(np.abs(y.astype(np.float64) - ref.astype(np.float64)) <= ulp)


def test_scale_invariance_eps0():
    d = synthetic.skip_rms_inputs((8, 64), np.float32, seed=3, bias=False)
    y1, _ = oracle.skip_rms(d["input"], d["skip"], d["gamma"], epsilon=0.0)
    y2, _ = oracle.skip_rms(d["input"] * np.float32(8), d["skip"] * np.float32(8),
                            d["gamma"], epsilon=0.0)
    assert np.array_equal(y1, y2)


def test_gamma_scales_columns():
    """Output column j is proportional to gamma[j]; a transposed or shifted
    gamma index fails this."""
    d = synthetic.skip_rms_inputs((16, 48), np.float32, seed=4, bias=True)
    ones = np.ones(48, np.float32)
    y1, _ = oracle.skip_rms(d["input"], d["skip"], ones, d["bias"])
    g = np.arange(1, 49, dtype=np.float32)
    yg, _ = oracle.skip_rms(d["input"], d["skip"], g, d["bias"])
    np.testing.assert_allclose(yg, y1 * g[None, :], rtol=2e-7)


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
def test_absent_bias_keeps_negative_zero(dtype):
    """An absent bias is no add: (-0) + (-0) stays -0.  Adding a +0 bias gives
    +0 under round-to-nearest."""
    x = np.array([[-0.0, 1.0]], dtype)
    sk = np.array([[-0.0, 1.0]], dtype)
    g = np.ones(2, dtype)
    _, s = oracle.skip_rms(x, sk, g)
    assert np.signbit(s[0, 0])
    _, s0 = oracle.skip_rms(x, sk, g, np.zeros(2, dtype))
    assert not np.signbit(s0[0, 0])


def test_stats_outputs():
    """mean is 0 for the simplified form; inv_std_var is the inverse RMS
    (README Outputs, mean / inv_std_var)."""
    d = synthetic.skip_rms_inputs((6, 40), np.float32, seed=2, bias=True)
    y, s, mean, inv = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"],
                                      epsilon=0.01, want_stats=True)
    assert mean.shape == (6, 1) and inv.shape == (6, 1)
    assert np.all(mean == 0)
    ms = (s.astype(np.float64) ** 2).mean(axis=1, keepdims=True)
    np.testing.assert_allclose(inv, 1 / np.sqrt(ms + np.float64(np.float32(0.01))), rtol=1e-7)


def test_zero_row_eps0_is_nan():
    """A zero row with epsilon 0 is 0 * inf = NaN by the definition."""
    x = np.zeros((1, 4), np.float32)
    y, _ = oracle.skip_rms(x, x, np.ones(4, np.float32), epsilon=0.0)
    assert np.all(np.isnan(y))
