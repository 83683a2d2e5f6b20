"""Pins for the oracle's GatedRMSNorm.

Operator (com.microsoft.GatedRMSNorm README, Description, Inputs):
Y = X * rsqrt(mean(X^2) + epsilon) * scale * SiLU(gate), the mean over each
contiguous span of C = numel(scale) elements.  Pins: the usage example's
C = 1 case in closed form, a C = 4 hand case, torch's float64 rms_norm and
silu on the (rows, C) reshape, and the scale-spelling equivalence.
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
                                     "usage_examples.json")))["gated_rms_norm"]


def silu(g):
    return g / (1.0 + math.exp(-g))


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
def test_golden_usage_shape_c1(dtype):
    """scale has one element, so C = 1 and every element is its own span:
    y = x / sqrt(x^2 + eps) * scale * silu(g).  eps = 16 keeps it visible."""
    shape = tuple(GOLDEN["X"])
    assert shape == (3, 4) and tuple(GOLDEN["scale"]) == (1,)
    x = np.array([[3, -3, 0, 4], [1, 2, -4, 3], [3, 3, 3, 3]], np.float64)
    l3 = math.log(3.0)
    g = np.array([[l3, l3, 5, 0], [1, -1, 2, -l3], [0, 0.5, -0.5, 7]], np.float64)
    xt, gt = x.astype(dtype), g.astype(dtype)
    scale = np.array([2.0], dtype)
    y = oracle.gated_rms(xt, gt, scale, epsilon=16.0)
    # hand values of x / sqrt(x^2 + 16): 3 -> 3/5, 4 -> 1/sqrt(2), 1 -> 1/sqrt(17),
    # 2 -> 1/sqrt(5), 0 -> 0.  silu(ln 3) = 0.75 ln 3, silu(0) = 0.
    norm = {3.0: 0.6, -3.0: -0.6, 0.0: 0.0, 4.0: 1 / math.sqrt(2), -4.0: -1 / math.sqrt(2),
            1.0: 1 / math.sqrt(17), 2.0: 1 / math.sqrt(5)}
    want = np.empty((3, 4))
    for i in range(3):
        for j in range(4):
            want[i, j] = norm[x[i, j]] * 2.0 * silu(float(gt[i, j]))
    assert want[0, 0] == pytest.approx(0.6 * 2 * 0.75 * l3, rel=1e-3)  # 0.9 ln 3
    got = y.astype(np.float64)
    ref = want.astype(dtype).astype(np.float64)
    ulp = np.abs(np.spacing(want.astype(dtype))).astype(np.float64)
    assert np.all(np.abs(got - ref) <= ulp)
    assert y[0, 3] == 0 and y[2, 0] == 0 and y[0, 2] == 0  # silu(0) = 0 and x = 0


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
def test_hand_case_c4(dtype):
    """C = 4, rows of +-1 have mean square 1; with eps = 0 the output is
    x * scale[j] * silu(g)."""
    x = np.array([[1, -1, 1, -1], [2, 2, -2, 2], [0.5, -0.5, 0.5, 0.5]], dtype)
    l3 = math.log(3.0)
    g = np.array([[l3, 0, l3, -l3], [l3, l3, l3, l3], [1, 1, 1, 1]], np.float64)
    scale = np.array([1, 2, 0.5, 1], dtype)
    y = oracle.gated_rms(x, g.astype(dtype), scale, epsilon=0.0)
    gs = g.astype(dtype).astype(np.float64)
    unit = x.astype(np.float64) / np.array([[1], [2], [0.5]])
    want = np.vectorize(silu)(gs) * unit * scale.astype(np.float64)[None, :]
    ulp = np.abs(np.spacing(want.astype(dtype))).astype(np.float64)
    assert np.all(np.abs(y.astype(np.float64) - want.astype(dtype).astype(np.float64)) <= ulp)


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
@pytest.mark.parametrize("C,shape", [(128, (2, 7, 256)), (24, (5, 72)), (1, (9,)),
                                     (96, (3, 96)), (4096, (2, 4096))])
@pytest.mark.parametrize("eps", [1e-5, 1e-6, 0.3])
def test_matches_torch_float64(dtype, C, shape, eps):
    d = synthetic.gated_rms_inputs(shape, C, dtype, seed=C + len(shape))
    y = oracle.gated_rms(d["x"], d["gate"], d["scale"], epsilon=eps)
    x64 = torch.from_numpy(d["x"].astype(np.float64)).reshape(-1, C)
    g64 = torch.from_numpy(d["gate"].astype(np.float64)).reshape(-1, C)
    s64 = torch.from_numpy(d["scale"].astype(np.float64))
    ref = torch.nn.functional.rms_norm(x64, (C,), weight=s64, eps=float(np.float32(eps)))
    ref = (ref * torch.nn.functional.silu(g64)).reshape(shape).numpy()
    refT = ref.astype(dtype)
    ulp = np.abs(np.spacing(refT)).astype(np.float64)
    assert np.all(np.abs(y.astype(np.float64) - refT.astype(np.float64)) <= ulp)


def test_scale_spellings_equivalent():
    """(C), (1, C) and (C, 1) spellings of scale carry the same span
    (README Inputs, scale)."""
    d = synthetic.gated_rms_inputs((4, 64), 16, np.float16, seed=1)
    y0 = oracle.gated_rms(d["x"], d["gate"], d["scale"])
    y1 = oracle.gated_rms(d["x"], d["gate"], d["scale"].reshape(1, 16))
    y2 = oracle.gated_rms(d["x"], d["gate"], d["scale"].reshape(16, 1))
    assert np.array_equal(y0.view(np.uint16), y1.view(np.uint16))
    assert np.array_equal(y0.view(np.uint16), y2.view(np.uint16))


def test_span_not_dividing_numel_rejected():
    with pytest.raises(ValueError):
        oracle.gated_rms(np.ones(10, np.float32), np.ones(10, np.float32),
                         np.ones(3, np.float32))
