"""Pins for the oracle's SkipGroupNorm.

Operator (com.microsoft.SkipGroupNorm README, Description, Inputs, Outputs,
Attributes): S = X + skip + bias rounded to T; Y = gamma * (S - mean) /
sqrt(var + epsilon) + beta, then SiLU if activation = 1; statistics per batch
item over the C/groups channels of a group and all spatial positions; NHWC
when channels_last != 0, else NCHW; skip full-shape or per-(n, c).

Pins: a closed-form case on the usage example's shape, the mean-0 /
var/(var+eps) invariant, torch's float64 group_norm / layer_norm, layout
permutation, broadcast-vs-materialised skip, the (N,1,1,C) at H = W = 1 rule,
Y independent of whether S is requested, and groups = C at H = W = 1.
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
                                     "usage_examples.json")))["skip_group_norm"]


def _silu(z):
    return z / (1.0 + np.exp(-z))


def _golden_case(dtype, mdtype):
    """X (2,3,2,8) NHWC with a +-1 checkerboard: every group of 4 channels x 6
    pixels has mean 0 and population variance 1.  skip (2,8) is constant over
    each group's channels, so it shifts the group mean and leaves
    S - mean = X.  With eps = 0: Y = gamma[c] * X + beta[c]."""
    N, H, W, C = GOLDEN["X"]
    assert GOLDEN["skip"] == [N, C] and GOLDEN["attrs"]["groups"] == 2
    h, w, c = np.meshgrid(np.arange(H), np.arange(W), np.arange(C), indexing="ij")
    pat = np.where((h * W + w + c) % 2 == 0, 1.0, -1.0)
    x = np.stack([pat, pat]).astype(dtype)
    skip = np.array([[1, 1, 1, 1, 2, 2, 2, 2], [-0.5] * 8], dtype)
    gamma = np.array([1, 2, 0.5, 1, 1, 1, -1, 3], mdtype)
    beta = np.array([0, 0.25, 0, -1, 0.5, 0, 0, 0], mdtype)
    return x, skip, gamma, beta


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
@pytest.mark.parametrize("mdtype", [np.float32, np.float16])
@pytest.mark.parametrize("act", [0, 1])
def test_golden_usage_shape(dtype, mdtype, act):
    x, skip, gamma, beta = _golden_case(dtype, mdtype)
    y, s = oracle.skip_group(x, skip, gamma, beta, groups=2, activation=act, epsilon=0.0)
    want_s = x.astype(np.float64) + skip.astype(np.float64)[:, None, None, :]
    assert np.array_equal(s, want_s.astype(dtype))
    z = gamma.astype(np.float64) * x.astype(np.float64) + beta.astype(np.float64)
    if act:
        z = _silu(z)
    zt = z.astype(dtype)
    ulp = np.abs(np.spacing(zt)).astype(np.float64)
    assert np.all(np.abs(y.astype(np.float64) - zt.astype(np.float64)) <= ulp)
    if not act:
        assert np.array_equal(y, zt)  # exact when no transcendental is involved


@pytest.mark.parametrize("cl", [1, 0])
@pytest.mark.parametrize("eps", [1e-5, 0.5])
def test_mean0_var_invariant(cl, eps):
    """gamma = 1, beta = 0, no activation: each group of Y has mean 0 and
    population variance var/(var + eps), var the group's variance of S."""
    N, C, H, W, G = 3, 12, 5, 7, 4
    shape = (N, H, W, C) if cl else (N, C, H, W)
    d = synthetic.skip_group_inputs(shape, np.float32, np.float32, seed=21, channels_last=cl,
                                    skip="full", bias=True, x_mean=3.0)
    ones, zeros = np.ones(C, np.float32), np.zeros(C, np.float32)
    y, s = oracle.skip_group(d["x"], d["skip"], ones, zeros, d["bias"], groups=G,
                             activation=0, epsilon=eps, channels_last=cl)
    if cl:
        s, y = s.transpose(0, 3, 1, 2), y.transpose(0, 3, 1, 2)
    sg = s.astype(np.float64).reshape(N, G, -1)
    yg = y.astype(np.float64).reshape(N, G, -1)
    var = sg.var(axis=2)
    np.testing.assert_allclose(yg.mean(axis=2), 0.0, atol=2e-6)
    np.testing.assert_allclose(yg.var(axis=2), var / (var + np.float64(np.float32(eps))),
                               rtol=2e-6)


@pytest.mark.parametrize("dtype,mdtype", [(np.float32, np.float16), (np.float16, np.float32),
                                          (np.float16, np.float16)])
@pytest.mark.parametrize("cl", [1, 0])
@pytest.mark.parametrize("act", [0, 1])
@pytest.mark.parametrize("G", [1, 3, 12])
def test_matches_torch_group_norm_float64(dtype, mdtype, cl, act, G):
    N, C, H, W = 2, 12, 4, 5
    shape = (N, H, W, C) if cl else (N, C, H, W)
    d = synthetic.skip_group_inputs(shape, dtype, mdtype, seed=G + 10 * cl + act,
                                    channels_last=cl, skip="nc", bias=True)
    y, s = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"], groups=G,
                             activation=act, epsilon=1e-5, channels_last=cl)
    s_nchw = s.transpose(0, 3, 1, 2) if cl else s
    ref = torch.nn.functional.group_norm(
        torch.from_numpy(s_nchw.astype(np.float64)), G,
        torch.from_numpy(d["gamma"].astype(np.float64)),
        torch.from_numpy(d["beta"].astype(np.float64)), eps=float(np.float32(1e-5)))
    if act:
        ref = torch.nn.functional.silu(ref)
    ref = ref.numpy()
    if cl:
        ref = ref.transpose(0, 2, 3, 1)
    refT = ref.astype(dtype)
    ulp = np.abs(np.spacing(refT)).astype(np.float64)
    assert np.all(np.abs(y.astype(np.float64) - refT.astype(np.float64)) <= ulp)


def test_groups1_is_layer_norm():
    N, C, H, W = 2, 6, 3, 4
    d = synthetic.skip_group_inputs((N, C, H, W), np.float32, np.float32, seed=5,
                                    channels_last=0, skip="full", bias=False)
    y, s = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], groups=1,
                             activation=0, epsilon=1e-5, channels_last=0)
    ga = np.broadcast_to(d["gamma"][:, None, None], (C, H, W)).astype(np.float64)
    be = np.broadcast_to(d["beta"][:, None, None], (C, H, W)).astype(np.float64)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(s.astype(np.float64)), (C, H, W),
                                         torch.from_numpy(ga.copy()), torch.from_numpy(be.copy()),
                                         eps=float(np.float32(1e-5))).numpy().astype(np.float32)
    ulp = np.abs(np.spacing(ref)).astype(np.float64)
    assert np.all(np.abs(y.astype(np.float64) - ref.astype(np.float64)) <= ulp)


@pytest.mark.parametrize("skip", ["full", "nc"])
def test_nhwc_is_permuted_nchw(skip):
    N, C, H, W = 2, 10, 3, 5
    d = synthetic.skip_group_inputs((N, C, H, W), np.float16, np.float32, seed=8,
                                    channels_last=0, skip=skip, bias=True)
    y0, s0 = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"], groups=5,
                               activation=1, channels_last=0)
    xl = d["x"].transpose(0, 2, 3, 1)
    sl = d["skip"].transpose(0, 2, 3, 1) if skip == "full" else d["skip"]
    y1, s1 = oracle.skip_group(xl, sl, d["gamma"], d["beta"], d["bias"], groups=5,
                               activation=1, channels_last=1)
    assert np.array_equal(y1.view(np.uint16), y0.transpose(0, 2, 3, 1).view(np.uint16))
    assert np.array_equal(s1.view(np.uint16), s0.transpose(0, 2, 3, 1).view(np.uint16))


@pytest.mark.parametrize("cl", [1, 0])
def test_broadcast_skip_equals_materialised(cl):
    N, C, H, W = 2, 16, 3, 3
    shape = (N, H, W, C) if cl else (N, C, H, W)
    d = synthetic.skip_group_inputs(shape, np.float16, np.float16, seed=2, channels_last=cl,
                                    skip="nc", bias=True)
    full = (np.broadcast_to(d["skip"][:, None, None, :], shape) if cl
            else np.broadcast_to(d["skip"][:, :, None, None], shape)).copy()
    a = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"], groups=4,
                          activation=0, channels_last=cl)
    b = oracle.skip_group(d["x"], full, d["gamma"], d["beta"], d["bias"], groups=4,
                          activation=0, channels_last=cl)
    n11c = oracle.skip_group(d["x"], d["skip"].reshape(N, 1, 1, C), d["gamma"], d["beta"],
                             d["bias"], groups=4, activation=0, channels_last=cl)
    for u, v in zip(a, b):
        assert np.array_equal(u.view(np.uint16), v.view(np.uint16))
    for u, v in zip(a, n11c):
        assert np.array_equal(u.view(np.uint16), v.view(np.uint16))


def test_n11c_at_hw1_takes_full_route():
    """(N,1,1,C) skip at H = W = 1 is an exact match for NHWC X (README Inputs,
    skip) and gives the same values as the (N, C) broadcast."""
    N, C = 3, 8
    d = synthetic.skip_group_inputs((N, 1, 1, C), np.float32, np.float32, seed=4,
                                    channels_last=1, skip="n11c", bias=True)
    assert not oracle._skip_is_broadcast((N, 1, 1, C), (N, 1, 1, C), 1)
    a = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"], groups=2,
                          activation=1)
    b = oracle.skip_group(d["x"], d["skip"].reshape(N, C), d["gamma"], d["beta"], d["bias"],
                          groups=2, activation=1)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_y_independent_of_s_request():
    d = synthetic.skip_group_inputs((2, 4, 4, 32), np.float16, np.float32, seed=6,
                                    channels_last=1, skip="full", bias=True)
    y1, s = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"], groups=8,
                              activation=1, want_sum=True)
    y2, none = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"], groups=8,
                                 activation=1, want_sum=False)
    assert none is None and s is not None
    assert np.array_equal(y1.view(np.uint16), y2.view(np.uint16))


@pytest.mark.parametrize("act", [0, 1])
def test_groups_eq_C_hw1_gives_beta(act):
    """One element per group: S - mean = 0, so Y = beta (then SiLU)."""
    N, C = 4, 6
    d = synthetic.skip_group_inputs((N, 1, 1, C), np.float32, np.float32, seed=1,
                                    channels_last=1, skip="full", bias=True)
    y, _ = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"], groups=C,
                             activation=act)
    want = d["beta"].astype(np.float64)
    if act:
        want = _silu(want)
    assert np.array_equal(y, np.broadcast_to(want.astype(np.float32), y.shape))


def test_invalid_attributes_rejected():
    d = synthetic.skip_group_inputs((1, 2, 2, 6), np.float32, np.float32, seed=1)
    with pytest.raises(ValueError):
        oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], groups=4, activation=0)
    with pytest.raises(ValueError):
        oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], groups=2, activation=2)
    with pytest.raises(ValueError):
        oracle.skip_group(d["x"], d["skip"][:, :1], d["gamma"], d["beta"], groups=2,
                          activation=0)
