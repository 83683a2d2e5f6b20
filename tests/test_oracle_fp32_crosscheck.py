"""The oracle's binary64 statistics against a plain binary32 restatement.

A second, deliberately naive implementation of each operator (numpy float32,
whole-array formulas, written here from the operator pages' definitions, not
from the oracle) must agree with the oracle's float32 outputs within
1e-5 absolute + 1e-5 relative on random inputs.  Its arithmetic is coarser
than the oracle's, so this catches indexing and layout mistakes (a wrong
channel for a group, a transposed skip, a statistic over the wrong axis), not
rounding ones.  With T = float32 the naive residual sum, (x + skip) + bias in
binary32, is the oracle's S bit for bit, which the tests check as well.

Operators: SkipSimplifiedLayerNormalization README, Description;
GatedRMSNorm README, Description; SkipGroupNorm README, Description.
"""
import numpy as np
import pytest

import oracle
from residual_add_normalization_gb300 import synthetic

F32 = np.float32


def close(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    bad = np.abs(got - ref) > 1e-5 + 1e-5 * np.abs(ref)
    assert not bad.any(), (int(bad.sum()), float(np.abs(got - ref).max()))


def silu32(z):
    return z / (F32(1) + np.exp(-z))


@pytest.mark.parametrize("shape,bias", [((64, 768), True), ((3, 5, 96), False), ((7, 1000), True)])
def test_skip_rms_naive_fp32(shape, bias):
    d = synthetic.skip_rms_inputs(shape, F32, seed=sum(shape), bias=bias)
    eps = F32(1e-6)
    s = d["input"] + d["skip"]
    if bias:
        s = s + d["bias"]
    ms = np.mean(s * s, axis=-1, keepdims=True, dtype=F32)
    y = s / np.sqrt(ms + eps) * d["gamma"]
    ry, rs = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"], epsilon=float(eps))
    assert np.array_equal(rs, s.astype(F32))
    close(y, ry)


@pytest.mark.parametrize("shape,C", [((2, 64, 256), 128), ((4096,), 64), ((3, 2048), 2048)])
def test_gated_rms_naive_fp32(shape, C):
    d = synthetic.gated_rms_inputs(shape, C, F32, seed=C + len(shape))
    eps = F32(1e-5)
    x = d["x"].reshape(-1, C)
    g = d["gate"].reshape(-1, C)
    ms = np.mean(x * x, axis=1, keepdims=True, dtype=F32)
    y = (x / np.sqrt(ms + eps) * d["scale"] * silu32(g)).reshape(shape)
    close(y, oracle.gated_rms(d["x"], d["gate"], d["scale"], epsilon=float(eps)))


CASES = [((2, 64, 8, 8), 8, 0, "full", True, 1), ((2, 6, 5, 48), 4, 1, "nc", True, 0),
         ((3, 96, 4, 4), 32, 0, "nc", False, 1), ((1, 7, 9, 64), 16, 1, "full", False, 1),
         ((2, 1, 1, 64), 8, 1, "n11c", True, 0)]


@pytest.mark.parametrize("shape,groups,cl,skip,bias,act", CASES)
def test_skip_group_naive_fp32(shape, groups, cl, skip, bias, act):
    d = synthetic.skip_group_inputs(shape, F32, F32, seed=sum(shape) + groups, channels_last=cl,
                                    skip=skip, bias=bias, x_std=1.5)
    x = d["x"]
    # everything in NCHW for the naive form
    xc = np.transpose(x, (0, 3, 1, 2)) if cl else x
    N, C, H, W = xc.shape
    sk = d["skip"]
    if sk.size == N * C:  # (N, C) or (N, 1, 1, C): one value per batch item and channel
        skc = sk.reshape(N, C, 1, 1)
    else:
        skc = np.transpose(sk, (0, 3, 1, 2)) if cl else sk
    s = xc + skc
    if bias:
        s = s + d["bias"].reshape(1, C, 1, 1)
    sg = s.reshape(N, groups, -1)
    mean = np.mean(sg, axis=2, keepdims=True, dtype=F32)
    var = np.mean((sg - mean) ** 2, axis=2, keepdims=True, dtype=F32)
    z = ((sg - mean) / np.sqrt(var + F32(1e-5))).reshape(N, C, H, W)
    z = z * d["gamma"].reshape(1, C, 1, 1) + d["beta"].reshape(1, C, 1, 1)
    if act:
        z = silu32(z)
    y = np.transpose(z, (0, 2, 3, 1)) if cl else z
    ry, rs = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"], groups=groups,
                               activation=act, channels_last=cl)
    s_back = np.transpose(s, (0, 2, 3, 1)) if cl else s
    assert np.array_equal(rs, s_back.astype(F32))
    close(y, ry)
