"""GPU parity: SkipGroupNorm statistics with outliers planted in every group.

The operator's statistics are the population mean and variance of each
(batch item, group) (SkipGroupNorm README, Description).  A single value far
from the rest of its group -- at the group's first element, at its quarter
points, or at random places -- must not cost the binary32 statistics their
accuracy: every route is compared with the oracle at the stated tolerance
(S bit-exact; float32 Y within 1e-5 + 1e-5 |y|; float16 / bfloat16 Y within
2 units in the last place, or 2e-3 where |y| < 1).

Spikes of A = 10, 100 and 1000 standard deviations of the residual sum go
to: each group's first element (positive and negative), each group's first
element and quarter points, and three random elements of each group.
Routes: NCHW one CTA per instance (10,240-element groups), clusters per
instance (10,240- and 40,960-element groups) and the forced two-phase route;
NHWC the automatic (cooperative) route and the forced routes 3, 4, 5 and 6.
"""
import numpy as np
import pytest
import torch

import oracle
import residual_add_normalization_gb300 as b2
from residual_add_normalization_gb300 import synthetic
from helpers import assert_bitexact, assert_y_close, to_dev, to_host, values

pytestmark = pytest.mark.gpu

BF16 = synthetic.BFLOAT16
PATTERNS = [("first", 10.0), ("first", 100.0), ("first", 1000.0), ("first", -1000.0),
            ("quarters", 1000.0), ("random", 1000.0)]


@pytest.fixture(autouse=True)
def _reset_force():
    yield
    b2.library().b200norm_testing_force(0, 0)


def group_offsets(shape, groups, cl, n, g, j):
    """Flat offsets of elements j (an array) of group instance (n, g)."""
    if cl:
        N, H, W, C = shape
        cpg = C // groups
        return (n * H * W + j // cpg) * C + g * cpg + j % cpg
    N, C, H, W = shape
    cpg = C // groups
    return (n * C + g * cpg) * H * W + j


def plant(d, shape, groups, cl, pattern, A, seed):
    """Put A standard deviations of S into X at the pattern's elements."""
    N = shape[0]
    C = shape[3] if cl else shape[1]
    HW = shape[1] * shape[2] if cl else shape[2] * shape[3]
    L = (C // groups) * HW
    x = d["x"].reshape(-1).copy()
    sig = float(np.std(values(x))) + 1.0  # std of X plus the skip's unit std, roughly
    rng = np.random.default_rng(seed)
    for n in range(N):
        for g in range(groups):
            if pattern == "first":
                j = np.array([0])
            elif pattern == "quarters":
                j = np.array([0, L // 4, L // 2, 3 * L // 4])
            else:
                j = rng.choice(L, size=min(3, L), replace=False)
            off = group_offsets(shape, groups, cl, n, g, j)
            v = np.full(off.shape, A * sig, dtype=np.float32)
            x[off] = synthetic.to_bfloat16(v) if synthetic.is_bf16(x.dtype) else v.astype(x.dtype)
    return dict(d, x=x.reshape(d["x"].shape))


def run_check(d, groups, act, cl):
    y, s = b2.skip_group(to_dev(d["x"]), to_dev(d["skip"]), to_dev(d["gamma"]),
                         to_dev(d["beta"]), to_dev(d["bias"]), groups=groups, activation=act,
                         channels_last=cl, want_sum=True)
    torch.cuda.synchronize()
    ry, rs = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"],
                               groups=groups, activation=act, channels_last=cl)
    assert_bitexact(to_host(s), rs)
    assert_y_close(to_host(y), ry)


TYPES = [(np.float32, np.float16), (np.float16, np.float32)]
NCHW = [((16, 1280, 16, 16), 32, 0),  # one CTA per 10,240-element instance
        ((2, 1280, 16, 16), 32, 0),   # 64 instances: a cluster of CTAs each
        ((1, 320, 64, 64), 32, 0),    # a cluster per 40,960-element instance
        ((2, 64, 16, 16), 8, 3)]      # forced two-phase


@pytest.mark.parametrize("pattern,A", PATTERNS)
@pytest.mark.parametrize("dtype,mdtype", TYPES)
@pytest.mark.parametrize("shape,groups,force", NCHW)
def test_nchw_outliers(shape, groups, force, dtype, mdtype, pattern, A):
    d = synthetic.skip_group_inputs(shape, dtype, mdtype, seed=21, channels_last=0,
                                    skip="full", bias=False, x_std=2.0)
    d = plant(d, shape, groups, 0, pattern, A, seed=5)
    assert b2.library().b200norm_testing_force(0, force) == 0
    run_check(d, groups, 0, 0)


@pytest.mark.parametrize("pattern,A", PATTERNS)
@pytest.mark.parametrize("dtype,mdtype", TYPES)
@pytest.mark.parametrize("route", [0, 3, 4, 5, 6])
def test_nhwc_outliers(route, dtype, mdtype, pattern, A):
    shape, groups = (2, 64, 64, 320), 32
    d = synthetic.skip_group_inputs(shape, dtype, mdtype, seed=22, channels_last=1, skip="nc",
                                    bias=True)
    d = plant(d, shape, groups, 1, pattern, A, seed=6)
    assert b2.library().b200norm_testing_force(0, route) == 0
    run_check(d, groups, 1, 1)


@pytest.mark.parametrize("route", [0, 3, 4, 5, 6])
@pytest.mark.parametrize("cl", [0, 1])
def test_bf16_outliers(cl, route):
    if not cl and route in (4, 5, 6):
        pytest.skip("NHWC-only route")
    shape = (2, 64, 64, 320) if cl else (2, 1280, 16, 16)
    d = synthetic.skip_group_inputs(shape, BF16, np.float32, seed=23, channels_last=cl,
                                    skip="nc" if cl else "full", bias=cl == 1)
    d = plant(d, shape, 32, cl, "first", 1000.0, seed=7)
    assert b2.library().b200norm_testing_force(0, route) == 0
    run_check(d, 32, cl, cl)


def test_outlier_routes_are_the_intended_ones():
    """The automatic plans behind the cases above: one CTA and clusters per
    NCHW instance, the cooperative grid for NHWC."""
    import ctypes
    lib = b2.library()
    out = (ctypes.c_int64 * 8)()
    for dt, mt in ((0, 1), (1, 0)):
        assert lib.b200norm_testing_plan_group(16, 1280, 16, 16, 32, dt, mt, 0, 1, out) == 0
        assert out[0] == 1 and out[4] == 1
        for N, C, H in ((2, 1280, 16), (1, 320, 64)):
            assert lib.b200norm_testing_plan_group(N, C, H, H, 32, dt, mt, 0, 1, out) == 0
            assert out[0] == 1 and out[4] > 1
    assert lib.b200norm_testing_plan_group(2, 320, 64, 64, 32, 1, 0, 1, 1, out) == 0
    assert out[0] == 2
