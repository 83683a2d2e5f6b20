"""GPU parity: SkipGroupNorm kernels against the CPU oracle on the same seeded
inputs, through the C ABI (via the binding).

Covers the six routes (NCHW: CTA / cluster per group instance; NHWC: a
cooperative grid with one bounded grid barrier holding its slabs in
registers or in shared memory, one cooperative grid or a statistics kernel
and an apply kernel through L2; two-phase for anything else),
both layouts, both T and both M, full / (N, C) / (N, 1, 1, C) skip, bias and S
on and off, SiLU on and off, vector and scalar paths, and ragged slabs.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import residual_add_normalization_gb300 as b2
from residual_add_normalization_gb300 import synthetic
from helpers import assert_bitexact, assert_y_close, to_dev, to_host

pytestmark = pytest.mark.gpu

F32, F16 = 0, 1
_CODE = {np.float32: F32, np.float16: F16}


@pytest.fixture(autouse=True)
def _reset_force():
    yield
    b2.library().b200norm_testing_force(0, 0)


def plan(shape, groups, dtype, mdtype, cl):
    if cl:
        N, H, W, C = shape
    else:
        N, C, H, W = shape
    out = (ctypes.c_int64 * 8)()
    st = b2.library().b200norm_testing_plan_group(N, C, H, W, groups, _CODE[dtype], _CODE[mdtype],
                                                  cl, 1, out)
    assert st == 0
    return dict(zip(("route", "ve", "nv", "block", "csize", "grid", "B", "ppc"), out))


def run(d, groups, act, cl, eps=1e-5, want_sum=True):
    y, s = b2.skip_group(to_dev(d["x"]), to_dev(d["skip"]), to_dev(d["gamma"]),
                         to_dev(d["beta"]), to_dev(d["bias"]), groups=groups, activation=act,
                         epsilon=eps, channels_last=cl, want_sum=want_sum)
    torch.cuda.synchronize()
    return to_host(y), to_host(s)


def check(d, groups, act, cl, eps=1e-5, want_sum=True):
    y, s = run(d, groups, act, cl, eps, want_sum)
    ry, rs = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"],
                               groups=groups, activation=act, epsilon=eps, channels_last=cl)
    if want_sum:
        assert_bitexact(s, rs)
    else:
        assert s is None
    assert_y_close(y, ry)


# (logical N, C, H, W, groups)
NCHW_CASES = [
    (2, 8, 3, 2, 2),        # usage-example sizes, scalar path (H*W = 6)
    (2, 12, 5, 7, 4),       # odd H*W: scalar path
    (3, 64, 8, 8, 8),       # small instances
    (2, 1280, 16, 16, 32),  # 10,240-element instances (the wide-group workload's)
    (1, 320, 64, 64, 32),   # 40,960-element instances: clusters
    (1, 64, 128, 128, 1),   # one 1M-element instance: two-phase
    (4, 6, 1, 1, 6),        # one element per group
    (6, 256, 8, 8, 32),     # 192 instances, more than one per SM
    (5, 96, 12, 12, 32),    # 160 instances of 432 elements
]


BF16 = synthetic.BFLOAT16
TYPE_PAIRS = [(np.float32, np.float16), (np.float16, np.float32), (np.float16, np.float16),
              (np.float32, np.float32), (BF16, np.float32), (BF16, BF16)]


@pytest.mark.parametrize("dtype,mdtype", TYPE_PAIRS)
@pytest.mark.parametrize("case", NCHW_CASES)
def test_nchw_matches_oracle(dtype, mdtype, case):
    N, C, H, W, G = case
    for skip, bias, act, want_sum in (("full", False, 0, False), ("nc", True, 1, True)):
        d = synthetic.skip_group_inputs((N, C, H, W), dtype, mdtype, seed=N * C + H,
                                        channels_last=0, skip=skip, bias=bias, x_std=2.0)
        check(d, G, act, 0, want_sum=want_sum)


# (logical N, H, W, C, groups)
NHWC_CASES = [
    (2, 3, 2, 8, 2),        # the usage example's shape
    (2, 64, 64, 320, 32),   # the NHWC workload's shape
    (2, 8, 8, 64, 4),
    (3, 5, 7, 12, 3),       # C % 8 != 0: scalar path
    (1, 33, 17, 40, 8),     # ragged last slab
    (2, 16, 16, 4104, 8),   # C / 8 = 513 vectors per pixel: two-phase
    (600, 2, 2, 16, 4),     # many batch items
    (4, 1, 1, 6, 6),
    (1, 256, 256, 64, 1),   # one 4M-element group
    (2, 64, 64, 96, 24),    # cpg 4: 8-channel vectors span two groups
    (64, 8, 8, 64, 8),      # 64 batch items: the cooperative route
    (1, 128, 128, 128, 32), # one item over every SM, 32 groups
    (64, 32, 32, 320, 32),  # 64 items, too many pixels for registers: one grid through L2
]


@pytest.mark.parametrize("dtype,mdtype", TYPE_PAIRS)
@pytest.mark.parametrize("case", NHWC_CASES)
def test_nhwc_matches_oracle(dtype, mdtype, case):
    N, H, W, C, G = case
    for skip, bias, act, want_sum in (("nc", True, 1, True), ("full", False, 0, False),
                                      ("n11c", True, 0, True)):
        d = synthetic.skip_group_inputs((N, H, W, C), dtype, mdtype, seed=N + H * W + C,
                                        channels_last=1, skip=skip, bias=bias)
        check(d, G, act, 1, want_sum=want_sum)


@pytest.mark.parametrize("cl", [0, 1])
@pytest.mark.parametrize("dtype", [np.float32, np.float16, BF16])
def test_forced_two_phase(cl, dtype):
    assert b2.library().b200norm_testing_force(0, 3) == 0
    shape = (2, 16, 16, 64) if cl else (2, 64, 16, 16)
    d = synthetic.skip_group_inputs(shape, dtype, np.float32, seed=7, channels_last=cl,
                                    skip="nc", bias=True)
    check(d, 8, 1, cl)


@pytest.mark.parametrize("route", [2, 4, 5, 6])
@pytest.mark.parametrize("dtype,mdtype", TYPE_PAIRS)
@pytest.mark.parametrize("case", NHWC_CASES)
def test_nhwc_forced_routes(route, dtype, mdtype, case):
    """The NHWC routes 2, 4, 5 and 6 on every NHWC case each can take (route
    2 holds a resident grid's pixels in registers, route 6 in shared memory;
    routes 4 and 5 re-read tensors that stay in L2, in two launches or in one
    cooperative grid)."""
    N, H, W, C, G = case
    assert b2.library().b200norm_testing_force(0, route) == 0
    for skip, bias, act, want_sum in (("nc", True, 1, True), ("full", False, 0, False)):
        d = synthetic.skip_group_inputs((N, H, W, C), dtype, mdtype, seed=N + H + W + C + route,
                                        channels_last=1, skip=skip, bias=bias, x_std=1.5)
        try:
            check(d, G, act, 1, want_sum=want_sum)
        except b2.B200NormError as e:
            if "forced route" in str(e):
                pytest.skip(f"route {route} cannot take {case}: {e}")
            raise


def test_route_coverage():
    routes = set()
    for N, C, H, W, G in NCHW_CASES:
        p = plan((N, C, H, W), G, np.float16, np.float32, 0)
        routes.add((p["route"], p["csize"] > 1))
    for N, H, W, C, G in NHWC_CASES:
        routes.add((plan((N, H, W, C), G, np.float16, np.float32, 1)["route"], False))
    assert {1, 2, 3} <= {r for r, _ in routes} <= {1, 2, 3, 5, 6}
    assert (1, True) in routes, "no cluster-per-instance case"
    # the cooperative route while its grid can hold the pixels in registers,
    # else the cooperative route with the slabs in shared memory, else one
    # cooperative grid through L2.  (The plan query assumes a full-shape skip,
    # whose slab in shared memory doubles that of X.)
    # small NCHW batches: instances split over clusters while the grid stays
    # within 2 x SMs (measured faster), not beyond
    for shape, cs in (((2, 1280, 16, 16), 4), ((1, 1280, 16, 16), 4), ((4, 1280, 16, 16), 2),
                      ((2, 640, 32, 32), 4)):
        p = plan(shape, 32, np.float16, np.float32, 0)
        assert (p["route"], p["csize"]) == (1, cs), (shape, p)
    assert plan((2, 64, 64, 320), 32, np.float16, np.float32, 1)["route"] == 2
    assert plan((64, 8, 8, 64), 8, np.float16, np.float32, 1)["route"] == 2
    assert plan((4, 64, 64, 320), 32, np.float16, np.float32, 1)["route"] == 6
    assert plan((16, 32, 32, 320), 32, np.float16, np.float32, 1)["route"] == 6
    assert plan((2, 128, 128, 320), 32, np.float16, np.float32, 1)["route"] == 5
    assert plan((64, 24, 24, 320), 32, np.float16, np.float32, 1)["route"] == 5


def test_n11c_at_hw1_equals_nc_route():
    d = synthetic.skip_group_inputs((3, 1, 1, 16), np.float16, np.float32, seed=4,
                                    channels_last=1, skip="n11c", bias=True)
    y1, s1 = run(d, 4, 1, 1)
    d2 = dict(d, skip=d["skip"].reshape(3, 16))
    y2, s2 = run(d2, 4, 1, 1)
    assert_bitexact(y1, y2, "Y")
    assert_bitexact(s1, s2)


def test_y_independent_of_s_request():
    d = synthetic.skip_group_inputs((2, 16, 16, 64), np.float16, np.float32, seed=9,
                                    channels_last=1, skip="full", bias=True)
    y1, _ = run(d, 8, 1, 1, want_sum=True)
    y2, _ = run(d, 8, 1, 1, want_sum=False)
    assert_bitexact(y1, y2, "Y")


def test_large_mean_small_variance():
    """Groups whose mean is far from zero against their spread: carrying the
    mean as an exact data value plus a small offset keeps float32 Y inside
    1e-5."""
    for cl, shape in ((0, (2, 64, 16, 16)), (1, (2, 16, 16, 64))):
        d = synthetic.skip_group_inputs(shape, np.float32, np.float32, seed=12,
                                        channels_last=cl, skip="full", bias=False,
                                        x_mean=1000.0, x_std=0.5)
        check(d, 8, 0, cl)
        assert b2.library().b200norm_testing_force(0, 3) == 0
        check(d, 8, 0, cl)
        assert b2.library().b200norm_testing_force(0, 0) == 0


def test_empty_batch():
    x = torch.empty((0, 4, 4, 8), dtype=torch.float16, device="cuda")
    g = torch.ones(8, dtype=torch.float32, device="cuda")
    y, s = b2.skip_group(x, torch.empty((0, 8), dtype=torch.float16, device="cuda"), g, g,
                         groups=2, activation=0)
    assert y.shape == x.shape


def test_one_workspace_serves_every_route_in_turn():
    """One explicit workspace, calls of different shapes and routes in turn
    (the L2 route's per-item counters and the cooperative route's barrier live
    in its control block; partial slots are overwritten by every route)."""
    calls = [((2, 64, 64, 320), 1, 32, None), ((1, 128, 128, 128), 1, 32, None),
             ((5, 16, 16, 64), 1, 8, 4), ((2, 64, 16, 16), 0, 8, None),
             ((1, 128, 128, 128), 1, 32, None), ((3, 16, 16, 96), 1, 12, 3),
             ((2, 64, 64, 320), 1, 32, 4), ((64, 8, 8, 64), 1, 8, None),
             ((4, 32, 32, 320), 1, 32, 5), ((1, 128, 128, 128), 1, 32, 5),
             ((2, 64, 64, 320), 1, 32, None)]
    need = max(b2.workspace_size(*(s[0], s[3], s[1], s[2]) if cl else s, g, torch.float16, cl)
               for s, cl, g, _ in calls)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    lib = b2.library()
    for i, (shape, cl, G, force) in enumerate(calls):
        assert lib.b200norm_testing_force(0, force or 0) == 0
        d = synthetic.skip_group_inputs(shape, np.float16, np.float32, seed=40 + i,
                                        channels_last=cl, skip="nc", bias=True)
        y, s = b2.skip_group(to_dev(d["x"]), to_dev(d["skip"]), to_dev(d["gamma"]),
                             to_dev(d["beta"]), to_dev(d["bias"]), groups=G, activation=1,
                             channels_last=cl, want_sum=True, workspace=ws)
        torch.cuda.synchronize()
        ry, rs = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"], groups=G,
                                   activation=1, channels_last=cl)
        assert_bitexact(to_host(s), rs)
        assert_y_close(to_host(y), ry)
    b2.workspace_status(ws)


@pytest.mark.parametrize("flag", [1, 2, 7, -1])
def test_any_nonzero_channels_last_means_nhwc(flag):
    """The C entry reads every non-zero channels_last as NHWC (SkipGroupNorm
    README, Attributes, channels_last): raw calls with 1, 2, 7 and -1 give the
    NHWC result bit for bit."""
    shape, G = (2, 8, 8, 64), 8
    d = synthetic.skip_group_inputs(shape, np.float16, np.float32, seed=17, channels_last=1,
                                    skip="nc", bias=True)
    x, sk, ga, be, bi = (to_dev(d[k]) for k in ("x", "skip", "gamma", "beta", "bias"))
    N, H, W, C = shape
    y = torch.empty_like(x)
    s = torch.empty_like(x)
    ws = torch.zeros(b2.workspace_size(N, C, H, W, G, torch.float16, 1), dtype=torch.uint8,
                     device="cuda")
    dims = (ctypes.c_int64 * 4)(N, C, 0, 0)
    st = b2.library().b200norm_skip_group(
        ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(sk.data_ptr()), 2, dims,
        ctypes.c_void_p(bi.data_ptr()), ctypes.c_void_p(ga.data_ptr()),
        ctypes.c_void_p(be.data_ptr()), ctypes.c_void_p(y.data_ptr()),
        ctypes.c_void_p(s.data_ptr()), N, C, H, W, F16, F32, G, 1e-5, 1, flag,
        ctypes.c_void_p(ws.data_ptr()), ws.numel(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    ry, rs = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"], groups=G,
                               activation=1, channels_last=1)
    assert_bitexact(to_host(s), rs)
    assert_y_close(to_host(y), ry)


def test_cached_workspace_on_a_non_current_stream():
    """skip_group(stream=s) without an explicit workspace: the binding makes
    and clears its cached workspace on s itself (so the clear is ordered
    before the kernels on s), and replaces it on s when a larger shape needs
    more; results match the oracle on both shapes."""
    side = torch.cuda.Stream()
    cur = torch.cuda.current_stream()
    for shape, G in (((2, 16, 16, 64), 8), ((2, 64, 64, 320), 32)):
        d = synthetic.skip_group_inputs(shape, np.float16, np.float32, seed=61, channels_last=1,
                                        skip="nc", bias=True)
        t = {k: to_dev(v) for k, v in d.items()}
        side.wait_stream(cur)
        y, s = b2.skip_group(t["x"], t["skip"], t["gamma"], t["beta"], t["bias"], groups=G,
                             activation=1, channels_last=1, want_sum=True, stream=side)
        cur.wait_stream(side)
        torch.cuda.synchronize()
        ry, rs = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"],
                                   groups=G, activation=1, channels_last=1)
        assert_bitexact(to_host(s), rs)
        assert_y_close(to_host(y), ry)
