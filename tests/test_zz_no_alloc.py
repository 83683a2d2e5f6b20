"""The allocation-free SkipGroupNorm entry point, b200norm_skip_group_noalloc.

It serves callers that cannot allocate device memory -- a plugin whose host
hands it only its input and output buffers, or a service that reserved its
memory up front and must not allocate mid-request -- by using a fixed scratch
array inside the library instead of a caller workspace.  These tests call it
through the C ABI and compare its outputs with those of the regular entry
point, b200norm_skip_group (caller-provided workspace), on two calls in a row,
so the second call also sees the scratch the first one left behind.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.  It also passes on its own in a
fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import residual_add_normalization_gb300 as b2
from residual_add_normalization_gb300 import synthetic
from helpers import assert_bitexact, assert_y_close, to_dev, to_host

pytestmark = pytest.mark.gpu

_CODE = {np.dtype(np.float32): 0, np.dtype(np.float16): 1}


def _lib():
    lib = b2.library()
    fn = lib.b200norm_skip_group_noalloc
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [vp, vp, i32, ctypes.POINTER(ctypes.c_int64), vp, vp, vp, vp, vp, i64, i64, i64,
                   i64, i32, i32, i32, ctypes.c_float, i32, i32, vp]
    fn.restype = i32
    return lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(d, groups, act, cl, want_sum, eps=1e-5):
    lib = _lib()
    x = to_dev(d["x"])
    sk, ga, be, bi = (to_dev(d[k]) for k in ("skip", "gamma", "beta", "bias"))
    N, C, H, W = ((x.shape[0], x.shape[3], x.shape[1], x.shape[2]) if cl else tuple(x.shape))
    y = torch.full_like(x, float("nan"))
    s = torch.full_like(x, float("nan")) if want_sum else None
    dims = (ctypes.c_int64 * 4)(*([int(v) for v in sk.shape] + [0] * (4 - sk.dim())))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.b200norm_skip_group_noalloc(
        _p(x), _p(sk), sk.dim(), dims, _p(bi), _p(ga), _p(be), _p(y), _p(s), N, C, H, W,
        _CODE[d["x"].dtype], _CODE[d["gamma"].dtype], groups, eps, act, cl, stream)
    assert st == 0, (lib.b200norm_status_string(st), lib.b200norm_last_error())
    torch.cuda.synchronize()
    return to_host(y), to_host(s)


def _call_regular(d, groups, act, cl, want_sum, eps=1e-5):
    y, s = b2.skip_group(to_dev(d["x"]), to_dev(d["skip"]), to_dev(d["gamma"]),
                         to_dev(d["beta"]), to_dev(d["bias"]), groups=groups, activation=act,
                         epsilon=eps, channels_last=cl, want_sum=want_sum)
    torch.cuda.synchronize()
    return to_host(y), to_host(s)


# The NHWC case uses the cooperative route (grid barrier and moment slots in
# the scratch); the NCHW cases cover the resident route and the two-phase
# route (moment slots).
CASES = [
    dict(shape=(2, 64, 64, 320), cl=1, dtype=np.float16, mdtype=np.float32, skip="nc",
         bias=True, groups=32, act=1, want_sum=True),
    dict(shape=(16, 1280, 16, 16), cl=0, dtype=np.float32, mdtype=np.float16, skip="full",
         bias=False, groups=32, act=0, want_sum=False),
    dict(shape=(1, 64, 128, 128), cl=0, dtype=np.float16, mdtype=np.float32, skip="nc",
         bias=True, groups=4, act=1, want_sum=True),
]


@pytest.mark.parametrize("case", CASES, ids=["nhwc_coop", "nchw_resident", "nchw_two_phase"])
def test_noalloc_matches_regular_entry_two_calls_in_a_row(case):
    outs = []
    for seed in (101, 202):  # two calls in a row on the shared scratch
        d = synthetic.skip_group_inputs(case["shape"], case["dtype"], case["mdtype"], seed=seed,
                                        channels_last=case["cl"], skip=case["skip"],
                                        bias=case["bias"])
        y, s = _call_noalloc(d, case["groups"], case["act"], case["cl"], case["want_sum"])
        ry, rs = _call_regular(d, case["groups"], case["act"], case["cl"], case["want_sum"])
        assert_y_close(y, ry)
        if case["want_sum"]:
            assert_bitexact(s, rs)
        outs.append(y)
    assert not np.array_equal(outs[0], outs[1])  # the second call really recomputed


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = _lib()
    x = torch.zeros(1, dtype=torch.float16, device="cuda")
    dims = (ctypes.c_int64 * 4)(2, 4096, 0, 0)
    # 4096 groups need 2048 * 4096 * 16 bytes of moment slots, beyond the 2 MiB scratch
    st = lib.b200norm_skip_group_noalloc(_p(x), _p(x), 2, dims, None, _p(x), _p(x), _p(x), None,
                                         2, 4096, 8, 8, 1, 1, 4096, 1e-5, 0, 1, None)
    assert st == 2  # B200NORM_ERR_UNSUPPORTED
    assert b"static scratch" in lib.b200norm_last_error()
