"""The allocation-free SkipGroupNorm entry point, b200norm_skip_group_noalloc.

It serves callers that cannot allocate device memory -- a plugin whose host
hands it only its input and output buffers, or a service that reserved its
memory up front and must not allocate mid-request -- by using a fixed scratch
array inside the library instead of a caller workspace.  These tests call it
through the C ABI on two calls in a row (so the second call also sees the
scratch the first one left behind) and compare its outputs with the oracle
and, bit for bit, with those of the regular entry point, b200norm_skip_group
(caller-provided workspace).  They also check the size rule, that a call
refused for any reason enqueues nothing, and that a device-side timeout
recorded in the scratch is reported by b200norm_skip_group_noalloc_status.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.  It also passes on its own in a
fresh process.
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

_CODE = {np.dtype(np.float32): 0, np.dtype(np.float16): 1}
SCRATCH = 256 + (2 << 20)
OK, INVALID, UNSUPPORTED, TIMEOUT = 0, 1, 2, 5


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(s=None):
    return ctypes.c_void_p((s or torch.cuda.current_stream()).cuda_stream)


def _args(d, groups, act, cl, want_sum, eps=1e-5):
    """Device tensors and the C arguments of a call on inputs `d` (NaN-filled
    outputs)."""
    x = to_dev(d["x"])
    sk, ga, be, bi = (to_dev(d[k]) for k in ("skip", "gamma", "beta", "bias"))
    N, C, H, W = ((x.shape[0], x.shape[3], x.shape[1], x.shape[2]) if cl else tuple(x.shape))
    y = torch.full_like(x, float("nan"))
    s = torch.full_like(x, float("nan")) if want_sum else None
    dims = (ctypes.c_int64 * 4)(*([int(v) for v in sk.shape] + [0] * (4 - sk.dim())))
    keep = (x, sk, ga, be, bi, y, s, dims)
    args = [_p(x), _p(sk), sk.dim(), dims, _p(bi), _p(ga), _p(be), _p(y), _p(s), N, C, H, W,
            _CODE[d["x"].dtype], _CODE[d["gamma"].dtype], groups, eps, act, cl]
    return keep, args


def _call_noalloc(d, groups, act, cl, want_sum, eps=1e-5):
    lib = b2.library()
    keep, args = _args(d, groups, act, cl, want_sum, eps)
    st = lib.b200norm_skip_group_noalloc(*args, _stream())
    assert st == OK, (lib.b200norm_status_string(st), lib.b200norm_last_error())
    torch.cuda.synchronize()
    return to_host(keep[5]), to_host(keep[6])


def _call_regular(d, groups, act, cl, want_sum, eps=1e-5):
    y, s = b2.skip_group(to_dev(d["x"]), to_dev(d["skip"]), to_dev(d["gamma"]),
                         to_dev(d["beta"]), to_dev(d["bias"]), groups=groups, activation=act,
                         epsilon=eps, channels_last=cl, want_sum=want_sum)
    torch.cuda.synchronize()
    return to_host(y), to_host(s)


# The NHWC cases use the cooperative routes (grid barrier and piece slots in
# the scratch): slabs in registers (route 2), slabs in shared memory with bulk
# copies (route 6) and one grid re-reading through L2 (route 5); the NCHW
# cases cover the resident route (no slots), the two-phase route (piece
# slots) and 64 groups (the workspace size of NCHW shapes counts only the
# two-phase slots).
CASES = [
    dict(shape=(2, 64, 64, 320), cl=1, dtype=np.float16, mdtype=np.float32, skip="nc",
         bias=True, groups=32, act=1, want_sum=True, route=2),
    dict(shape=(4, 64, 64, 320), cl=1, dtype=np.float16, mdtype=np.float32, skip="full",
         bias=True, groups=32, act=1, want_sum=True, route=6),
    dict(shape=(2, 128, 128, 320), cl=1, dtype=np.float16, mdtype=np.float32, skip="nc",
         bias=True, groups=32, act=0, want_sum=True, route=5),
    dict(shape=(16, 1280, 16, 16), cl=0, dtype=np.float32, mdtype=np.float16, skip="full",
         bias=False, groups=32, act=0, want_sum=False),
    dict(shape=(1, 64, 128, 128), cl=0, dtype=np.float16, mdtype=np.float32, skip="nc",
         bias=True, groups=4, act=1, want_sum=True),
    dict(shape=(2, 128, 16, 16), cl=0, dtype=np.float32, mdtype=np.float32, skip="nc",
         bias=True, groups=64, act=1, want_sum=True),
]


@pytest.mark.parametrize("case", CASES,
                         ids=["nhwc_coop", "nhwc_slab", "nhwc_coop_l2", "nchw_resident",
                              "nchw_two_phase", "nchw_64_groups"])
def test_noalloc_matches_oracle_and_regular_entry_two_calls_in_a_row(case):
    if "route" in case:  # the route the case is here for
        N, H, W, C = case["shape"]
        out = (ctypes.c_int64 * 8)()
        assert b2.library().b200norm_testing_plan_group(
            N, C, H, W, case["groups"], _CODE[np.dtype(case["dtype"])],
            _CODE[np.dtype(case["mdtype"])], 1, 1, out) == 0
        assert out[0] == case["route"]
    outs = []
    for seed in (101, 202):  # two calls in a row on the shared scratch
        d = synthetic.skip_group_inputs(case["shape"], case["dtype"], case["mdtype"], seed=seed,
                                        channels_last=case["cl"], skip=case["skip"],
                                        bias=case["bias"])
        y, s = _call_noalloc(d, case["groups"], case["act"], case["cl"], case["want_sum"])
        oy, os_ = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"],
                                    groups=case["groups"], activation=case["act"],
                                    channels_last=case["cl"])
        assert_y_close(y, oy)
        ry, rs = _call_regular(d, case["groups"], case["act"], case["cl"], case["want_sum"])
        assert_bitexact(y, ry, "Y (against the regular entry)")
        if case["want_sum"]:
            assert_bitexact(s, os_)
            assert_bitexact(s, rs)
        outs.append(y)
    assert not np.array_equal(outs[0], outs[1])  # the second call really recomputed


def _cudart():
    """The CUDA runtime torch has loaded (for stream capture)."""
    torch.cuda.init()
    paths = []
    with open("/proc/self/maps") as fh:
        for line in fh:
            f = line.split()[-1]
            if "libcudart.so" in f and f not in paths:
                paths.append(f)
    for path in paths + ["libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so"]:
        try:
            rt = ctypes.CDLL(path)
            break
        except OSError:
            continue
    else:
        pytest.skip("no CUDA runtime library to capture a stream with")
    rt.cudaStreamBeginCapture.argtypes = [ctypes.c_void_p, ctypes.c_int]
    rt.cudaStreamEndCapture.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]
    rt.cudaGraphGetNodes.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.POINTER(ctypes.c_size_t)]
    rt.cudaGraphDestroy.argtypes = [ctypes.c_void_p]
    return rt


def _captured_nodes(fn):
    """Runs fn(stream) while a side stream is being captured (relaxed mode);
    returns (fn's result, the number of graph nodes it enqueued)."""
    rt = _cudart()
    side = torch.cuda.Stream()
    h = _stream(side)
    assert rt.cudaStreamBeginCapture(h, 2) == 0  # cudaStreamCaptureModeRelaxed
    try:
        res = fn(h)
    finally:
        graph = ctypes.c_void_p()
        assert rt.cudaStreamEndCapture(h, ctypes.byref(graph)) == 0
    n = ctypes.c_size_t(0)
    assert rt.cudaGraphGetNodes(graph, None, ctypes.byref(n)) == 0
    rt.cudaGraphDestroy(graph)
    return res, n.value


def test_refused_calls_enqueue_nothing():
    lib = b2.library()
    d = synthetic.skip_group_inputs((2, 64, 16, 16), np.float32, np.float32, seed=3,
                                    channels_last=0, skip="nc", bias=True)
    _call_noalloc(d, 8, 1, 0, True)  # set-up on this device, before any capture
    keep, good = _args(d, 8, 1, 0, True)
    x, y = keep[0], keep[5]
    bad = {
        "groups do not divide C": (15, lambda a: a.__setitem__(15, 7), INVALID),
        "activation 2": (17, lambda a: a.__setitem__(17, 2), INVALID),
        "epsilon NaN": (16, lambda a: a.__setitem__(16, float("nan")), INVALID),
        "skip shape": (2, lambda a: a.__setitem__(2, 3), INVALID),
        "no Y": (7, lambda a: a.__setitem__(7, None), INVALID),
        "Y overlaps X": (7, lambda a: a.__setitem__(7, _p(x)), INVALID),
        "misaligned Y": (7, lambda a: a.__setitem__(7, ctypes.c_void_p(y.data_ptr() + 2)),
                         INVALID),
        "types": (13, lambda a: a.__setitem__(13, 9), UNSUPPORTED),
    }
    for what, (_, edit, want) in bad.items():
        args = list(good)
        edit(args)
        st, n = _captured_nodes(lambda h: lib.b200norm_skip_group_noalloc(*args, h))
        assert st == want, (what, lib.b200norm_last_error())
        assert n == 0, f"{what}: a refused call enqueued {n} graph nodes"
    # beyond the scratch: 64 groups of an NHWC shape the L2 route can take
    dn = synthetic.skip_group_inputs((2, 8, 8, 64), np.float16, np.float32, seed=4,
                                     channels_last=1, skip="nc", bias=True)
    assert b2.workspace_size(2, 64, 8, 8, 64, torch.float16, 1) > SCRATCH
    keep2, big = _args(dn, 64, 1, 1, False)
    st, n = _captured_nodes(lambda h: lib.b200norm_skip_group_noalloc(*big, h))
    assert st == UNSUPPORTED and n == 0
    assert b"static scratch" in lib.b200norm_last_error()
    # positive control: a valid call under the same capture enqueues its work
    st, n = _captured_nodes(lambda h: lib.b200norm_skip_group_noalloc(*good, h))
    assert st == OK and n > 0


def test_size_rule_is_the_workspace_size():
    """A shape is served exactly when b200norm_skip_group_workspace_size() of
    it fits the scratch; the documented families land on the right side."""
    lib = b2.library()
    for shape, G, cl in (((2, 64, 64, 320), 32, 1), ((56, 8, 8, 64), 32, 1),
                         ((2, 128, 16, 16), 64, 0), ((16, 1280, 16, 16), 1280, 0)):
        N, C, H, W = (shape[0], shape[3], shape[1], shape[2]) if cl else shape
        assert b2.workspace_size(N, C, H, W, G, torch.float16, cl) <= SCRATCH, shape
    for shape, G, cl in (((2, 8, 8, 64), 64, 1), ((1, 8, 8, 4096), 4096, 1)):
        N, C, H, W = (shape[0], shape[3], shape[1], shape[2]) if cl else shape
        assert b2.workspace_size(N, C, H, W, G, torch.float16, cl) > SCRATCH, shape
    d = synthetic.skip_group_inputs((2, 8, 8, 4096), np.float16, np.float16, seed=6,
                                    channels_last=1, skip="nc", bias=False)
    keep, args = _args(d, 4096, 0, 1, False)
    st = lib.b200norm_skip_group_noalloc(*args, _stream())
    assert st == UNSUPPORTED
    assert b"static scratch" in lib.b200norm_last_error()


def test_timeout_in_the_scratch_is_reported_and_calls_keep_working():
    """A bounded wait that gives up records its timeout in the scratch; later
    calls still work (their counters are cleared, the record is kept), and
    b200norm_skip_group_noalloc_status reports the record once, then clears
    it.  The probe's wait is bounded by %globaltimer: nothing faults."""
    lib = b2.library()
    d = synthetic.skip_group_inputs((2, 16, 16, 64), np.float16, np.float32, seed=5,
                                    channels_last=1, skip="nc", bias=True)
    _call_noalloc(d, 8, 1, 1, True)  # set-up on this device
    assert lib.b200norm_skip_group_noalloc_status(_stream()) == OK
    assert lib.b200norm_testing_noalloc_barrier_timeout(20_000_000, _stream()) == OK
    y, s = _call_noalloc(d, 8, 1, 1, True)  # the cooperative route, after the timeout
    oy, os_ = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"], groups=8,
                                activation=1, channels_last=1)
    assert_y_close(y, oy)
    assert_bitexact(s, os_)
    st = lib.b200norm_skip_group_noalloc_status(_stream())
    assert st == TIMEOUT, lib.b200norm_status_string(st)
    assert b"gave up" in lib.b200norm_last_error()
    b2.noalloc_status()  # the read above cleared the record: no error now
    assert lib.b200norm_skip_group_noalloc_status(_stream()) == OK
