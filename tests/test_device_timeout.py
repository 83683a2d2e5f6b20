"""The bounded device-side wait: a grid barrier that can never complete gives
up after its limit, records B200NORM_ERR_DEVICE_TIMEOUT in the workspace, and
leaves the CUDA context usable.  Nothing here faults or hangs the GPU: the
probe kernel's only wait is bounded by %globaltimer."""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import residual_add_normalization_gb300 as b2
from residual_add_normalization_gb300 import synthetic
from helpers import assert_y_close, to_dev, to_host

pytestmark = pytest.mark.gpu

TIMEOUT = 5


def test_unsatisfiable_barrier_reports_timeout_and_context_survives():
    lib = b2.library()
    ws = torch.zeros(b2.workspace_size(2, 64, 8, 8, 4), dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t0 = time.time()
    assert lib.b200norm_testing_barrier_timeout(ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                                20_000_000, stream) == 0
    st = lib.b200norm_workspace_status(ctypes.c_void_p(ws.data_ptr()), stream)
    elapsed = time.time() - t0
    assert st == TIMEOUT, lib.b200norm_status_string(st)
    assert b"gave up" in lib.b200norm_last_error()
    assert elapsed < 10.0
    with pytest.raises(b2.B200NormError):
        b2.workspace_status(ws)
    # every CTA left the barrier after giving up, so the counts are back at zero
    ctl = ws[:16].view(torch.int32).cpu().numpy()
    assert ctl[0] == 0 and ctl[1] == 0 and ctl[2] == TIMEOUT
    # re-initialise, then the same workspace serves a real call
    b2.workspace_init(ws)
    b2.workspace_status(ws)
    d = synthetic.skip_group_inputs((2, 8, 8, 64), np.float16, np.float32, seed=1,
                                    channels_last=1, skip="nc", bias=True)
    y, _ = b2.skip_group(to_dev(d["x"]), to_dev(d["skip"]), to_dev(d["gamma"]),
                         to_dev(d["beta"]), to_dev(d["bias"]), groups=4, activation=1,
                         workspace=ws)
    b2.workspace_status(ws)
    ry, _ = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"], groups=4,
                              activation=1)
    assert_y_close(to_host(y), ry)


def test_workspace_left_ready_after_many_calls():
    """The cooperative route's barrier resets itself: many back-to-back calls
    on one workspace, alternating two shapes whose cooperative grids differ in
    size, keep working and leave the arrival and departure counts at zero and
    no error."""
    shapes = [((2, 64, 64, 320), 32), ((1, 16, 16, 512), 16)]
    grids = set()
    for (N, H, W, C), G in shapes:
        out = (ctypes.c_int64 * 8)()
        # float16 X, float32 gamma/beta, NHWC, 16-byte aligned
        assert b2.library().b200norm_testing_plan_group(N, C, H, W, G, 1, 0, 1, 1, out) == 0
        assert out[0] == 2  # the cooperative route
        grids.add(out[5])
    assert len(grids) == 2
    ws = torch.zeros(max(b2.workspace_size(N, C, H, W, G, torch.float16, 1)
                         for (N, H, W, C), G in shapes), dtype=torch.uint8, device="cuda")
    cases = []
    for k, (shape, G) in enumerate(shapes):
        d = synthetic.skip_group_inputs(shape, np.float16, np.float32, seed=3 + k,
                                        channels_last=1, skip="nc", bias=True)
        cases.append((d, G, [to_dev(d[key]) for key in ("x", "skip", "gamma", "beta", "bias")]))
    ys = [None, None]
    for i in range(50):
        d, G, args = cases[i % 2]
        ys[i % 2], _ = b2.skip_group(*args, groups=G, activation=1, channels_last=1, workspace=ws)
    b2.workspace_status(ws)
    ctl = ws[:16].view(torch.int32).cpu().numpy()
    # arrivals and departures back at zero, no error recorded
    assert ctl[0] == 0 and ctl[1] == 0 and ctl[2] == 0
    for (d, G, _), y in zip(cases, ys):
        ry, _ = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"], groups=G,
                                  activation=1, channels_last=1)
        assert_y_close(to_host(y), ry)


def test_pipelined_rows_stall_reports_timeout_and_recovers():
    """The pipelined row schedule's waits are bounded: with its producer
    stalled (no copy is issued, so no tile ever lands) every consumer gives up
    after the limit, the status call reports the timeout once and clears it,
    and the next normal launch is correct."""
    lib = b2.library()
    d = synthetic.gated_rms_inputs((40000, 128), 128, np.float16, seed=2)
    x, g, sc = (to_dev(d[k]) for k in ("x", "gate", "scale"))
    assert lib.b200norm_testing_force(3, 0) == 0
    try:
        assert lib.b200norm_testing_pipe_stall(1, 20_000_000) == 0
        t0 = time.time()
        b2.gated_rms(x, g, sc, epsilon=1e-5)
        with pytest.raises(b2.B200NormError) as e:
            b2.rows_status()
        assert e.value.status == TIMEOUT
        assert time.time() - t0 < 10.0
        b2.rows_status()  # the record was cleared
    finally:
        lib.b200norm_testing_pipe_stall(0, 0)
    try:
        y = b2.gated_rms(x, g, sc, epsilon=1e-5)
        b2.rows_status()
    finally:
        lib.b200norm_testing_force(0, 0)
    ry = oracle.gated_rms(d["x"], d["gate"], d["scale"], epsilon=1e-5)
    assert_y_close(to_host(y), ry)
