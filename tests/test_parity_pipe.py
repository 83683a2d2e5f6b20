"""GPU parity of the pipelined lane-group row schedule (inputs streamed through
shared memory by bulk copies) against the CPU oracle, forced through the
testing hook so that every case runs it whatever the planner would choose.

Shapes cover lane groups of 1..32 threads, rows with fewer vectors than their
lane group, ragged last tiles, and more tiles per CTA than the ring has
stages (so every stage is reused and its barrier parity flips).  Bar: S
bit-exact; Y within the stated tolerance (tests/helpers.py).
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

DTYPES = [np.float32, np.float16, synthetic.BFLOAT16]
PIPE_WARPS = 31      # consumer warps per CTA
STAGES = 6


def _vectors(n, dtype):
    return n * np.dtype(dtype).itemsize // 16


def _tile_rows(n, dtype):
    tpr = 1
    while tpr < _vectors(n, dtype):
        tpr *= 2
    return PIPE_WARPS * (32 // tpr)


@pytest.fixture(autouse=True)
def _force_pipe():
    assert b2.library().b200norm_testing_force(3, 0) == 0
    yield
    b2.library().b200norm_testing_force(0, 0)
    b2.rows_status()


def _gated_cases():
    cases = []
    for dt in DTYPES:
        ve = 16 // np.dtype(dt).itemsize
        for nvec in (1, 2, 3, 8, 12, 16, 32):
            C = nvec * ve
            tr = _tile_rows(C, dt)
            for rows in (1, tr - 1, 3 * tr + 5):
                cases.append((dt, C, rows))
    return cases


@pytest.mark.parametrize("dtype,C,rows", _gated_cases())
def test_gated_pipe(dtype, C, rows):
    d = synthetic.gated_rms_inputs((rows, C), C, dtype, seed=rows % 97 + C)
    y = b2.gated_rms(to_dev(d["x"]), to_dev(d["gate"]), to_dev(d["scale"]), epsilon=1e-5)
    ry = oracle.gated_rms(d["x"], d["gate"], d["scale"], epsilon=1e-5)
    assert_y_close(to_host(y), ry)


@pytest.mark.parametrize("dtype", DTYPES)
def test_gated_pipe_stage_reuse(dtype):
    """Enough tiles that every CTA of a full GPU takes more than twice the
    ring's stages (C = 128: 64-row tiles for 16-bit types, 32 for float32)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    C = 128
    rows = sms * (2 * STAGES + 3) * _tile_rows(C, dtype) + 37
    d = synthetic.gated_rms_inputs((rows, C), C, dtype, seed=11)
    y = b2.gated_rms(to_dev(d["x"]), to_dev(d["gate"]), to_dev(d["scale"]), epsilon=1e-5)
    ry = oracle.gated_rms(d["x"], d["gate"], d["scale"], epsilon=1e-5)
    assert_y_close(to_host(y), ry)


def _ssln_cases():
    cases = []
    for dt in DTYPES:
        ve = 16 // np.dtype(dt).itemsize
        for nvec in (1, 3, 8, 32):
            n = nvec * ve
            tr = _tile_rows(n, dt)
            for rows in (2, 2 * tr + 3):
                for bias in (True, False):
                    cases.append((dt, n, rows, bias))
    return cases


@pytest.mark.parametrize("dtype,n,rows,bias", _ssln_cases())
def test_skip_rms_pipe(dtype, n, rows, bias):
    d = synthetic.skip_rms_inputs((rows, n), dtype, seed=rows + n, bias=bias)
    y, s, m, inv = b2.skip_rms_stats(to_dev(d["input"]), to_dev(d["skip"]), to_dev(d["gamma"]),
                                     to_dev(d["bias"]), epsilon=1e-5, want_sum=True)
    ry, rs, rm, rinv = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"],
                                       epsilon=1e-5, want_stats=True)
    assert_bitexact(to_host(s), rs)
    assert_y_close(to_host(y), ry)
    assert np.all(to_host(m) == 0)
    np.testing.assert_allclose(to_host(inv), rinv, rtol=2e-6)


@pytest.mark.parametrize("dtype", DTYPES)
def test_skip_rms_pipe_without_sum(dtype):
    d = synthetic.skip_rms_inputs((1000, 64), dtype, seed=4, bias=True)
    y, s = b2.skip_rms(to_dev(d["input"]), to_dev(d["skip"]), to_dev(d["gamma"]),
                       to_dev(d["bias"]), epsilon=1e-6, want_sum=False)
    ry, _ = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"], epsilon=1e-6)
    assert s is None
    assert_y_close(to_host(y), ry)


def test_pipe_refuses_long_rows_and_unaligned_tensors():
    d = synthetic.gated_rms_inputs((4, 4096), 4096, np.float16, seed=1)
    with pytest.raises(b2.B200NormError) as e:
        b2.gated_rms(to_dev(d["x"]), to_dev(d["gate"]), to_dev(d["scale"]), epsilon=1e-5)
    assert e.value.status == 2  # B200NORM_ERR_UNSUPPORTED
    x = torch.empty(4 * 128 + 1, dtype=torch.float16, device="cuda")[1:].view(4, 128)
    x.copy_(to_dev(d["x"][:, :128]))
    g = to_dev(d["gate"][:, :128])
    with pytest.raises(b2.B200NormError) as e:
        b2.gated_rms(x, g, to_dev(d["scale"][:128]), epsilon=1e-5)
    assert e.value.status == 2


def test_pipe_status_clean_after_runs():
    d = synthetic.gated_rms_inputs((20000, 128), 128, np.float16, seed=3)
    for _ in range(3):
        b2.gated_rms(to_dev(d["x"]), to_dev(d["gate"]), to_dev(d["scale"]), epsilon=1e-5)
    st = b2.library().b200norm_rows_status(
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0


def _stalled_call_times_out(fn):
    """Runs fn with the pipelined schedule stalled; True if a pipelined kernel
    ran (only it waits on copies, so only it records a timeout)."""
    lib = b2.library()
    assert lib.b200norm_testing_pipe_stall(1, 20_000_000) == 0
    try:
        fn()
        try:
            b2.rows_status()
            return False
        except b2.B200NormError as e:
            assert e.status == 5  # B200NORM_ERR_DEVICE_TIMEOUT
            return True
    finally:
        lib.b200norm_testing_pipe_stall(0, 0)


# tiles from which automatic choice pipelines SkipSimplifiedLayerNormalization
MIN_TILES = {np.float16: 8192, np.float32: 256, synthetic.BFLOAT16: 256}


@pytest.mark.parametrize("dtype", DTYPES)
def test_skip_rms_short_rows_take_pipe_automatically(dtype):
    """Automatic choice gives long runs of short SkipSimplifiedLayerNormalization
    rows the pipelined schedule, shorter runs and GatedRMSNorm the lane kernel,
    and row mode 1 never the pipelined one; every path matches the oracle."""
    lib = b2.library()
    n = 64 if dtype == np.float16 else 128
    tr = _tile_rows(n, dtype)
    big = MIN_TILES[dtype] * tr - 5       # the last of MIN_TILES tiles is ragged
    small = (MIN_TILES[dtype] - 1) * tr   # one tile fewer
    for rows, mode, pipelined in ((big, 0, True), (big, 1, False), (small, 0, False)):
        d = synthetic.skip_rms_inputs((rows, n), dtype, seed=rows + mode, bias=True)
        args = [to_dev(d[k]) for k in ("input", "skip", "gamma", "bias")]
        assert lib.b200norm_testing_force(mode, 0) == 0
        assert _stalled_call_times_out(lambda: b2.skip_rms(*args, epsilon=1e-5)) == pipelined
        y, s = b2.skip_rms(*args, epsilon=1e-5)
        b2.rows_status()
        ry, rs = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"], epsilon=1e-5)
        assert_bitexact(to_host(s), rs)
        assert_y_close(to_host(y), ry)
    assert lib.b200norm_testing_force(0, 0) == 0
    d = synthetic.gated_rms_inputs((big, n), n, dtype, seed=5)
    args = [to_dev(d[k]) for k in ("x", "gate", "scale")]
    assert not _stalled_call_times_out(lambda: b2.gated_rms(*args, epsilon=1e-5))


def test_pipe_stage_reuse_stress():
    """Many passes over large short-row inputs through the pipelined schedule.
    A stage handed back before every read of it completed lets the next
    tile's copy land under a reader: rows then mix two tiles.  S must equal
    the oracle's bits in every pass, and GatedRMSNorm's Y every pass's bits."""
    n, dtype = 64, np.float16
    rows = 8192 * _tile_rows(n, dtype) - 5
    d = synthetic.skip_rms_inputs((rows, n), dtype, seed=21, bias=True)
    args = [to_dev(d[k]) for k in ("input", "skip", "gamma", "bias")]
    _, rs = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"], epsilon=1e-5)
    want = to_dev(rs).view(torch.int16)
    y = torch.empty_like(args[0])
    s = torch.empty_like(args[0])
    for i in range(16):
        b2.skip_rms(*args, epsilon=1e-5, output=y, sum_out=s)
        bad = int((s.view(torch.int16) != want).sum())
        assert bad == 0, f"pass {i}: {bad} elements of S differ"
    g = synthetic.gated_rms_inputs((rows, n), n, dtype, seed=22)
    gargs = [to_dev(g[k]) for k in ("x", "gate", "scale")]
    first = b2.gated_rms(*gargs, epsilon=1e-5).view(torch.int16)
    out = torch.empty_like(gargs[0])
    for i in range(16):
        b2.gated_rms(*gargs, epsilon=1e-5, y=out)
        bad = int((out.view(torch.int16) != first).sum())
        assert bad == 0, f"pass {i}: {bad} elements of Y differ from the first pass"
    ry = oracle.gated_rms(g["x"], g["gate"], g["scale"], epsilon=1e-5)
    assert_y_close(to_host(out), ry)
