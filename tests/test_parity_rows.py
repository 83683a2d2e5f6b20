"""GPU parity: SkipSimplifiedLayerNormalization and GatedRMSNorm kernels against
the CPU oracle on the same seeded inputs, through the C ABI (via the binding).

Bar: S bit-exact; Y within the stated tolerance (tests/helpers.py).  Shapes
span every row schedule: lane groups of 1..32 threads with several rows per
warp, warp-per-row, CTA-per-row, cluster-per-row (DSMEM reduction) and the
walking schedule, on vector and scalar paths, with ragged tails.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import residual_add_normalization_gb300 as b2
from residual_add_normalization_gb300 import synthetic
import helpers
from helpers import assert_bitexact, assert_y_close, to_dev, to_host

pytestmark = pytest.mark.gpu

DTYPES = [np.float32, np.float16, synthetic.BFLOAT16]


def _plan(n, T, rows=4):
    out = (ctypes.c_int64 * 8)()
    assert b2.library().b200norm_testing_plan_rows(rows, n, T, 1, out) == 0
    return dict(zip(("mode", "ve", "tpr", "nv", "rpg", "block", "csize", "grid"), out))


@pytest.fixture(autouse=True)
def _reset_force():
    yield
    b2.library().b200norm_testing_force(0, 0)


def _dev(a, shift):
    """Device copy of ``a``; with ``shift`` > 0 it starts ``shift`` elements
    into its allocation (16-byte misalignment -> scalar path)."""
    if a is None:
        return None
    if not shift:
        return to_dev(a)
    t = to_dev(a, "cpu")
    flat = torch.empty(a.size + shift, dtype=t.dtype, device="cuda")
    v = flat[shift:].view(a.shape)
    v.copy_(t)
    return v


def run_ssln(d, eps, want_sum=True, stats=False, shift=0):
    x, sk, g, b = (_dev(d[k], shift) for k in ("input", "skip", "gamma", "bias"))
    out = _dev(np.zeros_like(d["input"]), shift) if shift else None
    sout = _dev(np.zeros_like(d["input"]), shift) if (shift and want_sum) else None
    if stats:
        y, s, m, inv = b2.skip_rms_stats(x, sk, g, b, epsilon=eps, want_sum=want_sum, output=out,
                                         sum_out=sout)
        torch.cuda.synchronize()
        return to_host(y), to_host(s), to_host(m), to_host(inv)
    y, s = b2.skip_rms(x, sk, g, b, epsilon=eps, want_sum=want_sum, output=out, sum_out=sout)
    torch.cuda.synchronize()
    return to_host(y), to_host(s)


SSLN_SHAPES = [
    (1, 8), (3, 5), (7, 24), (64, 16), (33, 256), (9, 200), (17, 1000), (64, 768),
    (5, 4096), (3, 12288), (2, 33000), (2, 65536), (1, 262144),
]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", SSLN_SHAPES)
@pytest.mark.parametrize("bias,want_sum", [(True, True), (False, False), (True, False)])
def test_skip_rms_matches_oracle(dtype, shape, bias, want_sum):
    d = synthetic.skip_rms_inputs(shape, dtype, seed=shape[0] * 7 + shape[1] % 101 + bias,
                                  bias=bias)
    eps = synthetic.SSLN_EPS
    y, s = run_ssln(d, eps, want_sum)
    ry, rs = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"], epsilon=eps)
    if want_sum:
        assert_bitexact(s, rs)
    else:
        assert s is None
    assert_y_close(y, ry)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", [(4, 4096), (6, 200), (3, 7)])
def test_skip_rms_unaligned_scalar_path(dtype, shape):
    d = synthetic.skip_rms_inputs(shape, dtype, seed=3, bias=True)
    y, s = run_ssln(d, 1e-6, True, shift=1)
    ry, rs = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"], epsilon=1e-6)
    assert_bitexact(s, rs)
    assert_y_close(y, ry)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", [(5, 4096), (7, 24), (2, 33000)])
def test_skip_rms_forced_walk(dtype, shape):
    assert b2.library().b200norm_testing_force(2, 0) == 0
    d = synthetic.skip_rms_inputs(shape, dtype, seed=5, bias=True)
    y, s = run_ssln(d, 1e-5, True)
    ry, rs = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"], epsilon=1e-5)
    assert_bitexact(s, rs)
    assert_y_close(y, ry)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape", [(6, 40), (3, 4096), (2, 70000)])
def test_skip_rms_stats_outputs(dtype, shape):
    d = synthetic.skip_rms_inputs(shape, dtype, seed=8, bias=True)
    y, s, m, inv = run_ssln(d, 0.01, True, stats=True)
    ry, rs, rm, rinv = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"],
                                       epsilon=0.01, want_stats=True)
    assert_bitexact(s, rs)
    assert_y_close(y, ry)
    assert np.all(m == 0) and m.shape == rm.shape
    np.testing.assert_allclose(inv, rinv, rtol=2e-6)


def test_skip_rms_edge_values():
    """Zero rows with eps = 0 give NaN on both sides; a +0 bias turns -0 into
    +0 while an absent bias keeps -0; large values stay finite in float32."""
    x = np.zeros((4, 64), np.float16)
    x[1] = -0.0
    x[2] = np.float16(60000)
    x[3, ::2] = np.float16(-3.5)
    sk = x.copy()
    sk[2] = np.float16(0.5)
    g = np.ones(64, np.float16)
    for bias in (None, np.zeros(64, np.float16)):
        y, s = run_ssln(dict(input=x, skip=sk, gamma=g, bias=bias), 0.0)
        ry, rs = oracle.skip_rms(x, sk, g, bias, epsilon=0.0)
        assert_bitexact(s, rs)
        assert_y_close(y, ry)
        assert np.isnan(y[0]).all()


def test_skip_rms_edge_values_bf16():
    """bfloat16: zero rows with eps = 0 give NaN on both sides, -0 survives an
    absent bias, and values up to 1e18 (squares far beyond float16's range,
    row sums of squares still finite in float32) give matching S and Y."""
    x = np.zeros((4, 64), np.float32)
    x[1] = -0.0
    x[2] = 1e18
    x[2, 1::2] = -3e17
    x[3, ::2] = -3.5
    sk = x.copy()
    sk[2] = 0.5
    x, sk = synthetic.to_bfloat16(x), synthetic.to_bfloat16(sk)
    g = synthetic.to_bfloat16(np.ones(64, np.float32))
    for bias in (None, synthetic.to_bfloat16(np.zeros(64, np.float32))):
        y, s = run_ssln(dict(input=x, skip=sk, gamma=g, bias=bias), 0.0)
        ry, rs = oracle.skip_rms(x, sk, g, bias, epsilon=0.0)
        assert_bitexact(s, rs)
        assert_y_close(y, ry)
        assert np.isnan(helpers.values(y[0])).all()


def test_skip_rms_empty_rows():
    x = torch.empty((0, 64), dtype=torch.float16, device="cuda")
    g = torch.ones(64, dtype=torch.float16, device="cuda")
    y, s = b2.skip_rms(x, x, g)
    assert y.shape == (0, 64) and s.shape == (0, 64)


def test_skip_rms_plan_coverage():
    """The shape list above reaches every schedule."""
    modes = set()
    for shape in SSLN_SHAPES:
        for T in (0, 1):
            p = _plan(shape[-1], T, shape[0])
            modes.add((p["mode"], p["csize"] > 1, p["ve"] > 1, p["tpr"] < 32 and p["mode"] == 0))
    assert {m[0] for m in modes} >= {0, 1}
    assert any(m[1] for m in modes), "no cluster plan"
    assert any(not m[2] for m in modes) and any(m[2] for m in modes)
    assert any(m[3] for m in modes), "no sub-warp lane groups"


# ---------------------------------------------------------------------------
# GatedRMSNorm
# ---------------------------------------------------------------------------

def run_gated(d, eps, scale_shape=None):
    x, g = to_dev(d["x"]), to_dev(d["gate"])
    sc = to_dev(d["scale"] if scale_shape is None else d["scale"].reshape(scale_shape))
    y = b2.gated_rms(x, g, sc, epsilon=eps)
    torch.cuda.synchronize()
    return to_host(y)


GATED_CASES = [
    ((3, 4), 1), ((2, 64, 8192), 128), ((5, 72), 24), ((4, 96), 96), ((3, 512), 64),
    ((2, 4096), 4096), ((7, 100), 100), ((2, 2, 20000), 20000), ((9,), 3), ((16, 8), 8),
    ((1, 131072), 131072),
]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shape,C", GATED_CASES)
def test_gated_matches_oracle(dtype, shape, C):
    d = synthetic.gated_rms_inputs(shape, C, dtype, seed=C % 97)
    y = run_gated(d, 1e-5)
    ry = oracle.gated_rms(d["x"], d["gate"], d["scale"], epsilon=1e-5)
    assert_y_close(y, ry)


@pytest.mark.parametrize("spelling", [(128,), (1, 128), (128, 1)])
def test_gated_scale_spellings(spelling):
    d = synthetic.gated_rms_inputs((4, 256), 128, np.float16, seed=2)
    y = run_gated(d, 1e-5, spelling)
    ry = oracle.gated_rms(d["x"], d["gate"], d["scale"], epsilon=1e-5)
    assert_y_close(y, ry)


@pytest.mark.parametrize("dtype", DTYPES)
def test_gated_forced_walk(dtype):
    assert b2.library().b200norm_testing_force(2, 0) == 0
    d = synthetic.gated_rms_inputs((4, 1024), 128, dtype, seed=6)
    y = run_gated(d, 1e-6)
    ry = oracle.gated_rms(d["x"], d["gate"], d["scale"], epsilon=1e-6)
    assert_y_close(y, ry)


def test_gated_extreme_gates():
    """Large positive / negative gates (SiLU saturation) and eps = 0 zero spans."""
    x = np.random.default_rng(1).standard_normal((8, 16)).astype(np.float32)
    x[0] = 0.0
    g = np.linspace(-120, 120, 128, dtype=np.float32).reshape(8, 16)
    sc = np.ones(16, np.float32)
    y = run_gated(dict(x=x, gate=g, scale=sc), 0.0)
    ry = oracle.gated_rms(x, g, sc, epsilon=0.0)
    assert_y_close(y, ry)
