"""Tensors of more than 2^31 elements (64-bit offsets everywhere): one call of
each operator on the device, then the oracle on sampled rows, spans or group
instances copied back to the host (the oracle computes them one by one).
Inputs are drawn on the device with a seeded generator; every check compares
the library's outputs with the oracle's on the same bits."""
import numpy as np
import pytest
import torch

import oracle
import residual_add_normalization_gb300 as b2
from residual_add_normalization_gb300 import synthetic
from helpers import assert_bitexact, assert_y_close, to_host

pytestmark = pytest.mark.gpu

BIG = (1 << 31) + 4096  # just over 2^31 elements


def _free_gb():
    free, _ = torch.cuda.mem_get_info()
    return free / 1e9


def test_huge_skip_rms():
    hidden = 2048
    rows = -(-BIG // hidden)
    if _free_gb() < 4 * rows * hidden * 2 / 1e9 + 4:
        pytest.skip("not enough device memory")
    x = synthetic.device_normal((rows, hidden), torch.float16, 1, "cuda")
    sk = synthetic.device_normal((rows, hidden), torch.float16, 2, "cuda")
    ga = synthetic.device_normal((hidden,), torch.float16, 3, "cuda", 1.0, 0.1)
    bi = synthetic.device_normal((hidden,), torch.float16, 4, "cuda", 0.0, 0.1)
    y, s = b2.skip_rms(x, sk, ga, bi, epsilon=1e-6)
    torch.cuda.synchronize()
    pick = np.unique(np.concatenate([[0, 1], np.linspace(2, rows - 3, 12).astype(np.int64),
                                     [rows - 2, rows - 1]]))
    idx = torch.from_numpy(pick).cuda()
    hx, hs, hy = to_host(x[idx]), to_host(s[idx]), to_host(y[idx])
    ry, rs = oracle.skip_rms(hx, to_host(sk[idx]), to_host(ga), to_host(bi), epsilon=1e-6)
    assert_bitexact(hs, rs)
    assert_y_close(hy, ry)


def test_huge_gated_rms():
    C = 128
    spans = -(-BIG // C)
    if _free_gb() < 3 * spans * C * 2 / 1e9 + 4:
        pytest.skip("not enough device memory")
    x = synthetic.device_normal((spans, C), torch.float16, 5, "cuda")
    g = synthetic.device_normal((spans, C), torch.float16, 6, "cuda")
    sc = synthetic.device_normal((C,), torch.float16, 7, "cuda", 1.0, 0.1)
    y = b2.gated_rms(x, g, sc)
    torch.cuda.synchronize()
    pick = np.unique(np.concatenate([[0], np.linspace(1, spans - 2, 14).astype(np.int64),
                                     [spans - 1]]))
    idx = torch.from_numpy(pick).cuda()
    ry = oracle.gated_rms(to_host(x[idx]), to_host(g[idx]), to_host(sc), epsilon=1e-5)
    assert_y_close(to_host(y[idx]), ry)


def test_huge_skip_rms_pipelined():
    """Short bfloat16 rows take the pipelined schedule automatically: tiles
    and stores past 2^31 elements."""
    hidden = 256
    rows = -(-BIG // hidden)
    if _free_gb() < 4 * rows * hidden * 2 / 1e9 + 4:
        pytest.skip("not enough device memory")
    x = synthetic.device_normal((rows, hidden), torch.bfloat16, 21, "cuda")
    sk = synthetic.device_normal((rows, hidden), torch.bfloat16, 22, "cuda")
    ga = synthetic.device_normal((hidden,), torch.bfloat16, 23, "cuda", 1.0, 0.1)
    bi = synthetic.device_normal((hidden,), torch.bfloat16, 24, "cuda", 0.0, 0.1)
    y, s = b2.skip_rms(x, sk, ga, bi, epsilon=1e-6)
    b2.rows_status()
    pick = np.unique(np.concatenate([[0, 1], np.linspace(2, rows - 3, 12).astype(np.int64),
                                     [rows - 2, rows - 1]]))
    idx = torch.from_numpy(pick).cuda()
    ry, rs = oracle.skip_rms(to_host(x[idx]), to_host(sk[idx]), to_host(ga), to_host(bi),
                             epsilon=1e-6)
    assert_bitexact(to_host(s[idx]), rs)
    assert_y_close(to_host(y[idx]), ry)


def test_huge_gated_rms_pipelined():
    """GatedRMSNorm through the pipelined schedule (forced) past 2^31 elements."""
    C = 128
    spans = -(-BIG // C)
    if _free_gb() < 3 * spans * C * 2 / 1e9 + 4:
        pytest.skip("not enough device memory")
    x = synthetic.device_normal((spans, C), torch.float16, 25, "cuda")
    g = synthetic.device_normal((spans, C), torch.float16, 26, "cuda")
    sc = synthetic.device_normal((C,), torch.float16, 27, "cuda", 1.0, 0.1)
    assert b2.library().b200norm_testing_force(3, 0) == 0
    try:
        y = b2.gated_rms(x, g, sc)
        b2.rows_status()
    finally:
        b2.library().b200norm_testing_force(0, 0)
    pick = np.unique(np.concatenate([[0], np.linspace(1, spans - 2, 14).astype(np.int64),
                                     [spans - 1]]))
    idx = torch.from_numpy(pick).cuda()
    ry = oracle.gated_rms(to_host(x[idx]), to_host(g[idx]), to_host(sc), epsilon=1e-5)
    assert_y_close(to_host(y[idx]), ry)


@pytest.mark.parametrize("cl", [0, 1])
def test_huge_skip_group(cl):
    N, C, groups = 1, 256, 32
    HW = -(-BIG // C)
    H = 2048
    W = -(-HW // H)
    shape = (N, H, W, C) if cl else (N, C, H, W)
    numel = N * C * H * W
    if _free_gb() < 3 * numel * 2 / 1e9 + 4:
        pytest.skip("not enough device memory")
    x = synthetic.device_normal(shape, torch.float16, 8 + cl, "cuda")
    sk = synthetic.device_normal((N, C), torch.float16, 10, "cuda")
    ga = synthetic.device_normal((C,), torch.float32, 11, "cuda", 1.0, 0.1)
    be = synthetic.device_normal((C,), torch.float32, 12, "cuda", 0.0, 0.1)
    y, s = b2.skip_group(x, sk, ga, be, None, groups=groups, activation=1, channels_last=cl,
                         want_sum=True)
    torch.cuda.synchronize()
    cpg = C // groups
    for g in (0, groups - 1):  # the first and the last group (offsets beyond 2^31)
        cs = slice(g * cpg, (g + 1) * cpg)
        part = (lambda t: t[..., cs]) if cl else (lambda t: t[:, cs])
        hx = to_host(part(x).contiguous())
        ry, rs = oracle.skip_group(hx, to_host(sk[:, cs].contiguous()), to_host(ga[cs]),
                                   to_host(be[cs]), None, groups=1, activation=1,
                                   channels_last=cl)
        assert_bitexact(to_host(part(s).contiguous()), rs)
        assert_y_close(to_host(part(y).contiguous()), ry)
