"""Out-of-bounds and unwritten-element checks for every schedule and route.

Each output tensor is a view into a larger buffer whose every byte starts as
0xFF (a NaN pattern in float32, float16 and bfloat16).  After one call:
- the guard regions before and after the view must still be all 0xFF (no
  write outside the output), and
- the view must hold no NaN (with finite inputs every element is written).
The view starts 4096 bytes into its buffer (16-byte aligned, so the vector
paths run) or, for the scalar-path cases, one element further.
"""
import numpy as np
import pytest
import torch

import residual_add_normalization_gb300 as b2
from residual_add_normalization_gb300 import synthetic
from helpers import to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side


@pytest.fixture(autouse=True)
def _reset_force():
    yield
    b2.library().b200norm_testing_force(0, 0)


def guarded(shape, dtype, shift=0):
    """(buffer, view): a view of `shape` inside a 0xFF-filled byte buffer."""
    es = torch.tensor([], dtype=dtype).element_size()
    n = int(np.prod(shape))
    front = GUARD + shift * es
    raw = torch.full((front + n * es + GUARD,), 0xFF, dtype=torch.uint8, device="cuda")
    view = raw[front:front + n * es].view(dtype).view(shape)
    return raw, view, front, n * es


def check_guarded(raw, front, nbytes, view, what):
    torch.cuda.synchronize()
    head = raw[:front]
    tail = raw[front + nbytes:]
    assert bool((head == 0xFF).all()), f"{what}: write before the output"
    assert bool((tail == 0xFF).all()), f"{what}: write after the output"
    assert not bool(torch.isnan(view.float()).any()), f"{what}: element left unwritten"


SSLN_CASES = [  # (rows, hidden, dtype, row_mode, shift)
    (37, 64, np.float16, 0, 0),        # lane groups
    (5, 4096, np.float16, 0, 0),       # CTA per row
    (3, 40000, np.float32, 0, 0),      # cluster per row
    (2, 70000, np.float16, 2, 0),      # walk
    (1000, 64, np.float32, 3, 0),      # pipelined, ragged last tile
    (7, 24, np.float16, 0, 1),         # scalar path (unaligned outputs)
    (9, 4096, synthetic.BFLOAT16, 0, 0),
]


@pytest.mark.parametrize("rows,hidden,dtype,mode,shift", SSLN_CASES)
def test_skip_rms_writes_exactly_its_outputs(rows, hidden, dtype, mode, shift):
    assert b2.library().b200norm_testing_force(mode, 0) == 0
    d = synthetic.skip_rms_inputs((rows, hidden), dtype, seed=rows + hidden, bias=True)
    args = [to_dev(d[k]) for k in ("input", "skip", "gamma", "bias")]
    ry, y, fy, ny = guarded((rows, hidden), args[0].dtype, shift)
    rs, s, fs, ns = guarded((rows, hidden), args[0].dtype, shift)
    b2.skip_rms(*args, epsilon=1e-5, output=y, sum_out=s)
    check_guarded(ry, fy, ny, y, "output")
    check_guarded(rs, fs, ns, s, "input_skip_bias_sum")


GATED_CASES = [  # (spans, C, dtype, row_mode, shift)
    (300, 128, np.float16, 0, 0),      # lane groups
    (300, 128, np.float16, 3, 0),      # pipelined
    (4, 8192, np.float32, 0, 0),       # CTA per row
    (5, 100, np.float32, 0, 1),        # scalar path
    (64, 256, synthetic.BFLOAT16, 0, 0),
]


@pytest.mark.parametrize("spans,C,dtype,mode,shift", GATED_CASES)
def test_gated_writes_exactly_its_output(spans, C, dtype, mode, shift):
    assert b2.library().b200norm_testing_force(mode, 0) == 0
    d = synthetic.gated_rms_inputs((spans, C), C, dtype, seed=spans + C)
    args = [to_dev(d[k]) for k in ("x", "gate", "scale")]
    ry, y, fy, ny = guarded((spans, C), args[0].dtype, shift)
    b2.gated_rms(*args, epsilon=1e-5, y=y)
    check_guarded(ry, fy, ny, y, "y")


GROUP_CASES = [  # (shape, channels_last, groups, skip, forced route, shift)
    ((2, 64, 8, 8), 0, 8, "full", 0, 0),          # route 1
    ((1, 320, 64, 64), 0, 32, "nc", 0, 0),        # route 1, clusters
    ((2, 12, 5, 7), 0, 4, "full", 0, 0),          # route 1, scalar path
    ((2, 16, 16, 64), 1, 8, "nc", 2, 0),          # route 2
    ((1, 33, 17, 40), 1, 8, "full", 2, 0),        # route 2, ragged last slab
    ((2, 16, 16, 64), 1, 8, "nc", 3, 0),          # route 3, NHWC
    ((2, 64, 16, 16), 0, 8, "full", 3, 0),        # route 3, NCHW
    ((4, 32, 32, 320), 1, 32, "nc", 4, 0),        # route 4
    ((4, 32, 32, 320), 1, 32, "nc", 5, 0),        # route 5
    ((4, 32, 32, 320), 1, 32, "full", 6, 0),      # route 6 (slab in shared memory, bulk copies)
    ((1, 33, 17, 40), 1, 8, "nc", 6, 0),          # route 6, ragged last slab
    ((3, 5, 7, 12), 1, 3, "full", 6, 1),          # route 6, scalar path, unaligned outputs
    ((3, 5, 7, 12), 1, 3, "nc", 0, 1),            # scalar path, unaligned outputs
]


@pytest.mark.parametrize("shape,cl,G,skip,route,shift", GROUP_CASES)
def test_skip_group_writes_exactly_its_outputs(shape, cl, G, skip, route, shift):
    assert b2.library().b200norm_testing_force(0, route) == 0
    d = synthetic.skip_group_inputs(shape, np.float16, np.float32, seed=sum(shape) + route,
                                    channels_last=cl, skip=skip, bias=True)
    args = [to_dev(d[k]) for k in ("x", "skip", "gamma", "beta", "bias")]
    ry, y, fy, ny = guarded(shape, args[0].dtype, shift)
    rs, s, fs, ns = guarded(shape, args[0].dtype, shift)
    b2.skip_group(*args, groups=G, activation=1, channels_last=cl, y=y, s=s)
    check_guarded(ry, fy, ny, y, "y")
    check_guarded(rs, fs, ns, s, "s")
