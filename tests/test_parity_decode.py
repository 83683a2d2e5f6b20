"""GPU parity for decode-shaped rows (a few rows of 4K-8K elements) and for
chains of dependent calls.

Decode-shaped SkipSimplifiedLayerNormalization / GatedRMSNorm calls have too
few rows to fill the GPU, so their rows may be split over a cluster of CTAs
(a DSMEM reduction across the cluster).  Every split the schedule code can
take is forced here and compared with the oracle.

Launches allow programmatic dependent launch: a kernel may be scheduled while
the one before it on the stream drains, and waits for it before touching
memory.  The chain tests feed each call's output into the next call (a
read-after-write on the stream) and reuse buffers the previous call read (a
write-after-read), eagerly and from a CUDA graph, and require the results to
equal those of the same chain run with the feature switched off.
"""
import numpy as np
import pytest
import torch

import oracle
import residual_add_normalization_gb300 as b2
from residual_add_normalization_gb300 import synthetic
from helpers import assert_bitexact, assert_y_close, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset():
    yield
    lib = b2.library()
    lib.b200norm_testing_force_split(0, 0)
    lib.b200norm_testing_set_pdl(1)


SPLITS = [(1, 8), (1, 4), (2, 4), (4, 2), (4, 1), (8, 1), (8, 2), (16, 1)]


def _force(csize, nv):
    assert b2.library().b200norm_testing_force_split(csize, nv) == 0


@pytest.mark.parametrize("dtype", [np.float16, np.float32, synthetic.BFLOAT16])
@pytest.mark.parametrize("rows,hidden", [(1, 4096), (3, 8192), (16, 4096), (2, 5000)])
@pytest.mark.parametrize("split", SPLITS)
def test_decode_skip_rms_forced_splits(dtype, rows, hidden, split):
    ve = 16 // np.dtype(dtype).itemsize
    nvec = hidden // ve if hidden % ve == 0 else hidden
    if -(-nvec // (split[0] * split[1])) > 512:
        pytest.skip("split needs more than 512 threads per CTA")
    d = synthetic.skip_rms_inputs((rows, hidden), dtype, seed=rows + hidden, bias=True)
    _force(*split)
    y, s = b2.skip_rms(to_dev(d["input"]), to_dev(d["skip"]), to_dev(d["gamma"]),
                       to_dev(d["bias"]), epsilon=synthetic.SSLN_EPS)
    torch.cuda.synchronize()
    ry, rs = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"],
                             epsilon=synthetic.SSLN_EPS)
    assert_bitexact(to_host(s), rs)
    assert_y_close(to_host(y), ry)


@pytest.mark.parametrize("dtype", [np.float16, np.float32, synthetic.BFLOAT16])
@pytest.mark.parametrize("rows,C", [(1, 8192), (4, 4096), (2, 2056)])
@pytest.mark.parametrize("split", SPLITS)
def test_decode_gated_forced_splits(dtype, rows, C, split):
    ve = 16 // np.dtype(dtype).itemsize
    nvec = C // ve if C % ve == 0 else C
    if -(-nvec // (split[0] * split[1])) > 512:
        pytest.skip("split needs more than 512 threads per CTA")
    d = synthetic.gated_rms_inputs((rows, C), C, dtype, seed=rows * 3 + C)
    _force(*split)
    y = b2.gated_rms(to_dev(d["x"]), to_dev(d["gate"]), to_dev(d["scale"]), epsilon=1e-5)
    torch.cuda.synchronize()
    ry = oracle.gated_rms(d["x"], d["gate"], d["scale"], epsilon=1e-5)
    assert_y_close(to_host(y), ry)


def test_forced_split_too_small_for_row_is_rejected():
    _force(1, 1)
    x = torch.zeros((1, 65536), dtype=torch.float16, device="cuda")
    g = torch.ones(65536, dtype=torch.float16, device="cuda")
    with pytest.raises(b2.B200NormError, match="512"):
        b2.skip_rms(x, x.clone(), g)


def _chain(n_links, graph):
    """n_links dependent calls: SSLN -> GatedRMSNorm -> SkipGroupNorm (NHWC and
    NCHW), each reading the previous output, on one stream.  Returns every
    intermediate as host arrays."""
    rows, hidden = 8, 4096  # 32768 elements = one (2, 16, 16, 64) image
    d = synthetic.skip_rms_inputs((rows, hidden), np.float16, seed=5, bias=True)
    x, sk, ga, bi = (to_dev(d[k]) for k in ("input", "skip", "gamma", "bias"))
    gate = to_dev(synthetic.gated_rms_inputs((rows, hidden), 128, np.float16, seed=6)["gate"])
    scale = to_dev(synthetic.gated_rms_inputs((rows, hidden), 128, np.float16, seed=6)["scale"])
    gd = synthetic.skip_group_inputs((2, 16, 16, 64), np.float16, np.float32, seed=7,
                                     channels_last=1, skip="nc", bias=True)
    gg, gb, gsk, gbi = (to_dev(gd[k]) for k in ("gamma", "beta", "skip", "bias"))
    cd = synthetic.skip_group_inputs((2, 64, 16, 16), np.float16, np.float32, seed=8,
                                     channels_last=0, skip="full", bias=False)
    cg, cb = to_dev(cd["gamma"]), to_dev(cd["beta"])
    outs = []
    bufs = {}

    def body():
        cur = x
        for i in range(n_links):
            y, s = b2.skip_rms(cur, sk, ga, bi, epsilon=1e-6, output=bufs.get(("y", i)),
                               sum_out=bufs.get(("s", i)))
            bufs[("y", i)], bufs[("s", i)] = y, s
            z = b2.gated_rms(y, gate, scale, epsilon=1e-5, y=bufs.get(("z", i)))
            bufs[("z", i)] = z
            img = z.view(2, 16, 16, 64)
            w, ws = b2.skip_group(img, gsk, gg, gb, gbi, groups=8, activation=1,
                                  channels_last=1, y=bufs.get(("w", i)),
                                  s=bufs.get(("ws", i)))
            bufs[("w", i)], bufs[("ws", i)] = w, ws
            v, _ = b2.skip_group(w.view(2, 64, 16, 16), w.view(2, 64, 16, 16).flip(0), cg, cb,
                                 groups=4, activation=0, channels_last=0, want_sum=False,
                                 y=bufs.get(("v", i)))
            bufs[("v", i)] = v
            cur = v.view(rows, hidden)

    body()  # allocates every output and warms the plan caches
    torch.cuda.synchronize()
    for t in bufs.values():
        if t is not None:
            t.fill_(float("nan"))
    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            body()
        g.replay()
    else:
        body()
    torch.cuda.synchronize()
    for key in sorted(bufs, key=str):
        if bufs[key] is not None:
            outs.append(to_host(bufs[key]))
    return outs


@pytest.mark.parametrize("graph", [False, True])
def test_dependent_chain_identical_with_and_without_pdl(graph):
    lib = b2.library()
    assert lib.b200norm_testing_set_pdl(0) == 0
    ref = _chain(6, graph)
    assert lib.b200norm_testing_set_pdl(1) == 0
    got = _chain(6, graph)
    assert len(ref) == len(got)
    for a, b in zip(ref, got):
        assert not np.isnan(b.astype(np.float32)).any()
        assert_bitexact(b, a, "chain output")


def test_decode_chain_first_link_matches_oracle():
    """The first SSLN of the chain against the oracle (the chain test above
    only compares the library with itself)."""
    d = synthetic.skip_rms_inputs((4, 4096), np.float16, seed=5, bias=True)
    y, s = b2.skip_rms(to_dev(d["input"]), to_dev(d["skip"]), to_dev(d["gamma"]),
                       to_dev(d["bias"]), epsilon=1e-6)
    torch.cuda.synchronize()
    ry, rs = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"], epsilon=1e-6)
    assert_bitexact(to_host(s), rs)
    assert_y_close(to_host(y), ry)
