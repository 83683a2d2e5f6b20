"""Host threads calling the library at once, each on its own stream (the
pages' operators are stateless; the library's plan caches are shared and
locked, its error text is per thread, and the binding caches one SkipGroupNorm
workspace per stream).  Every thread must get the results of a single-threaded
run, bit for bit."""
import threading

import numpy as np
import pytest
import torch

import residual_add_normalization_gb300 as b2
from residual_add_normalization_gb300 import synthetic
from helpers import assert_bitexact, to_dev, to_host

pytestmark = pytest.mark.gpu


def _work(seed):
    d1 = synthetic.skip_rms_inputs((64, 4096), np.float16, seed=seed, bias=True)
    d2 = synthetic.gated_rms_inputs((256, 1024), 128, np.float16, seed=seed)
    d3 = synthetic.skip_group_inputs((2, 32, 32, 320), np.float16, np.float32, seed=seed,
                                     channels_last=1, skip="nc", bias=True)
    d4 = synthetic.skip_group_inputs((2, 320, 16, 16), np.float32, np.float16, seed=seed,
                                     channels_last=0, skip="full", bias=False)
    # NHWC too large for the register-resident cooperative route: one grid
    # through L2 (route 5), also cooperative
    d5 = synthetic.skip_group_inputs((4, 64, 64, 320), np.float16, np.float32, seed=seed,
                                     channels_last=1, skip="nc", bias=True)
    t = [{k: to_dev(v) for k, v in d.items()} for d in (d1, d2, d3, d4, d5)]

    def run():
        y1, s1 = b2.skip_rms(t[0]["input"], t[0]["skip"], t[0]["gamma"], t[0]["bias"])
        y2 = b2.gated_rms(t[1]["x"], t[1]["gate"], t[1]["scale"])
        y3, s3 = b2.skip_group(t[2]["x"], t[2]["skip"], t[2]["gamma"], t[2]["beta"], t[2]["bias"],
                               groups=32, activation=1, channels_last=1, want_sum=True)
        y4, _ = b2.skip_group(t[3]["x"], t[3]["skip"], t[3]["gamma"], t[3]["beta"], None,
                              groups=32, activation=0, channels_last=0)
        y5, s5 = b2.skip_group(t[4]["x"], t[4]["skip"], t[4]["gamma"], t[4]["beta"], t[4]["bias"],
                               groups=32, activation=1, channels_last=1, want_sum=True)
        return [y1, s1, y2, y3, s3, y4, y5, s5]
    return run


def test_concurrent_threads_match_single_thread():
    runs = [_work(seed) for seed in range(4)]
    expected = []
    for run in runs:
        outs = run()
        torch.cuda.synchronize()
        expected.append([to_host(o) for o in outs])
    errors, results = [], [None] * len(runs)

    def worker(i):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for _ in range(20):
                    outs = runs[i]()
                stream.synchronize()
            results[i] = [to_host(o) for o in outs]
        except Exception as e:  # noqa: BLE001 -- reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(runs))]
    for th in threads:
        th.start()
    for th in threads:
        th.join(120)
    assert not errors, errors
    for exp, got in zip(expected, results):
        assert got is not None
        for a, b in zip(got, exp):
            assert_bitexact(a, b, "threaded result")


def test_error_text_is_per_thread():
    lib = b2.library()
    seen = {}

    def worker(name, hidden):
        st = lib.b200norm_skip_rms(None, None, None, None, None, None, 2, hidden, 1, 1e-5, None)
        seen[name] = (st, lib.b200norm_last_error())

    threads = [threading.Thread(target=worker, args=("zero", 0)),
               threading.Thread(target=worker, args=("big", 1 << 31))]
    for th in threads:
        th.start()
    for th in threads:
        th.join(30)
    assert seen["zero"][0] == 1 and b"hidden must be > 0" in seen["zero"][1]
    assert seen["big"][0] == 2 and b"2^31" in seen["big"][1]
