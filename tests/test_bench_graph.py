"""Parity in the exact launch configuration the benchmark times: bench.py's
own call closures (explicit workspaces, rotating buffer sets), captured into
one CUDA graph per step and replayed, at the four step workloads' full sizes,
against the oracle element by element."""
import os
import sys

import numpy as np
import pytest
import torch

import oracle
import residual_add_normalization_gb300 as b2
from helpers import assert_bitexact, assert_y_close, to_host

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_step_graph_outputs_match_oracle():
    sys.path.insert(0, ROOT)
    import bench
    dev = torch.device("cuda", 0)
    calls = bench.make_calls(torch, b2, dev)
    stream = torch.cuda.current_stream(dev)
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)

    def step():
        for c in calls:
            c["fn"]()

    with torch.cuda.stream(cap):
        step()  # warm the plan caches on the capture stream, as the benchmark does
    torch.cuda.synchronize()
    for c in calls:
        for o in c["outs"]:
            o.fill_(float("nan"))
    graph = bench.capture(torch, step, cap)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()

    for c in calls:
        spec, d = c["spec"], c["host"]
        outs = [to_host(o) for o in c["outs"]]
        if spec["op"] == "skip_rms":
            ry, rs = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"],
                                     epsilon=spec["epsilon"])
            assert_y_close(outs[0], ry, c["name"] + " Y")
            assert_bitexact(outs[1], rs, c["name"] + " S")
        elif spec["op"] == "gated_rms":
            ry = oracle.gated_rms(d["x"], d["gate"], d["scale"], epsilon=spec["epsilon"])
            assert_y_close(outs[0], ry, c["name"] + " Y")
        else:
            ry, rs = oracle.skip_group(d["x"], d["skip"], d["gamma"], d["beta"], d["bias"],
                                       groups=spec["groups"], activation=spec["activation"],
                                       epsilon=spec["epsilon"],
                                       channels_last=spec["channels_last"])
            assert_y_close(outs[0], ry, c["name"] + " Y")
            if spec["want_sum"]:
                assert_bitexact(outs[1], rs, c["name"] + " S")
    assert not any(np.isnan(o.astype(np.float32)).any() for c in calls
                   for o in [to_host(t) for t in c["outs"]])
