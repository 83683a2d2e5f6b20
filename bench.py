"""Benchmark: effective HBM GB/s of the fused residual-add + normalization path.

One step = one call of each operator on its large workload, i.e. one pass of
the whole hot path:
  SkipSimplifiedLayerNormalization fp16 (8, 2048, 4096), bias, S
  GatedRMSNorm fp16 (4, 4096, 8192), C = 128
  SkipGroupNorm NHWC fp16 (2, 64, 64, 320), (N, C) skip, bias, S, SiLU
  SkipGroupNorm NCHW fp32 (16, 1280, 16, 16), full skip, fp16 gamma/beta
value = algorithmic bytes (every input element read once, every output
written once) / device time, summed over the step.  A step moves 1.42 GB, far
more than the 129 MB L2, so every operator starts with its inputs evicted by
the other operators' traffic.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica on its own GPU (the
operators have no cross-device step); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from residual_add_normalization_gb300 import synthetic  # noqa: E402

METRIC = ("effective HBM GB/s and % of GB300 peak per op; rows/s (1 GPU, device-timed)")
STEP_WORKLOADS = ["ssln_fp16_8x2048x4096", "gated_fp16_4x4096x8192_c128",
                  "sgn_nhwc_fp16_2x64x64x320", "sgn_nchw_fp32_16x1280x16x16"]
# Decode-shaped calls, timed on their own (per-call latency, rows/s).
DECODE_WORKLOADS = ["ssln_fp16_decode_1x4096", "ssln_fp16_decode_64x4096",
                    "gated_fp16_decode_64x8192_c8192"]
# bfloat16 variants of the large workloads, timed like the step workloads.
BF16_WORKLOADS = ["ssln_bf16_8x2048x4096", "gated_bf16_4x4096x8192_c128",
                  "sgn_nhwc_bf16_2x64x64x320", "sgn_nchw_bf16_16x1280x16x16"]
# short SkipSimplifiedLayerNormalization rows: the pipelined bulk-copy schedule
SHORT_WORKLOADS = ["ssln_fp32_262144x128"]
# mid-size NHWC SkipGroupNorm: the cooperative route with slabs in shared memory
MID_WORKLOADS = ["sgn_nhwc_fp16_4x64x64x320"]
# the small SkipSimplifiedLayerNormalization batch: latency-bound, timed on its own
SMALL_WORKLOADS = ["ssln_fp32_64x768"]
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes per launch of the dominant kernel from an ncu capture, keyed by
# the digest of its kernel family's sources when it was taken (None: not
# captured for the current sources).
NCU_TRAFFIC = {
    # ncu (dram__bytes_read.sum + dram__bytes_write.sum) of the GatedRMSNorm lane
    # kernel: 536,887,296 B read + 230,401,280 B written
    ("gated_fp16_4x4096x8192_c128", "eef15244cf9415ca"): 767288576,
}


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [f.strip() for f in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        note = "sampled during the timed region"
        if not inside and self.samples:
            # timed region shorter than the sampling period: nearest samples
            inside = [min(self.samples, key=lambda ts: abs(ts[0] - (t0 + t1) / 2))[1]]
            note = "timed region shorter than the sampling period; nearest sample"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "no samples"}
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(s[0]) for s in inside if num(s[0]) is not None]
        mx = [num(s[1]) for s in inside if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4)
                          if len(s) > 4 + i and s[4 + i].lower().startswith("active")})
        pw = [num(s[2]) for s in inside if num(s[2]) is not None]
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(inside), "note": note}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def host_tensor(torch, a):
    """A CPU tensor over a host array (bfloat16 arrays are uint16 patterns)."""
    if synthetic.is_bf16(a.dtype):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(a)


def l2_bytes(torch, dev):
    try:
        return int(torch.cuda.get_device_properties(dev).L2_cache_size)
    except (AttributeError, RuntimeError):
        return 129 * 2**20


def make_calls(torch, b2, dev, names=None, rotate=True):
    """Device inputs, preallocated outputs and call closures per workload.

    With `rotate`, each workload gets `nsets` independent input/output sets,
    enough that the other sets move at least 3 x L2 of traffic between two
    uses of one set; the per-operator timing cycles through them, so the
    inputs it reads come from HBM, not from L2.  Without it there is one set
    (latency-bound calls, whose inputs a preceding kernel has just written)."""
    calls = []
    l2 = l2_bytes(torch, dev)
    for name in (STEP_WORKLOADS if names is None else names):
        spec, d = synthetic.workload(name)
        nsets = 1 + -(-3 * l2 // synthetic.algorithmic_bytes(name)) if rotate else 1
        fns, sets = [], []
        for _ in range(nsets):
            t = {k: (None if v is None else host_tensor(torch, v).to(dev)) for k, v in d.items()}
            if spec["op"] == "skip_rms":
                y, s = torch.empty_like(t["input"]), torch.empty_like(t["input"])
                def fn(t=t, y=y, s=s, spec=spec):
                    b2.skip_rms(t["input"], t["skip"], t["gamma"], t["bias"],
                                epsilon=spec["epsilon"], output=y, sum_out=s)
                outs = [y, s]
            elif spec["op"] == "gated_rms":
                y = torch.empty_like(t["x"])
                def fn(t=t, y=y, spec=spec):
                    b2.gated_rms(t["x"], t["gate"], t["scale"], epsilon=spec["epsilon"], y=y)
                outs = [y]
            else:
                y = torch.empty_like(t["x"])
                s = torch.empty_like(t["x"]) if spec["want_sum"] else None
                shape = spec["shape"]
                N, C, H, W = ((shape[0], shape[3], shape[1], shape[2]) if spec["channels_last"]
                              else shape)
                ws = torch.zeros(b2.workspace_size(N, C, H, W, spec["groups"], t["x"].dtype,
                                                   spec["channels_last"]),
                                 dtype=torch.uint8, device=dev)
                def fn(t=t, y=y, s=s, spec=spec, ws=ws):
                    b2.skip_group(t["x"], t["skip"], t["gamma"], t["beta"], t["bias"],
                                  groups=spec["groups"], activation=spec["activation"],
                                  epsilon=spec["epsilon"], channels_last=spec["channels_last"],
                                  y=y, s=s, workspace=ws)
                outs = [y] + ([s] if s is not None else [])
            fns.append(fn)
            sets.append((t, outs))
        calls.append(dict(name=name, spec=spec, fns=fns, fn=fns[0], inputs=sets[0][0],
                          outs=sets[0][1], host=d, bytes=synthetic.algorithmic_bytes(name),
                          units=synthetic.units(name)))
    return calls


def capture(torch, fn, stream):
    """A CUDA graph of whatever `fn` enqueues on the current stream."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def max_over_ranks(torch, dist, ms, device):
    """The largest of every rank's `ms` (the job takes as long as its slowest
    replica); `ms` itself without a process group."""
    if not dist:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(step_bytes, world, ms_per_step):
    """Whole-job throughput: every replica moves `step_bytes` per step, and a
    step of the job takes `ms_per_step` (the slowest replica's)."""
    return step_bytes * world / (ms_per_step * 1e-3) / 1e9


OP_MIN_LAUNCHES = 100  # per operator, over all timed replays
OP_MIN_ROUNDS = 10     # timed replays per operator (median and best over them)


def op_graphs_of(torch, calls, stream):
    """One graph per workload: 2 x nsets calls cycling through its sets (at
    least 8)."""
    graphs, reps = [], []
    for c in calls:
        rep = max(8, 2 * len(c["fns"]))
        def many(c=c, rep=rep):
            for r in range(rep):
                c["fns"][r % len(c["fns"])]()
        graphs.append(capture(torch, many, stream))
        reps.append(rep)
    return graphs, reps


def time_op_graphs(torch, graphs, reps, stream):
    """Milliseconds per call of each workload over back-to-back replays of
    its graph (after one untimed replay) -- at least OP_MIN_ROUNDS replays and
    OP_MIN_LAUNCHES calls -- with an event between consecutive replays:
    (mean, median, best, calls) per workload.  The mean is the whole run's
    time over its calls; median and best are over the replays."""
    out = []
    for g, rep in zip(graphs, reps):
        rounds = max(OP_MIN_ROUNDS, -(-OP_MIN_LAUNCHES // rep))
        g.replay()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(rounds + 1)]
        ev[0].record(stream)
        for k in range(rounds):
            g.replay()
            ev[k + 1].record(stream)
        torch.cuda.synchronize()
        per = np.array([ev[k].elapsed_time(ev[k + 1]) / rep for k in range(rounds)])
        out.append((ev[0].elapsed_time(ev[rounds]) / (rounds * rep), float(np.median(per)),
                    float(per.min()), rounds * rep))
    return out


UNIT_NAMES = {"skip_rms": "rows", "gated_rms": "C-spans", "skip_group": "group instances"}


def op_entry(c, t):
    ms, med, best, n = t
    peak, _ = peak_hbm()
    gbs = c["bytes"] / (ms * 1e-3) / 1e9
    return {"us_per_call": round(ms * 1e3, 3), "us_median": round(med * 1e3, 3),
            "us_best": round(best * 1e3, 3), "GB_s": round(gbs, 1),
            "of_measured_peak": round(gbs / peak, 4), "of_8TBs": round(gbs / NOMINAL_HBM_GBS, 4),
            "units_per_s": float(f"{c['units'] / (ms * 1e-3):.4g}"),
            "units": UNIT_NAMES[c["spec"]["op"]], "sets": len(c["fns"]), "calls": n}


def launches_per_call(b2, spec):
    import ctypes
    if spec["op"] != "skip_group":
        return 1
    shape = spec["shape"]
    N, C, H, W = ((shape[0], shape[3], shape[1], shape[2]) if spec["channels_last"]
                  else shape)
    code = {np.dtype(np.float32): 0, np.dtype(np.float16): 1}
    out = (ctypes.c_int64 * 8)()
    b2.library().b200norm_testing_plan_group(N, C, H, W, spec["groups"],
                                             code[np.dtype(spec["dtype"])],
                                             code[np.dtype(spec["mdtype"])],
                                             spec["channels_last"], 1, out)
    return 2 if out[0] in (3, 4) else 1


def run_ours(args, rank, world, dist):
    import torch
    import residual_add_normalization_gb300 as b2
    from residual_add_normalization_gb300 import buildlib

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    b2.library()  # raises if the CUDA library is missing: no fallback
    calls = make_calls(torch, b2, dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        for c in calls:
            c["fn"]()

    for _ in range(args.warmup):
        for c in calls:
            for f in c["fns"]:
                f()
    torch.cuda.synchronize()

    # The timed work is replayed from CUDA graphs captured once, so the device
    # timeline is not stretched by the host-side cost of the Python calls.
    # `step_graph` holds one step (one call of each operator, in order);
    # `op_graphs[i]` holds REP calls of operator i cycling through its sets.
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        step()  # an eager pass on the capture stream (library caches warm)
    torch.cuda.synchronize()
    step_graph = capture(torch, step, cap)
    op_graphs, reps = op_graphs_of(torch, calls, cap)
    torch.cuda.synchronize()
    for _ in range(3):
        step_graph.replay()
    torch.cuda.synchronize()

    # --- device-timed region: K steps --------------------------------------
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        step_graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    total_ms = max_over_ranks(torch, dist, start.elapsed_time(end), dev)

    # --- per-operator launch durations (events around each operator graph) --
    per_call_ms = time_op_graphs(torch, op_graphs, reps, stream)
    del op_graphs

    # --- bfloat16 variants of the large workloads, timed the same way -------
    bf16_ops = {}
    if not args.no_bf16:
        bcalls = make_calls(torch, b2, dev, BF16_WORKLOADS)
        for c in bcalls:
            for f in c["fns"]:
                f()
        torch.cuda.synchronize()
        graphs, breps = op_graphs_of(torch, bcalls, cap)
        bms = time_op_graphs(torch, graphs, breps, stream)
        bf16_ops = {c["name"]: op_entry(c, ms) for c, ms in zip(bcalls, bms)}
        del graphs, bcalls
        torch.cuda.synchronize()

    # --- short rows (the pipelined schedule) and mid-size NHWC SkipGroupNorm
    # (slabs in shared memory), timed the same way -------------------------------
    def timed_section(names):
        scalls = make_calls(torch, b2, dev, names)
        for c in scalls:
            for f in c["fns"]:
                f()
        torch.cuda.synchronize()
        graphs, sreps = op_graphs_of(torch, scalls, cap)
        sms_ = time_op_graphs(torch, graphs, sreps, stream)
        out = {c["name"]: op_entry(c, ms) for c, ms in zip(scalls, sms_)}
        del graphs, scalls
        torch.cuda.synchronize()
        return out

    short_ops = {}
    if not args.no_short:
        short_ops = timed_section(SHORT_WORKLOADS)
        b2.rows_status()
    mid_ops = {} if args.no_mid else timed_section(MID_WORKLOADS)

    # --- latency-bound calls: per-call time in a graph of back-to-back calls -
    def latency_section(names):
        out = {}
        for c in make_calls(torch, b2, dev, names, rotate=False):
            rep = 200
            c["fn"]()
            torch.cuda.synchronize()
            g = capture(torch, lambda c=c, rep=rep: [c["fn"]() for _ in range(rep)], cap)
            g.replay()
            per = []
            for _ in range(OP_MIN_ROUNDS):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                per.append(e0.elapsed_time(e1) / rep)
            best, med = min(per), float(np.median(per))
            out[c["name"]] = {
                "us_per_call": round(best * 1e3, 3), "us_median": round(med * 1e3, 3),
                "units_per_s": float(f"{c['units'] / (best * 1e-3):.4g}"),
                "units": UNIT_NAMES[c["spec"]["op"]],
                "GB_s": round(c["bytes"] / (best * 1e-3) / 1e9, 1),
                "algorithmic_bytes": c["bytes"], "calls": rep * OP_MIN_ROUNDS}
            del g
        torch.cuda.synchronize()
        return out

    # the small SkipSimplifiedLayerNormalization batch (fp32 64 x 768): latency-bound
    small = {} if args.only else latency_section(SMALL_WORKLOADS)
    decode = {} if args.no_decode else latency_section(DECODE_WORKLOADS)

    # --- end to end through the public API with host buffers ---------------
    e2e_steps = 0 if args.no_e2e else min(args.steps, 20)
    pinned_in = [{k: (None if v is None or not e2e_steps else host_tensor(torch, v).pin_memory())
                  for k, v in c["host"].items()} for c in calls]
    pinned_out = [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in c["outs"]]
                  if e2e_steps else [] for c in calls]
    h2d = sum(v.numel() * v.element_size() for d in pinned_in for v in d.values()
              if v is not None)
    d2h = sum(o.numel() * o.element_size() for c in calls for o in c["outs"])

    # Three streams: host->device copies of each operator's inputs, the
    # operator calls (public API on the compute stream), device->host copies
    # of its outputs.  Events order each operator after its inputs, each
    # download after its operator, and each reuse of a device buffer after
    # the previous step's use of it, so uploads, compute and downloads of
    # different operators overlap.
    s_up, s_comp, s_down = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in calls]
    ev_done = [torch.cuda.Event() for _ in calls]
    ev_out = [torch.cuda.Event() for _ in calls]
    first = [True]

    def e2e_step():
        for i, (c, pin, pout) in enumerate(zip(calls, pinned_in, pinned_out)):
            with torch.cuda.stream(s_up):
                if not first[0]:
                    s_up.wait_event(ev_done[i])  # previous step no longer reads them
                for k, v in pin.items():
                    if v is not None:
                        c["inputs"][k].copy_(v, non_blocking=True)
                ev_in[i].record(s_up)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in[i])
                if not first[0]:
                    s_comp.wait_event(ev_out[i])  # previous outputs downloaded
                c["fn"]()
                ev_done[i].record(s_comp)
            with torch.cuda.stream(s_down):
                s_down.wait_event(ev_done[i])
                for o, p in zip(c["outs"], pout):
                    p.copy_(o, non_blocking=True)
                ev_out[i].record(s_down)
        first[0] = False

    e2e_ms = float("nan")
    if e2e_steps:
        e2e_step()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for st in (s_up, s_comp, s_down):
            st.wait_event(e0)
        for _ in range(e2e_steps):
            e2e_step()
        for st in (s_up, s_comp, s_down):
            stream.wait_stream(st)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(torch, dist, e0.elapsed_time(e1) / e2e_steps, dev)

    t_gpu1 = time.time()
    time.sleep(0.1)
    clocks.stop()
    if rank != 0:
        return None

    step_bytes = sum(c["bytes"] for c in calls)
    ms_per_step = total_ms / args.steps
    value = job_gbs(step_bytes, world, ms_per_step)
    peak, peak_src = peak_hbm()
    per_op = {c["name"]: op_entry(c, ms) for c, ms in zip(calls, per_call_ms)}
    mean_ms = [t[0] for t in per_call_ms]
    dom = int(np.argmax(mean_ms))
    dom_c = calls[dom]
    achieved = dom_c["bytes"] / (mean_ms[dom] * 1e-3) / 1e9
    digest = buildlib.source_digest()
    family = "group" if dom_c["spec"]["op"] == "skip_group" else "rows"
    traffic = NCU_TRAFFIC.get((dom_c["name"], buildlib.source_digest(family)))
    launches = sum(launches_per_call(b2, c["spec"]) for c in calls) * args.steps
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": " + ".join(STEP_WORKLOADS),
            "bytes_per_step": step_bytes,
            "storage_types": "f16 / f32 tensors (fp32 arithmetic, one rounding at each store)",
            "l2": "inputs larger than L2: a step moves 1.42 GB against a 129 MB L2",
            "parallelism": f"replicas x{world}",
            "launch": "one CUDA graph per step (one call of each operator), replayed K times; "
                      "per-operator times from graphs of repeated calls over rotating buffers",
        },
        "per_op_bf16": ({"timing": "as per_op; bfloat16 storage, same shapes; not part of "
                                   "`value`", **bf16_ops} if bf16_ops else None),
        "per_op_short_rows": ({"timing": "as per_op; short rows, which take the pipelined "
                                          "bulk-copy schedule; not part of `value`",
                               **short_ops} if short_ops else None),
        "per_op_nhwc_mid": ({"timing": "as per_op; NHWC SkipGroupNorm with more pixels than "
                                       "the cooperative grid holds in registers (slabs in "
                                       "shared memory, bulk copies); not part of `value`",
                             **mid_ops} if mid_ops else None),
        "decode": ({"timing": f"best and median of {OP_MIN_ROUNDS} replays of a CUDA graph of "
                              "200 back-to-back calls on one buffer set (inputs L2-resident, as "
                              "when a preceding kernel has just written them); not part of "
                              "`value`",
                    **decode} if decode else None),
        "small": ({"timing": "as decode: the small batch is latency-bound (rows/s); not part "
                             "of `value`", **small} if small else None),
        "roofline": {"bound": "hbm", "kernel": dom_c["name"], "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": peak_src, "traffic": traffic,
                     "algorithmic_bytes_per_launch": dom_c["bytes"]},
        "e2e": ({"value": round(step_bytes * world / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                 "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                 "steps": e2e_steps, "ms_per_step": round(e2e_ms, 3)} if e2e_steps else None),
        "gpu_launches": launches,
        "clocks": clocks.summary(t_wall0, t_wall1),
        "clocks_all_timing": clocks.summary(t_wall0, t_gpu1),
        "source_digest": digest,
        "per_op_timing": (f"each step workload alone: a CUDA graph of 2 x sets (>= 8) calls "
                          f"cycling over `sets` input/output sets (>= 3 x L2 of other sets' "
                          f"traffic between two uses of one), replayed >= {OP_MIN_ROUNDS} times "
                          f"and >= {OP_MIN_LAUNCHES} calls with an event between replays; "
                          f"us_per_call = mean (the roofline's launch duration), median and "
                          f"best over the replays"),
        "per_op": per_op,
    }
    return line


# ---------------------------------------------------------------------------
# the CPU oracle (the baseline and the reference arm)
# ---------------------------------------------------------------------------
_WORKLOAD_CACHE = {}


def _workload(name):
    if name not in _WORKLOAD_CACHE:
        _WORKLOAD_CACHE[name] = synthetic.workload(name)
    return _WORKLOAD_CACHE[name]


def _parallel(fn, parts, threads):
    """Run fn(lo, hi) over `threads` contiguous slices of range(parts) (the C
    oracle releases the GIL) and return the wall time."""
    import concurrent.futures as cf
    k = max(1, min(threads, parts))
    bounds = [(parts * i // k, parts * (i + 1) // k) for i in range(k)]
    t0 = time.perf_counter()
    if k == 1:
        fn(0, parts)
    else:
        with cf.ThreadPoolExecutor(k) as ex:
            list(ex.map(lambda b: fn(*b), bounds))
    return time.perf_counter() - t0


def oracle_sample(fraction, threads=1):
    """Run the oracle on ``fraction`` of every step workload (leading rows /
    spans / batch items), split over ``threads`` host threads along that
    leading axis, and return (algorithmic bytes covered, seconds)."""
    import oracle
    total_bytes, total_s = 0.0, 0.0
    for name in STEP_WORKLOADS:
        spec, d = _workload(name)
        shape = spec["shape"]
        lead = max(1, int(round(shape[0] * fraction)))
        if spec["op"] == "skip_rms":
            rows = max(1, int(round(np.prod(shape[:-1]) * fraction)))
            x = d["input"].reshape(-1, shape[-1])
            sk = d["skip"].reshape(-1, shape[-1])
            total_s += _parallel(lambda lo, hi: oracle.skip_rms(
                x[lo:hi], sk[lo:hi], d["gamma"], d["bias"], epsilon=spec["epsilon"]), rows, threads)
            total_bytes += synthetic.algorithmic_bytes(name) * rows / np.prod(shape[:-1])
        elif spec["op"] == "gated_rms":
            spans = max(1, int(round(np.prod(shape) // spec["C"] * fraction)))
            x = d["x"].reshape(-1, spec["C"])
            g = d["gate"].reshape(-1, spec["C"])
            total_s += _parallel(lambda lo, hi: oracle.gated_rms(
                x[lo:hi], g[lo:hi], d["scale"], epsilon=spec["epsilon"]), spans, threads)
            total_bytes += synthetic.algorithmic_bytes(name) * spans / (np.prod(shape) // spec["C"])
        else:
            total_s += _parallel(lambda lo, hi: oracle.skip_group(
                d["x"][lo:hi], d["skip"][lo:hi], d["gamma"], d["beta"], d["bias"],
                groups=spec["groups"], activation=spec["activation"], epsilon=spec["epsilon"],
                channels_last=spec["channels_last"], want_sum=spec["want_sum"]), lead, threads)
            total_bytes += synthetic.algorithmic_bytes(name) * lead / shape[0]
    return total_bytes, total_s


def cpu_baseline(budget_s=15.0):
    b, s = oracle_sample(1 / 64)
    frac = min(1.0, (1 / 64) * budget_s / max(s, 1e-3))
    b, s = oracle_sample(frac)
    return {"value": round(b / s / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"leading {frac:.4f} of the rows / C-spans / batch items of each step "
                      f"workload, single-threaded C oracle ({s:.1f} s)"}


def cpu_baseline_all_cores():
    """The same oracle partitioned over every host core this process may use
    (rows, spans, or batch items; the results do not depend on the split)."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    b, s = oracle_sample(1.0, threads=cores)
    return {"value": round(b / s / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"every step workload, split over {cores} threads along the leading axis "
                      f"(SkipGroupNorm by batch item: 2 and 16 items) ({s:.1f} s)"}


def run_reference(args):
    """The oracle as the reference arm: each step is a bounded slice of the
    step workloads, sized so the whole run takes about a minute."""
    import oracle
    oracle.build()
    b, s = oracle_sample(1 / 256)
    per_step = 60.0 / max(1, args.steps + args.warmup)
    frac = min(1.0, (1 / 256) * per_step / max(s, 1e-4))
    for _ in range(args.warmup):
        oracle_sample(frac)
    tb, ts = 0.0, 0.0
    for _ in range(args.steps):
        bb, ss = oracle_sample(frac)
        tb += bb
        ts += ss
    value = tb / ts / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ts / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": " + ".join(STEP_WORKLOADS),
                       "sample_fraction_per_step": frac},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                             "kind": "oracle",
                             "sample": f"leading {frac:.6f} of each step workload per step"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer end-to-end leg (for profiler runs)")
    ap.add_argument("--no-bf16", action="store_true",
                    help="skip the bfloat16 per-operator measurements")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the decode-shaped latency measurements")
    ap.add_argument("--no-short", action="store_true",
                    help="skip the short-row (pipelined schedule) measurement")
    ap.add_argument("--no-mid", action="store_true",
                    help="skip the mid-size NHWC SkipGroupNorm measurement")
    ap.add_argument("--only", choices=STEP_WORKLOADS + BF16_WORKLOADS + DECODE_WORKLOADS +
                    SHORT_WORKLOADS + MID_WORKLOADS,
                    help="run a single workload (for profiler runs; not a bench line)")
    args = ap.parse_args()
    if args.only:
        STEP_WORKLOADS[:] = [args.only]
        args.no_bf16 = args.no_decode = args.no_short = args.no_mid = True
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    line = run_ours(args, rank, world, dist)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
            line["cpu_baseline_all_cores"] = cpu_baseline_all_cores()
        # the step workloads' per-operator figures last: a reader keeping only
        # the end of the line still has them
        for k in ("per_op_timing", "per_op"):
            if k in line:
                line[k] = line.pop(k)
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
