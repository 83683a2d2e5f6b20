"""The C ABI library: it loads, exports every function the public headers
declare, and rejects bad arguments before touching a GPU.

These run without a GPU: argument validation happens on the host before any
CUDA call, and the planner for row schedules is pure host logic.
"""
import ctypes
import os
import re
import subprocess

import pytest

import residual_add_normalization_gb300 as b2
from residual_add_normalization_gb300 import buildlib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("b200norm.h", "b200norm_testing.h")]

OK, INVALID, UNSUPPORTED, CUDA, WORKSPACE, TIMEOUT = range(6)
F32, F16 = 0, 1
SSLN_EPS = 9.999999960041972e-13


@pytest.fixture(scope="module")
def lib():
    buildlib.build()
    return b2.library()


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        names += re.findall(r"B200NORM_API\s+[\w\s\*]*?\b(b200norm_\w+)\s*\(", text)
    return names


def test_headers_declare_the_boundary():
    names = set(declared_functions())
    for required in ("b200norm_skip_rms", "b200norm_gated_rms", "b200norm_skip_group",
                     "b200norm_skip_group_workspace_size", "b200norm_workspace_status",
                     "b200norm_status_string", "b200norm_version"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_only_the_abi_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", buildlib.LIB], capture_output=True,
                         text=True, check=True).stdout.splitlines()
    exported = {ln.split()[-1] for ln in out if " T " in ln}
    assert exported == set(declared_functions())


def test_version_and_status_strings(lib):
    assert lib.b200norm_version() == 1
    assert lib.b200norm_status_string(OK) == b"B200NORM_OK"
    assert lib.b200norm_status_string(TIMEOUT) == b"B200NORM_ERR_DEVICE_TIMEOUT"
    assert lib.b200norm_status_string(77) == b"B200NORM_UNKNOWN_STATUS"


FAKE = 1 << 40  # never dereferenced: every call below fails validation first


def ssln(lib, **kw):
    a = dict(input=FAKE, skip=FAKE + (1 << 30), gamma=FAKE + (2 << 30), bias=None,
             output=FAKE + (3 << 30), s=None, rows=4, hidden=64, T=F16, eps=SSLN_EPS)
    a.update(kw)
    return lib.b200norm_skip_rms(a["input"], a["skip"], a["gamma"], a["bias"], a["output"],
                                 a["s"], a["rows"], a["hidden"], a["T"], a["eps"], None)


def test_skip_rms_validation(lib):
    assert ssln(lib, T=3) == UNSUPPORTED                    # no such element type
    assert ssln(lib, rows=-1) == INVALID
    assert ssln(lib, hidden=0) == INVALID
    assert ssln(lib, eps=-1.0) == INVALID                   # epsilon is non-negative
    assert ssln(lib, eps=float("nan")) == INVALID
    assert ssln(lib, rows=0, input=None, skip=None, gamma=None, output=None) == OK  # empty
    assert ssln(lib, gamma=None) == INVALID
    assert ssln(lib, input=FAKE + 1) == INVALID              # not element-aligned
    assert ssln(lib, output=FAKE) == INVALID                 # output aliases input
    assert ssln(lib, s=FAKE + (3 << 30) + 64) == INVALID      # S overlaps output
    assert b"overlap" in lib.b200norm_last_error()
    assert ssln(lib, hidden=1 << 31) == UNSUPPORTED


def test_gated_validation(lib):
    def call(**kw):
        a = dict(x=FAKE, gate=FAKE + (1 << 30), scale=FAKE + (2 << 30), y=FAKE + (3 << 30),
                 numel=12, C=4, T=F32, eps=1e-5)
        a.update(kw)
        return lib.b200norm_gated_rms(a["x"], a["gate"], a["scale"], a["y"], a["numel"], a["C"],
                                      a["T"], a["eps"], None)
    assert call(C=5) == INVALID          # numel not a multiple of C
    assert call(C=0) == INVALID
    assert call(numel=-4) == INVALID
    assert call(eps=-1e-3) == INVALID
    assert call(T=5) == UNSUPPORTED
    assert call(numel=0, x=None, gate=None, scale=None, y=None) == OK
    assert call(y=FAKE + 8) == INVALID   # overlaps x


def sgn(lib, **kw):
    a = dict(x=FAKE, skip=FAKE + (1 << 30), rank=2, dims=(2, 8, 0, 0), bias=None,
             gamma=FAKE + (2 << 30), beta=FAKE + (2 << 30) + 4096, y=FAKE + (3 << 30), s=None,
             N=2, C=8, H=3, W=2, T=F16, M=F32, groups=2, eps=1e-5, act=0, cl=1,
             ws=FAKE + (4 << 30), wsb=1 << 20)
    a.update(kw)
    dims = (ctypes.c_int64 * 4)(*a["dims"])
    return lib.b200norm_skip_group(a["x"], a["skip"], a["rank"], dims, a["bias"], a["gamma"],
                                   a["beta"], a["y"], a["s"], a["N"], a["C"], a["H"], a["W"],
                                   a["T"], a["M"], a["groups"], a["eps"], a["act"], a["cl"],
                                   a["ws"], a["wsb"], None)


def test_skip_group_validation(lib):
    assert sgn(lib, groups=3) == INVALID            # groups must divide C
    assert sgn(lib, groups=0) == INVALID
    assert sgn(lib, act=2) == INVALID               # activation is 0 or 1
    assert sgn(lib, act=-1) == INVALID
    assert sgn(lib, eps=-1.0) == INVALID
    assert sgn(lib, M=2) == UNSUPPORTED             # bfloat16 gamma under float16 X
    assert sgn(lib, T=2, M=1) == UNSUPPORTED        # float16 gamma under bfloat16 X
    assert sgn(lib, T=0, M=2) == UNSUPPORTED
    assert sgn(lib, T=3, M=0) == UNSUPPORTED
    assert sgn(lib, rank=2, dims=(2, 4, 0, 0)) == INVALID          # skip (N, C') wrong
    assert sgn(lib, rank=3, dims=(2, 1, 8, 0)) == INVALID
    assert sgn(lib, rank=4, dims=(2, 3, 2, 4)) == INVALID          # not X's shape
    assert sgn(lib, ws=None) == WORKSPACE
    assert sgn(lib, wsb=100) == WORKSPACE
    assert sgn(lib, ws=FAKE + (4 << 30) + 16) == WORKSPACE         # not 256-byte aligned
    assert sgn(lib, y=FAKE + 2) == INVALID                         # aliases X
    assert sgn(lib, N=0, dims=(0, 8, 0, 0), x=None, skip=None, y=None, ws=None) == OK  # empty
    assert sgn(lib, beta=None) == INVALID


def test_workspace_size_covers_every_route(lib):
    # the workspace holds a control block plus one 16-byte slot per piece of
    # the largest route the layout can take
    small = lib.b200norm_skip_group_workspace_size(2, 320, 64, 64, 32, F16, 1)
    assert small >= 256 + 16 * 32
    big = lib.b200norm_skip_group_workspace_size(1, 64, 1024, 1024, 1, F16, 0)
    assert big >= 256 + 16 * ((64 * 1024 * 1024 + 4095) // 4096)


def test_workspace_size_follows_the_layout(lib):
    # NCHW calls run the resident route (no slots) or the two-phase route
    # (one slot per 4,096-element chunk of every group instance); NHWC calls
    # can also take the cooperative and L2 routes (up to 2,048 CTAs' pieces
    # per group, and the L2 route's statistics)
    nchw = lib.b200norm_skip_group_workspace_size(16, 1280, 16, 16, 32, F32, 0)
    assert nchw == 256 + 16 * (16 * 32 * 3)
    nhwc = lib.b200norm_skip_group_workspace_size(16, 1280, 16, 16, 32, F32, 1)
    assert nhwc >= 256 + 16 * 2048 * 32
    # any non-zero channels_last means NHWC
    assert lib.b200norm_skip_group_workspace_size(16, 1280, 16, 16, 32, F32, 7) == nhwc


def noalloc(lib, **kw):
    a = dict(x=FAKE, skip=FAKE + (1 << 30), rank=2, dims=(2, 8, 0, 0), bias=None,
             gamma=FAKE + (2 << 30), beta=FAKE + (2 << 30) + 4096, y=FAKE + (3 << 30), s=None,
             N=2, C=8, H=3, W=2, T=F16, M=F32, groups=2, eps=1e-5, act=0, cl=1)
    a.update(kw)
    dims = (ctypes.c_int64 * 4)(*a["dims"])
    return lib.b200norm_skip_group_noalloc(a["x"], a["skip"], a["rank"], dims, a["bias"],
                                           a["gamma"], a["beta"], a["y"], a["s"], a["N"], a["C"],
                                           a["H"], a["W"], a["T"], a["M"], a["groups"], a["eps"],
                                           a["act"], a["cl"], None)


def test_noalloc_refuses_before_touching_a_device(lib):
    """The allocation-free entry makes the regular entry's argument checks
    and its own size check before any CUDA call (none of these reach a GPU)."""
    assert noalloc(lib, groups=3) == INVALID
    assert noalloc(lib, act=2) == INVALID
    assert noalloc(lib, eps=float("nan")) == INVALID
    assert noalloc(lib, M=2) == UNSUPPORTED
    assert noalloc(lib, rank=4, dims=(2, 3, 2, 4)) == INVALID
    assert noalloc(lib, y=FAKE + 2) == INVALID                      # aliases X
    assert noalloc(lib, y=None) == INVALID
    assert noalloc(lib, N=0, dims=(0, 8, 0, 0), x=None, skip=None, y=None) == OK  # empty
    # 64 groups of a small NHWC shape the L2 route could take: more slots than
    # the 256 + 2 MiB scratch holds
    dims64 = (2, 64, 0, 0)
    assert noalloc(lib, C=64, H=8, W=8, groups=64, dims=dims64, cl=1) == UNSUPPORTED
    assert b"static scratch" in lib.b200norm_last_error()
    assert lib.b200norm_skip_group_workspace_size(2, 64, 8, 8, 64, F16, 1) > 256 + (2 << 20)


def plan_rows(lib, rows, n, T, aligned=1, gated=False):
    out = (ctypes.c_int64 * 8)()
    fn = lib.b200norm_testing_plan_gated if gated else lib.b200norm_testing_plan_rows
    assert fn(rows, n, T, aligned, out) == OK
    return dict(zip(("mode", "ve", "tpr", "nv", "rpg", "block", "csize", "grid"), out))


def test_row_planner_shapes(lib):
    # GatedRMSNorm C = 128 fp16: 16 vectors of 8 -> 16-lane groups, 2 spans per warp
    p = plan_rows(lib, 1 << 20, 128, F16, gated=True)
    assert (p["mode"], p["ve"], p["tpr"]) == (0, 8, 16)
    assert p["grid"] * (p["block"] // p["tpr"]) * p["rpg"] >= 1 << 20
    # SSLN hidden 4096 fp16: CTA per row, every vector covered
    p = plan_rows(lib, 16384, 4096, F16)
    assert p["mode"] == 1 and p["csize"] == 1 and p["tpr"] * p["nv"] * p["ve"] >= 4096
    # few rows (latency-bound): the widest CTA, fewest vectors per thread;
    # many rows: CTAs of about 256 threads
    assert (plan_rows(lib, 1, 4096, F16)["nv"], plan_rows(lib, 1, 4096, F16)["block"]) == (1, 512)
    assert (plan_rows(lib, 64, 8192, F16)["nv"], plan_rows(lib, 64, 8192, F16)["block"]) == (2, 512)
    assert (plan_rows(lib, 16384, 4096, F16)["nv"], plan_rows(lib, 16384, 4096, F16)["block"]) == (2, 256)
    assert (plan_rows(lib, 16384, 4096, F32)["nv"], plan_rows(lib, 16384, 4096, F32)["block"]) == (4, 256)
    assert (plan_rows(lib, 16384, 8192, F32)["nv"], plan_rows(lib, 16384, 8192, F32)["block"]) == (4, 512)
    # many rows (measured): SSLN rows of 97-159 vectors on a CTA each, two
    # vectors per thread unless the row is a whole number of warps; GatedRMSNorm
    # CTA rows with at least two vectors per thread, rows of up to 128 vectors
    # on a warp each
    for n, T, want in ((768, F16, (0, 4)), (896, F16, (1, 2)), (1024, F16, (1, 1)),
                       (1152, F16, (1, 2)), (1280, F16, (1, 1)), (512, F32, (1, 1)),
                       (448, F32, (1, 1)), (576, F32, (1, 1))):
        p = plan_rows(lib, 65536, n, T)
        assert (p["mode"], p["nv"]) == want, (n, T, p)
    # ... two vectors per thread only from 8,192 rows; 16-bit SSLN rows of 1,024
    # vectors in 512-thread CTAs (float32 keeps 256 threads of four)
    assert plan_rows(lib, 4096, 1152, F16)["nv"] == 1
    assert plan_rows(lib, 4096, 2048, F16, gated=True)["nv"] == 1
    assert (plan_rows(lib, 4096, 8192, F16)["nv"], plan_rows(lib, 4096, 8192, F16)["block"]) == (2, 512)
    assert (plan_rows(lib, 4096, 4096, F32)["nv"], plan_rows(lib, 4096, 4096, F32)["block"]) == (4, 256)
    for n, T, want in ((1024, F16, (0, 4)), (1536, F16, (1, 2)), (2048, F16, (1, 2)),
                       (8192, F16, (1, 4)), (1024, F32, (1, 2))):
        p = plan_rows(lib, 65536, n, T, gated=True)
        assert (p["mode"], p["nv"]) == want, (n, T, p)
    # ... but few rows keep the latency-bound choice (the widest CTA up to 512 rows)
    assert plan_rows(lib, 64, 1024, F16)["mode"] == 0
    assert plan_rows(lib, 64, 2048, F16, gated=True)["nv"] == 1
    assert (plan_rows(lib, 512, 4096, F16)["nv"], plan_rows(lib, 512, 4096, F16)["block"]) == (1, 512)
    # odd hidden: scalar path
    p = plan_rows(lib, 3, 5, F32)
    assert p["ve"] == 1 and p["tpr"] >= 5
    # unaligned pointers force the scalar path
    assert plan_rows(lib, 8, 4096, F16, aligned=0)["ve"] == 1
    # long rows go to a cluster, then to the walking schedule
    p = plan_rows(lib, 2, 65536, F16)
    assert p["mode"] == 1 and p["csize"] >= 2 and p["tpr"] * p["nv"] * p["ve"] >= 65536
    assert plan_rows(lib, 1, 1 << 24, F16)["mode"] == 2
    # every plan covers the row
    for n, rows, gated in [(n, r, g) for n in (1, 3, 8, 24, 100, 256, 257, 768, 896, 1000, 1152,
                                                4096, 12288, 40000, 300000)
                           for r in (5, 65536) for g in (False, True)]:
        for T in (F32, F16):
            for al in (0, 1):
                p = plan_rows(lib, rows, n, T, al, gated)
                nvec = n // p["ve"]
                assert n % p["ve"] == 0
                if p["mode"] != 2:
                    assert p["tpr"] * p["nv"] >= nvec, (n, T, al, p)
                    assert p["block"] <= 1024 and p["block"] % 32 == 0
                if p["mode"] == 0:
                    assert p["tpr"] & (p["tpr"] - 1) == 0 and p["block"] % p["tpr"] == 0


def test_force_hook_validation(lib):
    assert lib.b200norm_testing_force(-1, 0) == INVALID
    assert lib.b200norm_testing_force(1, 0) == OK
    assert lib.b200norm_testing_force(0, 1) == INVALID
    assert lib.b200norm_testing_force(0, 6) == OK
    assert lib.b200norm_testing_force(0, 7) == INVALID
    assert lib.b200norm_testing_force(0, 5) == OK
    assert lib.b200norm_testing_force(0, 0) == OK
    assert lib.b200norm_testing_force(4, 0) == INVALID
    assert lib.b200norm_testing_force(3, 0) == OK
    assert lib.b200norm_testing_force(0, 0) == OK
    assert lib.b200norm_testing_pipe_stall(2, 1000) == INVALID
    assert lib.b200norm_testing_pipe_stall(1, 0) == INVALID
    assert lib.b200norm_testing_pipe_stall(1, 6_000_000_000) == INVALID
    assert lib.b200norm_testing_pipe_stall(0, 0) == OK
    for bad in ((3, 1), (2, 3), (0, 1), (32, 1), (1, 16)):
        assert lib.b200norm_testing_force_split(*bad) == INVALID, bad
    assert lib.b200norm_testing_force_split(16, 8) == OK
    assert lib.b200norm_testing_force_split(0, 0) == OK
    assert lib.b200norm_testing_set_pdl(2) == INVALID
    assert lib.b200norm_testing_set_pdl(1) == OK


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, 8)
    with pytest.raises(ValueError, match="CUDA"):
        b2.skip_rms(x, x, torch.ones(8))
    with pytest.raises(ValueError, match="CUDA"):
        b2.gated_rms(x, x, torch.ones(8))
