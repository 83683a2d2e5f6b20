"""The C ABI from a plain C program (tests/c/abi_example.c): compiled against
include/b200norm.h and linked to the in-tree libb200norm.so, with no Python in
the call path.  The CPU test runs the argument-error paths; the GPU test also
runs every operator on a closed-form case on the README usage examples'
shapes: SkipSimplifiedLayerNormalization, GatedRMSNorm with C = 1, and
SkipGroupNorm through a workspace sized by
b200norm_skip_group_workspace_size() and through the allocation-free entry."""
import os
import shutil
import subprocess

import pytest

import residual_add_normalization_gb300 as b2

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_example.c")


def _build(tmp_path, gpu):
    libdir = os.path.dirname(b2.library_path())
    exe = str(tmp_path / ("abi_example_gpu" if gpu else "abi_example"))
    if gpu:
        nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
        cmd = [nvcc, "-x", "c", "-DB200NORM_EXAMPLE_GPU", f"-I{ROOT}/include", SRC, "-o", exe,
               f"-L{libdir}", "-lb200norm", f"-Xlinker=-rpath,{libdir}", "-lcudart", "-lm"]
    else:
        cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", f"-I{ROOT}/include", SRC, "-o",
               exe, f"-L{libdir}", "-lb200norm", f"-Wl,-rpath,{libdir}", "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_caller_argument_errors(tmp_path):
    b2.library()  # builds/loads the in-tree library
    exe = _build(tmp_path, gpu=False)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"


@pytest.mark.gpu
def test_c_caller_runs_every_operator(tmp_path):
    b2.library()
    exe = _build(tmp_path, gpu=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "ok"
