"""Build ``libb200norm.so`` in-tree from ``csrc/*.cu`` with nvcc for sm_103a.

Each translation unit is compiled in parallel into ``_build/`` and the objects
are linked into one shared library next to this file.  Only the C ABI declared
in ``include/b200norm.h`` (and the test hooks of ``include/b200norm_testing.h``)
is exported; the statically linked CUDA runtime stays internal.

    python -m residual_add_normalization_gb300.buildlib [--force]
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libb200norm.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libb200norm.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


# The sources each kernel family is built from (for digests that identify one
# family's code, e.g. to key profiler counters taken on it).
FAMILY_SOURCES = {
    "rows": ("common.cuh", "bulk.cuh", "launch.h", "rows.cuh", "rows_launch.cuh", "rows_ops.cuh",
             "rows_pipe.cuh", "rows_gated.cu", "rows_ssln_f16.cu", "rows_ssln_f32.cu", "rows_bf16.cu"),
    "group": ("common.cuh", "bulk.cuh", "launch.h", "group_kernels.cuh", "group_norm.cu",
              "group_f32.cu", "group_f16.cu", "group_bf16.cu"),
}


def _inputs_digest(family: str | None = None) -> str:
    h = hashlib.sha256()
    if family is None:
        files = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC))
        files += sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE))
    else:
        files = [os.path.join(CSRC, f) for f in FAMILY_SOURCES[family]]
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    # flags without the include paths, so the digest does not depend on where
    # the tree sits
    h.update(" ".join(ARCH + [f for f in NVCC_FLAGS if not f.startswith("-I")]).encode())
    return h.hexdigest()


def source_digest(family: str | None = None) -> str:
    """Digest of the kernel sources and headers (identifies a kernel build), or
    of one kernel family's sources ("rows", "group")."""
    return _inputs_digest(family)[:16]


def _compile(src: str) -> str:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if its inputs changed.  Returns its path."""
    stamp = os.path.join(BUILD, "digest")
    digest = _inputs_digest()
    if (not force and os.path.exists(LIB) and os.path.exists(stamp)
            and open(stamp).read().strip() == digest):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(_compile, srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-Xlinker", "--exclude-libs,ALL"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as fh:
        fh.write(digest)
    if verbose:
        print(f"built {LIB}")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
