"""CPU oracle for the fused residual-add + normalization family.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The product
path (``residual_add_normalization_gb300``) never imports it, and this package
never imports the product: the two share nothing but the seeded input
generators, which hold none of the method's arithmetic.

The arithmetic lives in ``oracle.c`` (plain C, binary64 statistics, its own
IEEE binary16 conversion).  This module only compiles it with gcc and marshals
numpy arrays in and out through ctypes.

Operator definitions followed (web pages of the ``webgpu-kernels`` packages):
  * com.microsoft.SkipSimplifiedLayerNormalization README -- Description,
    Inputs, Outputs, Attributes.
  * com.microsoft.GatedRMSNorm README -- Description, Inputs, Attributes.
  * com.microsoft.SkipGroupNorm README -- Description, Inputs, Outputs,
    Attributes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, F16, BF16 = 0, 1, 2

# bfloat16 arrays are uint16 bit patterns whose dtype carries the metadata
# {"bfloat16": True} (numpy has no bfloat16 type).
BFLOAT16 = np.dtype(np.uint16, metadata={"bfloat16": True})


def is_bf16(dtype) -> bool:
    md = np.dtype(dtype).metadata
    return bool(md and md.get("bfloat16"))

# float32(1e-12): the SkipSimplifiedLayerNormalization epsilon default
# (README, Attributes).
SSLN_EPS_DEFAULT = 9.999999960041972e-13


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, no FMA
    contraction, no fast-math).  Returns the library path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB names an alternative build of oracle.c; the mutation
            # test uses it to check that the pins catch planted mistakes.
            path = os.environ.get("ORACLE_LIB") or build()
            lib = ctypes.CDLL(path)
            vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
            lib.orc_f64_to_f16.argtypes = [ctypes.c_double]
            lib.orc_f64_to_f16.restype = ctypes.c_uint16
            lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
            lib.orc_f32_to_f16.restype = ctypes.c_uint16
            lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_f16_to_f64.restype = ctypes.c_double
            lib.orc_f64_to_bf16.argtypes = [ctypes.c_double]
            lib.orc_f64_to_bf16.restype = ctypes.c_uint16
            lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_f64.restype = ctypes.c_double
            for name in ("orc_f64_to_f16_array", "orc_f32_to_f16_array",
                         "orc_f16_to_f32_array", "orc_f64_to_bf16_array",
                         "orc_f32_to_bf16_array", "orc_bf16_to_f32_array"):
                getattr(lib, name).argtypes = [vp, vp, i64]
                getattr(lib, name).restype = None
            lib.orc_skip_rms.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i32, f32]
            lib.orc_skip_rms.restype = i32
            lib.orc_gated_rms.argtypes = [vp, vp, vp, vp, i64, i64, i32, f32]
            lib.orc_gated_rms.restype = i32
            lib.orc_skip_group.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, i64, i64, i64,
                                           i64, i32, i32, i32, f32, i32, i32]
            lib.orc_skip_group.restype = i32
            _lib = lib
    return _lib


def _code(dtype) -> int:
    dt = np.dtype(dtype)
    if is_bf16(dt):
        return BF16
    if dt == np.float32:
        return F32
    if dt == np.float16:
        return F16
    raise TypeError(f"oracle supports float32, float16 and bfloat16 only, got {dt}")


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if dtype is not None and (a.dtype != dtype or is_bf16(a.dtype) != is_bf16(dtype)):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


# --------------------------------------------------------------------------
# IEEE binary16 conversions (written from the format definition in oracle.c)
# --------------------------------------------------------------------------

def f64_to_f16(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().orc_f64_to_f16_array(_ptr(a), _ptr(out), a.size)
    return out.view(np.float16)


def f32_to_f16(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().orc_f32_to_f16_array(_ptr(a), _ptr(out), a.size)
    return out.view(np.float16)


def f16_to_f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    bits = a.view(np.uint16) if a.dtype == np.float16 else a.astype(np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    _load().orc_f16_to_f32_array(_ptr(bits), _ptr(out), bits.size)
    return out


# --------------------------------------------------------------------------
# bfloat16 conversions (written from the format definition in oracle.c)
# --------------------------------------------------------------------------

def f64_to_bf16(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float64)
    out = np.empty(a.shape, dtype=BFLOAT16)
    _load().orc_f64_to_bf16_array(_ptr(a), _ptr(out), a.size)
    return out


def f32_to_bf16(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=BFLOAT16)
    _load().orc_f32_to_bf16_array(_ptr(a), _ptr(out), a.size)
    return out


def bf16_to_f32(a) -> np.ndarray:
    bits = np.ascontiguousarray(a).view(np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    _load().orc_bf16_to_f32_array(_ptr(bits), _ptr(out), bits.size)
    return out


# --------------------------------------------------------------------------
# Operators
# --------------------------------------------------------------------------

def skip_rms(input, skip, gamma, bias=None, epsilon=SSLN_EPS_DEFAULT,
             want_sum=True, want_stats=False):
    """SkipSimplifiedLayerNormalization over the last axis.

    Returns ``(output, input_skip_bias_sum or None)``, plus ``(mean, inv_std_var)``
    as float32 arrays of shape ``input.shape[:-1] + (1,)`` when ``want_stats``.
    """
    x = _c(input)
    code = _code(x.dtype)
    sk = _c(skip, x.dtype)
    ga = _c(gamma, x.dtype)
    bi = _c(bias, x.dtype)
    if sk.shape != x.shape:
        raise ValueError("skip must have the input's shape")
    hidden = x.shape[-1]
    rows = x.size // hidden if hidden else 0
    if ga.size != hidden or (bi is not None and bi.size != hidden):
        raise ValueError("gamma/bias must have hidden elements")
    y = np.empty_like(x)
    s = np.empty_like(x) if want_sum else None
    stat_shape = x.shape[:-1] + (1,)
    mean = np.empty(stat_shape, np.float32) if want_stats else None
    inv = np.empty(stat_shape, np.float32) if want_stats else None
    rc = _load().orc_skip_rms(_ptr(x), _ptr(sk), _ptr(ga), _ptr(bi), _ptr(y), _ptr(s),
                              _ptr(mean), _ptr(inv), rows, hidden, code, float(epsilon))
    if rc:
        raise ValueError(f"orc_skip_rms failed ({rc})")
    if want_stats:
        return y, s, mean, inv
    return y, s


def gated_rms(x, gate, scale, epsilon=1e-5):
    """GatedRMSNorm: per-C-span RMS norm times scale times SiLU(gate),
    C = scale.size."""
    xa = _c(x)
    code = _code(xa.dtype)
    ga = _c(gate, xa.dtype)
    sc = _c(scale, xa.dtype)
    if ga.shape != xa.shape:
        raise ValueError("gate must have X's shape")
    C = sc.size
    if C == 0 or xa.size % C:
        raise ValueError("numel(X) must be a multiple of numel(scale)")
    y = np.empty_like(xa)
    rc = _load().orc_gated_rms(_ptr(xa), _ptr(ga), _ptr(sc), _ptr(y), xa.size, C, code,
                               float(epsilon))
    if rc:
        raise ValueError(f"orc_gated_rms failed ({rc})")
    return y


def _skip_is_broadcast(x_shape, skip_shape, channels_last):
    """Classify skip per the SkipGroupNorm README, Inputs: either exactly X's
    shape (full), or (N, C) / (N, 1, 1, C) broadcast per (n, c).  A
    (N, 1, 1, C) skip at H = W = 1 is an exact match (full route)."""
    if channels_last:
        N, H, W, C = x_shape
    else:
        N, C, H, W = x_shape
    if tuple(skip_shape) == tuple(x_shape):
        return False
    if tuple(skip_shape) == (N, C):
        return True
    if tuple(skip_shape) == (N, 1, 1, C):
        return not (H == 1 and W == 1)
    raise ValueError(f"unsupported skip shape {skip_shape} for X {x_shape}")


def skip_group(x, skip, gamma, beta, bias=None, *, groups, activation,
               epsilon=1e-5, channels_last=1, want_sum=True):
    """SkipGroupNorm.  ``x`` is (N,H,W,C) if ``channels_last`` else (N,C,H,W).
    Returns ``(Y, S or None)``."""
    xa = _c(x)
    code = _code(xa.dtype)
    if xa.ndim != 4:
        raise ValueError("X must be rank 4")
    cl = 1 if channels_last else 0
    if cl:
        N, H, W, C = xa.shape
    else:
        N, C, H, W = xa.shape
    sk = _c(skip, xa.dtype)
    bcast = _skip_is_broadcast(xa.shape, sk.shape, cl)
    ga = _c(gamma)
    be = _c(beta, ga.dtype)
    mcode = _code(ga.dtype)
    bi = _c(bias, xa.dtype)
    if ga.size != C or be.size != C or (bi is not None and bi.size != C):
        raise ValueError("gamma/beta/bias must have C elements")
    y = np.empty_like(xa)
    s = np.empty_like(xa) if want_sum else None
    rc = _load().orc_skip_group(_ptr(xa), _ptr(sk), 1 if bcast else 0, _ptr(bi), _ptr(ga),
                                _ptr(be), _ptr(y), _ptr(s), N, C, H, W, code, mcode,
                                int(groups), float(epsilon), int(activation), cl)
    if rc:
        raise ValueError(f"orc_skip_group failed ({rc})")
    return y, s
