"""Fused residual-add + normalization on NVIDIA GB300 (sm_103a).

Thin Python binding over the C ABI of ``libb200norm.so`` (``include/b200norm.h``).
It only marshals arguments: checks that tensors are contiguous CUDA tensors of
matching shapes and types, allocates outputs with torch, and passes raw device
pointers and the current CUDA stream.  Every step of every operator runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback -- a missing or
unloadable library raises.

Operators (ONNX Runtime contrib operators, as the webgpu-kernels README pages
describe them):

  skip_rms        com.microsoft.SkipSimplifiedLayerNormalization
  skip_rms_stats  the same, plus the per-row mean / inv_std_var outputs
  gated_rms       com.microsoft.GatedRMSNorm
  skip_group      com.microsoft.SkipGroupNorm
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["skip_rms", "skip_rms_stats", "gated_rms", "skip_group", "workspace_size",
           "workspace_init", "workspace_status", "noalloc_status", "rows_status", "library",
           "library_path", "B200NormError", "SSLN_EPS_DEFAULT"]

# float32(1e-12): SkipSimplifiedLayerNormalization README, Attributes, epsilon.
SSLN_EPS_DEFAULT = 9.999999960041972e-13

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libb200norm.so")
_lock = threading.Lock()
_lib = None

_DTYPES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}


class B200NormError(RuntimeError):
    """A b200norm call returned a non-OK status."""

    def __init__(self, status: int, name: str, detail: str):
        super().__init__(f"{name}: {detail}" if detail else name)
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def library() -> ctypes.CDLL:
    """The loaded C library (loaded on first use; raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is not built; run `python -m residual_add_normalization_gb300.buildlib`"
                " (needs nvcc) -- there is no fallback implementation")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                 ctypes.c_size_t)
        sig = {
            "b200norm_version": ([], i32),
            "b200norm_status_string": ([i32], ctypes.c_char_p),
            "b200norm_last_error": ([], ctypes.c_char_p),
            "b200norm_skip_rms": ([vp, vp, vp, vp, vp, vp, i64, i64, i32, f32, vp], i32),
            "b200norm_skip_rms_stats": ([vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i32, f32, vp],
                                        i32),
            "b200norm_gated_rms": ([vp, vp, vp, vp, i64, i64, i32, f32, vp], i32),
            "b200norm_skip_group_workspace_size": ([i64, i64, i64, i64, i32, i32, i32], sz),
            "b200norm_skip_group": ([vp, vp, i32, ctypes.POINTER(ctypes.c_int64), vp, vp, vp,
                                     vp, vp, i64, i64, i64, i64, i32, i32, i32, f32, i32, i32,
                                     vp, sz, vp], i32),
            "b200norm_skip_group_noalloc": ([vp, vp, i32, ctypes.POINTER(ctypes.c_int64), vp,
                                             vp, vp, vp, vp, i64, i64, i64, i64, i32, i32, i32,
                                             f32, i32, i32, vp], i32),
            "b200norm_skip_group_noalloc_status": ([vp], i32),
            "b200norm_workspace_init": ([vp, sz, vp], i32),
            "b200norm_workspace_status": ([vp, vp], i32),
            "b200norm_rows_status": ([vp], i32),
            "b200norm_testing_barrier_timeout": ([vp, sz, ctypes.c_uint64, vp], i32),
            "b200norm_testing_noalloc_barrier_timeout": ([ctypes.c_uint64, vp], i32),
            "b200norm_testing_force": ([i32, i32], i32),
            "b200norm_testing_force_split": ([i32, i32], i32),
            "b200norm_testing_set_pdl": ([i32], i32),
            "b200norm_testing_pipe_stall": ([i32, ctypes.c_uint64], i32),
            "b200norm_testing_plan_rows": ([i64, i64, i32, i32, ctypes.POINTER(ctypes.c_int64)],
                                           i32),
            "b200norm_testing_plan_gated": ([i64, i64, i32, i32, ctypes.POINTER(ctypes.c_int64)],
                                            i32),
            "b200norm_testing_plan_group": ([i64, i64, i64, i64, i32, i32, i32, i32, i32,
                                             ctypes.POINTER(ctypes.c_int64)], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(status: int) -> None:
    if status != 0:
        lib = library()
        name = lib.b200norm_status_string(status).decode()
        detail = lib.b200norm_last_error().decode()
        raise B200NormError(status, name, detail)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _torch_stream(device, stream):
    return stream if stream is not None else torch.cuda.current_stream(device)


def _stream(device, stream):
    return ctypes.c_void_p(_torch_stream(device, stream).cuda_stream)


def _cuda(name, t, device=None, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device}); there is no CPU path")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if t.dtype not in _DTYPES:
        raise TypeError(f"{name}: only float32, float16 and bfloat16 are supported "
                        f"(got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _out(name, t, like, dtype=None):
    if t is None:
        return torch.empty(like.shape, dtype=dtype or like.dtype, device=like.device)
    _cuda(name, t, like.device, dtype or like.dtype)
    if t.numel() != like.numel():
        raise ValueError(f"{name} must have {like.numel()} elements")
    return t


# ---------------------------------------------------------------------------
# SkipSimplifiedLayerNormalization
# ---------------------------------------------------------------------------

def _skip_rms(input, skip, gamma, bias, epsilon, want_sum, output, sum_out, stats, stream):
    x = _cuda("input", input)
    dev, dt = x.device, x.dtype
    _cuda("skip", skip, dev, dt)
    _cuda("gamma", gamma, dev, dt)
    if bias is not None:
        _cuda("bias", bias, dev, dt)
    if x.dim() < 1 or skip.shape != x.shape:
        raise ValueError("skip must have input's shape")
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    if gamma.numel() != hidden or (bias is not None and bias.numel() != hidden):
        raise ValueError("gamma and bias must have hidden_size elements")
    y = _out("output", output, x)
    s = _out("input_skip_bias_sum", sum_out, x) if want_sum or sum_out is not None else None
    st = _stream(dev, stream)
    lib = library()
    if stats:
        stat_shape = tuple(x.shape[:-1]) + (1,)
        mean = torch.empty(stat_shape, dtype=torch.float32, device=dev)
        inv = torch.empty(stat_shape, dtype=torch.float32, device=dev)
        _check(lib.b200norm_skip_rms_stats(_ptr(x), _ptr(skip), _ptr(gamma), _ptr(bias), _ptr(y),
                                           _ptr(s), _ptr(mean), _ptr(inv), rows, hidden,
                                           _DTYPES[dt], float(epsilon), st))
        return y, s, mean, inv
    _check(lib.b200norm_skip_rms(_ptr(x), _ptr(skip), _ptr(gamma), _ptr(bias), _ptr(y), _ptr(s),
                                 rows, hidden, _DTYPES[dt], float(epsilon), st))
    return y, s


def skip_rms(input, skip, gamma, bias=None, *, epsilon=SSLN_EPS_DEFAULT, want_sum=True,
             output=None, sum_out=None, stream=None):
    """SkipSimplifiedLayerNormalization over the last axis of ``input``.

    Returns ``(output, input_skip_bias_sum)``; the second is ``None`` unless
    ``want_sum`` (default True) or ``sum_out`` is given.
    """
    return _skip_rms(input, skip, gamma, bias, epsilon, want_sum, output, sum_out, False, stream)


def skip_rms_stats(input, skip, gamma, bias=None, *, epsilon=SSLN_EPS_DEFAULT, want_sum=True,
                   output=None, sum_out=None, stream=None):
    """As :func:`skip_rms`, also returning the float32 ``mean`` (zeros) and
    ``inv_std_var`` outputs of shape ``input.shape[:-1] + (1,)``."""
    return _skip_rms(input, skip, gamma, bias, epsilon, want_sum, output, sum_out, True, stream)


# ---------------------------------------------------------------------------
# GatedRMSNorm
# ---------------------------------------------------------------------------

def gated_rms(x, gate, scale, *, epsilon=1e-5, y=None, stream=None):
    """GatedRMSNorm: RMS-normalize each contiguous span of ``C = scale.numel()``
    elements of ``x``, times ``scale`` times SiLU(``gate``)."""
    x = _cuda("X", x)
    _cuda("gate", gate, x.device, x.dtype)
    _cuda("scale", scale, x.device, x.dtype)
    if gate.shape != x.shape:
        raise ValueError("gate must have X's shape")
    if x.dim() < 1:
        raise ValueError("X must have rank >= 1")
    C = scale.numel()
    out = _out("Y", y, x)
    _check(library().b200norm_gated_rms(_ptr(x), _ptr(gate), _ptr(scale), _ptr(out), x.numel(),
                                        C, _DTYPES[x.dtype], float(epsilon),
                                        _stream(x.device, stream)))
    return out


# ---------------------------------------------------------------------------
# SkipGroupNorm
# ---------------------------------------------------------------------------

_workspaces = {}
_ws_lock = threading.Lock()


def rows_status(stream=None, device=None):
    """Synchronizes ``stream`` and raises B200NormError if a pipelined row
    kernel (short SkipSimplifiedLayerNormalization / GatedRMSNorm rows) on the
    device gave up a bounded wait since the last call; the record is then
    cleared."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        _check(library().b200norm_rows_status(_stream(dev, stream)))


def noalloc_status(stream=None, device=None):
    """Synchronizes ``stream`` and raises B200NormError if a bounded
    device-side wait of an allocation-free SkipGroupNorm call
    (``b200norm_skip_group_noalloc``) on the device gave up since the last
    call; the record is then cleared."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        _check(library().b200norm_skip_group_noalloc_status(_stream(dev, stream)))


def workspace_size(N, C, H, W, groups, dtype=torch.float16, channels_last=1) -> int:
    return int(library().b200norm_skip_group_workspace_size(N, C, H, W, groups, _DTYPES[dtype],
                                                            1 if channels_last else 0))


def workspace_init(ws, stream=None):
    _check(library().b200norm_workspace_init(_ptr(ws), ws.numel(), _stream(ws.device, stream)))


def workspace_status(ws, stream=None):
    """Synchronizes ``stream`` and raises B200NormError if a device-side wait
    recorded a timeout in ``ws``."""
    _check(library().b200norm_workspace_status(_ptr(ws), _stream(ws.device, stream)))


def _workspace_for(device, stream, nbytes):
    """A zero-filled workspace cached per (device, stream); calls on one
    stream are serialized, so they may share it.  It is allocated and zeroed
    on that stream, so the clear is ordered before the kernels that use it,
    and a smaller one it replaces goes back to the caching allocator on the
    stream its kernels ran on (its allocation stream)."""
    key = (device.index, stream.cuda_stream)
    with _ws_lock:
        ws = _workspaces.get(key)
        if ws is None or ws.numel() < nbytes:
            with torch.cuda.stream(stream):
                ws = torch.zeros(max(nbytes, 1 << 16), dtype=torch.uint8, device=device)
            _workspaces[key] = ws
        return ws


def skip_group(x, skip, gamma, beta, bias=None, *, groups, activation, epsilon=1e-5,
               channels_last=1, want_sum=False, y=None, s=None, workspace=None, stream=None):
    """SkipGroupNorm.  ``x`` is (N, H, W, C) when ``channels_last`` is non-zero
    (the default), else (N, C, H, W).  ``skip`` is x's shape, (N, C) or
    (N, 1, 1, C).  ``groups`` and ``activation`` (0 none, 1 SiLU) are required.
    Returns ``(Y, S)``; ``S`` is ``None`` unless ``want_sum`` or ``s`` is given.
    """
    x = _cuda("X", x)
    dev, dt = x.device, x.dtype
    if x.dim() != 4:
        raise ValueError("X must be rank 4")
    _cuda("skip", skip, dev, dt)
    _cuda("gamma", gamma, dev)
    _cuda("beta", beta, dev, gamma.dtype)
    if bias is not None:
        _cuda("bias", bias, dev, dt)
    cl = 1 if channels_last else 0
    if cl:
        N, H, W, C = x.shape
    else:
        N, C, H, W = x.shape
    if gamma.numel() != C or beta.numel() != C or (bias is not None and bias.numel() != C):
        raise ValueError("gamma, beta and bias must have C elements")
    out = _out("Y", y, x)
    ssum = _out("S", s, x) if want_sum or s is not None else None
    tst = _torch_stream(dev, stream)
    st = ctypes.c_void_p(tst.cuda_stream)
    nbytes = workspace_size(N, C, H, W, groups, dt, cl)
    if workspace is None:
        workspace = _workspace_for(dev, tst, nbytes)
    if skip.dim() > 4:
        raise ValueError("skip must have X's shape, (N, C) or (N, 1, 1, C)")
    dims = (ctypes.c_int64 * 4)(*([int(d) for d in skip.shape] + [0] * (4 - skip.dim())))
    _check(library().b200norm_skip_group(
        _ptr(x), _ptr(skip), skip.dim(), dims, _ptr(bias), _ptr(gamma), _ptr(beta), _ptr(out),
        _ptr(ssum), N, C, H, W, _DTYPES[dt], _DTYPES[gamma.dtype], int(groups), float(epsilon),
        int(activation), cl, _ptr(workspace), workspace.numel(), st))
    return out, ssum
