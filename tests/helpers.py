"""Shared test helpers: the numeric bar and host<->device marshalling.

Tolerances (the stated bar): S bit-exact; float32 Y within
1e-5 + 1e-5 * |y_ref|; float16 Y within 2 units in the last place (ordinal
distance of the binary16 patterns) or 2e-3 absolute where |y_ref| < 1.  NaN
must meet NaN.  bfloat16 (a type the pages do not have) takes the float16 bar's
form: 2 units in the last place of bfloat16, or 2e-3 absolute where
|y_ref| < 1 (a quarter of one bfloat16 unit at 1).

bfloat16 host arrays are uint16 bit patterns with the BFLOAT16 dtype of the
input generators (numpy has no bfloat16).
"""
import numpy as np

from residual_add_normalization_gb300.synthetic import BFLOAT16, is_bf16

FP32_ABS = 1e-5
FP32_REL = 1e-5
FP16_ULPS = 2
FP16_ABS_SMALL = 2e-3


def _ordinal16(a):
    b = a.view(np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def values(a):
    """Float values of a float32 / float16 / bfloat16 host array, as float64."""
    if is_bf16(a.dtype):
        return (np.ascontiguousarray(a).view(np.uint16).astype(np.uint32) << 16) \
            .view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def y_mismatch(got, ref):
    """Boolean mask of elements of ``got`` outside the tolerance around ``ref``
    (both numpy arrays of the same float type)."""
    assert got.dtype == ref.dtype and got.shape == ref.shape
    assert is_bf16(got.dtype) == is_bf16(ref.dtype)
    g = values(got)
    r = values(ref)
    gnan, rnan = np.isnan(g), np.isnan(r)
    if got.dtype == np.float32:
        with np.errstate(invalid="ignore"):
            bad = ~(np.abs(g - r) <= FP32_ABS + FP32_REL * np.abs(r))
            bad &= ~(g == r)  # equal infinities
    else:
        d = np.abs(_ordinal16(got) - _ordinal16(ref))
        with np.errstate(invalid="ignore"):
            small = (np.abs(r) < 1.0) & (np.abs(g - r) <= FP16_ABS_SMALL)
        bad = ~((d <= FP16_ULPS) | small)
    return np.where(gnan | rnan, gnan != rnan, bad)


def _examples(bad, got, ref):
    idx = np.argwhere(bad)[:8]
    return ", ".join(f"{tuple(int(i) for i in k)}: got {got[tuple(k)]!r} ref {ref[tuple(k)]!r}"
                     for k in idx)


def assert_y_close(got, ref, what="Y"):
    bad = y_mismatch(got, ref)
    if bad.any():
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside "
                             f"tolerance; e.g. {_examples(bad, got, ref)}")


def assert_bitexact(got, ref, what="S"):
    assert got.dtype == ref.dtype and got.shape == ref.shape
    assert is_bf16(got.dtype) == is_bf16(ref.dtype)
    u = np.uint16 if got.dtype.itemsize == 2 else np.uint32
    bad = got.view(u) != ref.view(u)
    if bad.any():
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements differ; "
                             f"e.g. {_examples(bad, got, ref)}")


def to_dev(a, device="cuda"):
    import torch
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if is_bf16(a.dtype):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def to_host(t):
    import torch
    if t is None:
        return None
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).view(BFLOAT16)
    return t.numpy()
