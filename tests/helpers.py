"""Shared test helpers: the numeric bar and host<->device marshalling.

Tolerances (the stated bar): S bit-exact; float32 Y within
1e-5 + 1e-5 * |y_ref|; float16 Y within 2 units in the last place (ordinal
distance of the binary16 patterns) or 2e-3 absolute where |y_ref| < 1.  NaN
must meet NaN.
"""
import numpy as np

FP32_ABS = 1e-5
FP32_REL = 1e-5
FP16_ULPS = 2
FP16_ABS_SMALL = 2e-3


def _ordinal16(a):
    b = a.view(np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def y_mismatch(got, ref):
    """Boolean mask of elements of ``got`` outside the tolerance around ``ref``
    (both numpy arrays of the same float type)."""
    assert got.dtype == ref.dtype and got.shape == ref.shape
    gnan, rnan = np.isnan(got), np.isnan(ref)
    g = got.astype(np.float64)
    r = ref.astype(np.float64)
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
    u = np.uint16 if got.dtype == np.float16 else np.uint32
    bad = got.view(u) != ref.view(u)
    if bad.any():
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements differ; "
                             f"e.g. {_examples(bad, got, ref)}")


def to_dev(a, device="cuda"):
    import torch
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host(t):
    return None if t is None else t.detach().cpu().numpy()
