"""Seeded synthetic inputs for the five reference workloads and for tests.

This module only draws random numbers (numpy ``default_rng``) and casts them to
the tensor types; it holds none of the operators' arithmetic.  The same host
arrays feed the CPU oracle and the CUDA path, so both see identical bits.

Workloads (shapes, distributions and attributes of the operators' typical
uses named on the pages: LLM residual stream, Mamba2 per-head gated norm,
diffusion-UNet group norm).  ``N(m, s)`` means mean ``m`` and standard
deviation ``s``.

  ssln_fp32_64x768     SkipSimplifiedLayerNormalization fp32, input/skip
                       (64, 768) N(0,1), bias N(0,0.1), gamma U(0.5,1.5),
                       eps float32(1e-12), S requested; seed 0.
  ssln_fp16_8x2048x4096  SkipSimplifiedLayerNormalization fp16, input/skip
                       (8, 2048, 4096) N(0,1), bias N(0,0.1), gamma N(1,0.1),
                       eps float32(1e-12), S requested; seed 1.
  gated_fp16_4x4096x8192_c128  GatedRMSNorm fp16, X/gate (4, 4096, 8192)
                       N(0,1), scale (128) N(1,0.1), eps 1e-5; seed 2.
  sgn_nhwc_fp16_2x64x64x320  SkipGroupNorm channels_last, X fp16
                       (2, 64, 64, 320) N(0,1), skip (2, 320) N(0,1), bias
                       N(0,0.1), gamma/beta fp32 N(1,0.1)/N(0,0.1), groups 32,
                       eps 1e-5, SiLU, S requested; seed 3.
  sgn_nchw_fp32_16x1280x16x16  SkipGroupNorm NCHW, X fp32 (16, 1280, 16, 16)
                       N(0,2), full skip N(0,1), no bias, gamma/beta fp16
                       N(1,0.1)/N(0,0.1), groups 32, eps 1e-5, no activation,
                       no S; seed 4.
  ssln_fp16_decode_1x4096, ssln_fp16_decode_64x4096  decode-shaped
                       SkipSimplifiedLayerNormalization fp16 (1 or 64 rows of
                       4096), distributions as ssln_fp16_8x2048x4096; seeds 5, 6.
  gated_fp16_decode_64x8192_c8192  decode-shaped GatedRMSNorm fp16, X/gate
                       (64, 8192) N(0,1), C = 8192; seed 7.
  ssln_bf16_8x2048x4096, gated_bf16_4x4096x8192_c128,
  sgn_nhwc_bf16_2x64x64x320, sgn_nchw_bf16_16x1280x16x16  bfloat16 variants
                       of the large workloads (the NCHW one with bfloat16
                       gamma/beta); seeds 8-11.
  ssln_fp32_262144x128  SkipSimplifiedLayerNormalization fp32 with short rows
                       (262,144 rows of 128), distributions as
                       ssln_fp16_8x2048x4096; seed 12 (the rows the pipelined
                       bulk-copy schedule takes).

bfloat16 host arrays are uint16 bit patterns whose dtype is ``BFLOAT16`` (a
uint16 dtype carrying the metadata {"bfloat16": True}); values are drawn in
float32 and converted with torch's round-to-nearest-even conversion.
"""
from __future__ import annotations

import numpy as np

SSLN_EPS = 9.999999960041972e-13  # float32(1e-12)

BFLOAT16 = np.dtype(np.uint16, metadata={"bfloat16": True})


def is_bf16(dtype) -> bool:
    md = np.dtype(dtype).metadata
    return bool(md and md.get("bfloat16"))


def to_bfloat16(a) -> np.ndarray:
    """float32 values -> BFLOAT16 bit patterns (torch's conversion)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).astype(BFLOAT16)


def _cast(z, dtype):
    return to_bfloat16(z) if is_bf16(dtype) else z.astype(dtype, copy=False)

WORKLOADS = {
    "ssln_fp32_64x768": dict(
        op="skip_rms", seed=0, dtype=np.float32, shape=(64, 768), bias=True,
        gamma=("uniform", 0.5, 1.5), epsilon=SSLN_EPS, want_sum=True),
    "ssln_fp16_8x2048x4096": dict(
        op="skip_rms", seed=1, dtype=np.float16, shape=(8, 2048, 4096), bias=True,
        gamma=("normal", 1.0, 0.1), epsilon=SSLN_EPS, want_sum=True),
    "gated_fp16_4x4096x8192_c128": dict(
        op="gated_rms", seed=2, dtype=np.float16, shape=(4, 4096, 8192), C=128,
        epsilon=1e-5),
    "sgn_nhwc_fp16_2x64x64x320": dict(
        op="skip_group", seed=3, dtype=np.float16, mdtype=np.float32,
        shape=(2, 64, 64, 320), channels_last=1, skip="nc", bias=True, x_std=1.0,
        groups=32, epsilon=1e-5, activation=1, want_sum=True),
    "sgn_nchw_fp32_16x1280x16x16": dict(
        op="skip_group", seed=4, dtype=np.float32, mdtype=np.float16,
        shape=(16, 1280, 16, 16), channels_last=0, skip="full", bias=False, x_std=2.0,
        groups=32, epsilon=1e-5, activation=0, want_sum=False),
    # Decode-shaped rows: one generated token per sequence, so a handful of
    # rows of a 4K / 8K hidden state per call (latency-bound, rows/s).
    "ssln_fp16_decode_1x4096": dict(
        op="skip_rms", seed=5, dtype=np.float16, shape=(1, 4096), bias=True,
        gamma=("normal", 1.0, 0.1), epsilon=SSLN_EPS, want_sum=True),
    "ssln_fp16_decode_64x4096": dict(
        op="skip_rms", seed=6, dtype=np.float16, shape=(64, 4096), bias=True,
        gamma=("normal", 1.0, 0.1), epsilon=SSLN_EPS, want_sum=True),
    "gated_fp16_decode_64x8192_c8192": dict(
        op="gated_rms", seed=7, dtype=np.float16, shape=(64, 8192), C=8192,
        epsilon=1e-5),
    # bfloat16 variants of the large workloads (same shapes and distributions).
    "ssln_bf16_8x2048x4096": dict(
        op="skip_rms", seed=8, dtype=BFLOAT16, shape=(8, 2048, 4096), bias=True,
        gamma=("normal", 1.0, 0.1), epsilon=SSLN_EPS, want_sum=True),
    "gated_bf16_4x4096x8192_c128": dict(
        op="gated_rms", seed=9, dtype=BFLOAT16, shape=(4, 4096, 8192), C=128,
        epsilon=1e-5),
    "sgn_nhwc_bf16_2x64x64x320": dict(
        op="skip_group", seed=10, dtype=BFLOAT16, mdtype=np.float32,
        shape=(2, 64, 64, 320), channels_last=1, skip="nc", bias=True, x_std=1.0,
        groups=32, epsilon=1e-5, activation=1, want_sum=True),
    "sgn_nchw_bf16_16x1280x16x16": dict(
        op="skip_group", seed=11, dtype=BFLOAT16, mdtype=BFLOAT16,
        shape=(16, 1280, 16, 16), channels_last=0, skip="full", bias=False, x_std=2.0,
        groups=32, epsilon=1e-5, activation=0, want_sum=False),
    "ssln_fp32_262144x128": dict(
        op="skip_rms", seed=12, dtype=np.float32, shape=(262144, 128), bias=True,
        gamma=("normal", 1.0, 0.1), epsilon=SSLN_EPS, want_sum=True),
    # The NHWC fp16 workload at batch 4: more pixels than the cooperative
    # grid holds in registers, so the slabs stay in shared memory.
    "sgn_nhwc_fp16_4x64x64x320": dict(
        op="skip_group", seed=13, dtype=np.float16, mdtype=np.float32,
        shape=(4, 64, 64, 320), channels_last=1, skip="nc", bias=True, x_std=1.0,
        groups=32, epsilon=1e-5, activation=1, want_sum=True),
}

# Order the workloads are listed in (small SSLN first, decode shapes last).
WORKLOAD_ORDER = list(WORKLOADS)


def _normal(rng, shape, mean, std, dtype):
    z = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        z *= np.float32(std)
    if mean != 0.0:
        z += np.float32(mean)
    return _cast(z, dtype)


def _uniform(rng, shape, lo, hi, dtype):
    z = rng.uniform(lo, hi, size=shape)
    return to_bfloat16(z.astype(np.float32)) if is_bf16(dtype) else z.astype(dtype)


def _draw(rng, spec, shape, dtype):
    kind, a, b = spec
    if kind == "normal":
        return _normal(rng, shape, a, b, dtype)
    return _uniform(rng, shape, a, b, dtype)


def skip_rms_inputs(shape, dtype, seed, bias=True, gamma=("normal", 1.0, 0.1),
                    x_std=1.0):
    """input, skip ~ N(0, x_std); bias ~ N(0, 0.1); gamma per ``gamma``."""
    rng = np.random.default_rng(seed)
    hidden = shape[-1]
    x = _normal(rng, shape, 0.0, x_std, dtype)
    sk = _normal(rng, shape, 0.0, x_std, dtype)
    b = _normal(rng, (hidden,), 0.0, 0.1, dtype) if bias else None
    g = _draw(rng, gamma, (hidden,), dtype)
    return dict(input=x, skip=sk, gamma=g, bias=b)


def gated_rms_inputs(shape, C, dtype, seed, x_std=1.0):
    """X, gate ~ N(0, x_std); scale (C) ~ N(1, 0.1)."""
    rng = np.random.default_rng(seed)
    x = _normal(rng, shape, 0.0, x_std, dtype)
    g = _normal(rng, shape, 0.0, x_std, dtype)
    sc = _normal(rng, (C,), 1.0, 0.1, dtype)
    return dict(x=x, gate=g, scale=sc)


def skip_group_inputs(shape, dtype, mdtype, seed, channels_last=1, skip="full",
                      bias=True, x_std=1.0, x_mean=0.0):
    """X ~ N(x_mean, x_std); skip ~ N(0,1) full, (N,C) or (N,1,1,C); bias ~
    N(0,0.1); gamma ~ N(1,0.1), beta ~ N(0,0.1) of type ``mdtype``."""
    rng = np.random.default_rng(seed)
    if channels_last:
        N, H, W, C = shape
    else:
        N, C, H, W = shape
    x = _normal(rng, shape, x_mean, x_std, dtype)
    if skip == "full":
        sk = _normal(rng, shape, 0.0, 1.0, dtype)
    elif skip == "nc":
        sk = _normal(rng, (N, C), 0.0, 1.0, dtype)
    elif skip == "n11c":
        sk = _normal(rng, (N, 1, 1, C), 0.0, 1.0, dtype)
    else:
        raise ValueError(skip)
    b = _normal(rng, (C,), 0.0, 0.1, dtype) if bias else None
    ga = _normal(rng, (C,), 1.0, 0.1, mdtype)
    be = _normal(rng, (C,), 0.0, 0.1, mdtype)
    return dict(x=x, skip=sk, gamma=ga, beta=be, bias=b)


def workload(name, seed=None):
    """Inputs and attributes of one named workload: ``(spec, arrays)``."""
    spec = dict(WORKLOADS[name])
    s = spec["seed"] if seed is None else seed
    if spec["op"] == "skip_rms":
        arrays = skip_rms_inputs(spec["shape"], spec["dtype"], s, bias=spec["bias"],
                                 gamma=spec["gamma"])
    elif spec["op"] == "gated_rms":
        arrays = gated_rms_inputs(spec["shape"], spec["C"], spec["dtype"], s)
    else:
        arrays = skip_group_inputs(spec["shape"], spec["dtype"], spec["mdtype"], s,
                                   channels_last=spec["channels_last"], skip=spec["skip"],
                                   bias=spec["bias"], x_std=spec["x_std"])
    return spec, arrays


def algorithmic_bytes(name) -> int:
    """Bytes that must be read plus written by one call on the workload:
    every input element read once, every requested output written once."""
    spec = WORKLOADS[name]
    it = np.dtype(spec["dtype"]).itemsize
    numel = int(np.prod(spec["shape"]))
    if spec["op"] == "skip_rms":
        hidden = spec["shape"][-1]
        rd = 2 * numel * it + hidden * it * (2 if spec["bias"] else 1)
        wr = numel * it * (2 if spec["want_sum"] else 1)
        return rd + wr
    if spec["op"] == "gated_rms":
        return 2 * numel * it + spec["C"] * it + numel * it
    if spec["channels_last"]:
        N, H, W, C = spec["shape"]
    else:
        N, C, H, W = spec["shape"]
    mit = np.dtype(spec["mdtype"]).itemsize
    skip_n = numel if spec["skip"] == "full" else N * C
    rd = numel * it + skip_n * it + (C * it if spec["bias"] else 0) + 2 * C * mit
    wr = numel * it * (2 if spec["want_sum"] else 1)
    return rd + wr


def units(name) -> int:
    """Rows (SSLN), C-spans (GatedRMSNorm) or group instances N*groups
    (SkipGroupNorm) processed by one call."""
    spec = WORKLOADS[name]
    numel = int(np.prod(spec["shape"]))
    if spec["op"] == "skip_rms":
        return numel // spec["shape"][-1]
    if spec["op"] == "gated_rms":
        return numel // spec["C"]
    return spec["shape"][0] * spec["groups"]


def device_normal(shape, dtype, seed, device, mean=0.0, std=1.0):
    """Seeded N(mean, std) values drawn directly on a CUDA device with torch's
    generator (float32, then cast to ``dtype``: a torch dtype).  For tensors
    too large to draw on the host; tests copy the parts they check back to the
    host for the oracle, so both sides still see the same bits."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        z.mul_(std)
    if mean != 0.0:
        z.add_(mean)
    return z.to(dtype)
