"""Pins for the oracle's bfloat16 support.

bfloat16 is not among the pages' element types; the library adds it as a
storage type with the same arithmetic (fp32 compute, one rounding at each
store).  The oracle's bfloat16 conversion is written from the format
definition; these tests pin it, and the operators' bfloat16 plumbing, against
facts that do not come from the oracle: bfloat16 is the upper half of a
binary32 (so every pattern's value is known exactly), torch's library
conversion, hand-derived boundary and tie cases, and the float32 oracle on
inputs whose residual sums are exact in bfloat16.
"""
import numpy as np
import pytest
import torch

import oracle
from residual_add_normalization_gb300 import synthetic


def _all_patterns():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _upper_half(bits):
    """The binary32 whose upper 16 bits are ``bits`` (exact bfloat16 value)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_bf16_to_f32_exhaustive_is_upper_half_of_binary32():
    bits = _all_patterns()
    ours = oracle.bf16_to_f32(bits)
    ref = _upper_half(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_round_trip_exhaustive():
    bits = _all_patterns()
    f = _upper_half(bits)
    back = oracle.f32_to_bf16(f).view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(back[~nan], bits[~nan])
    assert np.all(np.isnan(_upper_half(back[nan])))
    with np.errstate(invalid="ignore"):
        back64 = oracle.f64_to_bf16(f.astype(np.float64)).view(np.uint16)
    assert np.array_equal(back64[~nan], bits[~nan])


def test_f32_to_bf16_random_bits_match_torch():
    rng = np.random.default_rng(7)
    n = 2_000_000
    f = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32).view(np.float32)
    # every exponent, and patterns whose low 16 bits sit at or next to a tie
    low = np.array([0x7FFF, 0x8000, 0x8001, 0x0000, 0xFFFF], np.uint32)
    hi = rng.integers(0, 1 << 16, size=n // 4, dtype=np.uint32)
    ties = ((hi[:, None] << 16) | low[None, :]).reshape(-1).view(np.float32)
    f = np.concatenate([f, ties])
    f = f[~np.isnan(f)]
    ours = oracle.f32_to_bf16(f).view(np.uint16)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def _bits64(v):
    return int(oracle.f64_to_bf16(np.array([v], np.float64)).view(np.uint16)[0])


def test_bf16_hand_boundaries():
    # 1.0 = 0x3F80; ulp at 1 is 2^-7
    assert _bits64(1.0) == 0x3F80
    assert _bits64(1.0 + 2.0**-8) == 0x3F80              # tie -> even (1.0)
    assert _bits64(1.0 + 3 * 2.0**-8) == 0x3F82          # tie -> even (1 + 2^-6)
    assert _bits64(1.0 + 2.0**-8 + 2.0**-40) == 0x3F81   # above the tie: up
    assert _bits64(-2.0) == 0xC000
    # largest finite (2 - 2^-7) * 2^127 = 0x7F7F; overflow at the midpoint
    big = (2.0 - 2.0**-7) * 2.0**127
    mid = (2.0 - 2.0**-8) * 2.0**127
    assert _bits64(big) == 0x7F7F
    assert _bits64(np.nextafter(mid, 0.0)) == 0x7F7F
    assert _bits64(mid) == 0x7F80
    assert _bits64(-mid) == 0xFF80
    # subnormals: quantum 2^-133; half of it ties to zero, 1.5 quanta to 2
    assert _bits64(2.0**-133) == 0x0001
    assert _bits64(2.0**-134) == 0x0000
    assert _bits64(3 * 2.0**-134) == 0x0002
    assert _bits64(-2.0**-134) == 0x8000
    # 127.5 quanta ties to 128 quanta = the smallest normal 2^-126
    assert _bits64(127.5 * 2.0**-133) == 0x0080
    assert _bits64(2.0**-126) == 0x0080
    assert _bits64(np.inf) == 0x7F80 and _bits64(0.0) == 0 and _bits64(-0.0) == 0x8000
    assert _bits64(np.nan) & 0x7F80 == 0x7F80 and _bits64(np.nan) & 0x7F


def test_f64_to_bf16_single_rounding():
    """Double -> bfloat16 rounds once: a double just above a tie whose float32
    rounding lands on the tie must go up, not to even."""
    rng = np.random.default_rng(3)
    base = rng.integers(0x3000, 0x5000, size=10000).astype(np.uint16)
    lo = _upper_half(base).astype(np.float64)
    ulp = _upper_half(base + 1).astype(np.float64) - lo
    just_above = lo + ulp / 2 + ulp * 2.0**-30
    assert np.all(just_above.astype(np.float32).astype(np.float64) == lo + ulp / 2)
    got = oracle.f64_to_bf16(just_above).view(np.uint16)
    assert np.array_equal(got, base + 1)


def _bf(a):
    return synthetic.to_bfloat16(np.asarray(a, np.float32))


def test_bf16_residual_sum_matches_torch():
    """S = round_bf16((x + skip) + bias) with the adds in float32, against
    torch's float32 adds and bfloat16 conversion."""
    d = synthetic.skip_rms_inputs((16, 384), synthetic.BFLOAT16, seed=11, bias=True)
    _, s = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"], epsilon=1e-6)
    t = {k: torch.from_numpy(oracle.bf16_to_f32(v)) for k, v in d.items()}
    ref = ((t["input"] + t["skip"]) + t["bias"]).to(torch.bfloat16)
    assert np.array_equal(s.view(np.uint16), ref.view(torch.int16).numpy().view(np.uint16))
    assert oracle.is_bf16(s.dtype)


def _bf16_ulps(a, b):
    def ordinal(x):
        u = x.view(np.uint16).astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u & 0x7FFF)
    return np.abs(ordinal(a) - ordinal(b))


def test_bf16_operators_agree_with_float32_oracle_on_exact_sums():
    """With inputs whose float32 residual sums are exact in bfloat16 (small
    dyadic values), the bfloat16 oracle sees the same S as the float32 one, so
    its Y is the float32 oracle's Y rounded to bfloat16 (within one unit: the
    float32 result was itself rounded once)."""
    rng = np.random.default_rng(5)
    q = lambda *shape: (rng.integers(-16, 17, size=shape) / 8.0).astype(np.float32)
    x, sk, ga, bi = q(8, 64), q(8, 64), q(64) + 2.0, q(64)
    y16, s16 = oracle.skip_rms(_bf(x), _bf(sk), _bf(ga), _bf(bi), epsilon=1e-5)
    y32, s32 = oracle.skip_rms(x, sk, ga, bi, epsilon=1e-5)
    assert np.array_equal(oracle.bf16_to_f32(s16), s32)
    assert _bf16_ulps(y16, _bf(y32)).max() <= 1

    xg, g = q(4, 96), q(4, 96)
    sc = q(32) + 1.5
    yg16 = oracle.gated_rms(_bf(xg), _bf(g), _bf(sc), epsilon=1e-5)
    yg32 = oracle.gated_rms(xg, g, sc, epsilon=1e-5)
    assert _bf16_ulps(yg16, _bf(yg32)).max() <= 1

    for cl, shape in ((1, (2, 3, 5, 8)), (0, (2, 8, 3, 5))):
        X, SK = q(*shape), q(2, 8)
        gam, bet, b8 = q(8) + 1.0, q(8), q(8)
        for mgam, mbet in ((gam, bet), (_bf(gam), _bf(bet))):
            yy16, ss16 = oracle.skip_group(_bf(X), _bf(SK), mgam, mbet, _bf(b8), groups=4,
                                           activation=1, channels_last=cl)
            yy32, ss32 = oracle.skip_group(X, SK, gam, bet, b8, groups=4, activation=1,
                                           channels_last=cl)
            assert np.array_equal(oracle.bf16_to_f32(ss16), ss32)
            assert _bf16_ulps(yy16, _bf(yy32)).max() <= 1


def test_bf16_ssln_hand_case():
    """s = [3, 4], eps = 0: ms = 12.5, y = [3, 4] / sqrt(12.5) =
    [0.84852813..., 1.13137085...]; in bfloat16 0.84852813 lies between
    0.84765625 (0x3F59) and 0.8515625 (0x3F5A), nearer the first, and
    1.13137085 between 1.125 (0x3F90) and 1.1328125 (0x3F91), nearer the
    second."""
    x = _bf([[1.0, 3.0]])
    sk = _bf([[2.0, 1.0]])
    y, s = oracle.skip_rms(x, sk, _bf([1.0, 1.0]), None, epsilon=0.0)
    assert list(s.view(np.uint16)[0]) == [0x4040, 0x4080]  # 3.0, 4.0
    assert list(y.view(np.uint16)[0]) == [0x3F59, 0x3F91]


def test_bf16_arrays_are_rejected_against_other_types():
    x = _bf(np.ones((2, 8)))
    with pytest.raises(TypeError):
        oracle.skip_rms(x, np.ones((2, 8), np.float16), _bf(np.ones(8)))
    with pytest.raises(TypeError):
        oracle.skip_rms(x, np.ones((2, 8), np.uint16), _bf(np.ones(8)))


def test_bf16_y_matches_float64_reference_on_rounded_sums():
    """Y from the bfloat16-rounded S: the float64 textbook formulas (torch's
    rms and group norm in float64) on the oracle's S, rounded once to
    bfloat16, must give the oracle's Y bit for bit."""
    d = synthetic.skip_rms_inputs((16, 384), synthetic.BFLOAT16, seed=21, bias=True)
    y, s = oracle.skip_rms(d["input"], d["skip"], d["gamma"], d["bias"], epsilon=1e-6)
    S = torch.from_numpy(oracle.bf16_to_f32(s)).double()
    g = torch.from_numpy(oracle.bf16_to_f32(d["gamma"])).double()
    ref = S / torch.sqrt((S * S).mean(-1, keepdim=True) + float(np.float32(1e-6))) * g
    assert np.array_equal(y.view(np.uint16), oracle.f64_to_bf16(ref.numpy()).view(np.uint16))

    gd = synthetic.skip_group_inputs((2, 32, 6, 5), synthetic.BFLOAT16, np.float32, seed=22,
                                     channels_last=0, skip="full", bias=True, x_std=3.0)
    yg, sg = oracle.skip_group(gd["x"], gd["skip"], gd["gamma"], gd["beta"], gd["bias"],
                               groups=8, activation=1, epsilon=1e-5, channels_last=0)
    S = torch.from_numpy(oracle.bf16_to_f32(sg)).double()
    z = torch.nn.functional.group_norm(S, 8, torch.from_numpy(gd["gamma"]).double(),
                                       torch.from_numpy(gd["beta"]).double(),
                                       eps=float(np.float32(1e-5)))
    z = torch.nn.functional.silu(z)
    assert np.array_equal(yg.view(np.uint16), oracle.f64_to_bf16(z.numpy()).view(np.uint16))
