"""Pins of the oracle's bf16 conversions against definitions independent of
its bit trick: the nearest bf16 value found by comparing distances in
float64 (ties to the even mantissa), and torch's CPU float->bf16 conversion
(a library routine).  Rounding points: [ctx] round_bf16 / pack_bf16x2_rn on
the page "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.draft.context".
"""
import fractions

import numpy as np
import torch


def nearest_bf16_by_distance(f: np.ndarray) -> np.ndarray:
    """RNE by definition: candidates are the truncation toward zero and the
    next bf16 away from zero; the nearer wins, a tie goes to the even one."""
    u = f.view(np.uint32)
    lo = (u >> 16).astype(np.uint32)               # truncation, same sign
    hi = lo + 1                                    # next magnitude up
    lo_val = (lo << 16).view(np.float32).astype(np.float64)
    mag_hi = hi & 0x7FFF
    x = f.astype(np.float64)
    hi_val = np.where(mag_hi == 0x7F80,            # past max finite: Inf
                      np.copysign(2.0 ** 128, x),
                      (hi << 16).astype(np.uint32).view(np.float32).astype(np.float64))
    dlo = np.abs(x - lo_val)
    dhi = np.abs(hi_val - x)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((lo & 1) == 1))
    return np.where(pick_hi, hi, lo).astype(np.uint16)


def stratified_f32() -> np.ndarray:
    hi = np.arange(1 << 16, dtype=np.uint32)
    lows = np.array([0x0000, 0x0001, 0x0002, 0x3FFF, 0x4000, 0x7FFE, 0x7FFF, 0x8000,
                     0x8001, 0x8002, 0xBFFF, 0xC000, 0xFFFE, 0xFFFF, 0x1234, 0xEDCB],
                    dtype=np.uint32)
    u = (hi[:, None] << 16) | lows[None, :]
    u = u.reshape(-1)
    f = u.view(np.float32)
    return f[~np.isnan(f)]


def test_bf16_rn_matches_distance_definition(orc):
    f = stratified_f32()
    assert np.array_equal(orc.bf16_rn_array(f), nearest_bf16_by_distance(f))


def test_bf16_rn_matches_torch_on_stratified_and_random(orc):
    f = stratified_f32()
    rng = np.random.default_rng(7)
    r = rng.integers(0, 1 << 32, size=1 << 24, dtype=np.uint64).astype(np.uint32).view(np.float32)
    f = np.concatenate([f, r[~np.isnan(r)]])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.bf16_rn_array(f), ref)


def test_bf16_rn_special_values(orc):
    # ties: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1.0)
    assert orc.bf16_rn(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even)
    assert orc.bf16_rn(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert orc.bf16_rn(-0.0) == 0x8000
    assert orc.bf16_rn(float("inf")) == 0x7F80
    assert orc.bf16_rn(float("-inf")) == 0xFF80
    # largest finite float32 overflows bf16 to Inf
    assert orc.bf16_rn(float(np.finfo(np.float32).max)) == 0x7F80
    # smallest float32 subnormal rounds to +0, 2^-133 is the smallest bf16 subnormal
    assert orc.bf16_rn(float(np.float32(2.0 ** -149))) == 0x0000
    assert orc.bf16_rn(2.0 ** -133) == 0x0001
    # reading R4: NaN -> 0x7FFF
    for bits in (0x7FC00000, 0x7F800001, 0xFFC00000, 0x7FFFFFFF):
        f = np.array([bits], dtype=np.uint32).view(np.float32)
        assert orc.bf16_rn_array(f)[0] == 0x7FFF


def test_f32_widening_is_exact(orc):
    # 1.0, -1.0, the smallest bf16 subnormal 2^-133, its negative, the largest
    # finite bf16 (2 - 2^-7) * 2^127, and +Inf
    for v, want in ((0x0000, 0.0), (0x3F80, 1.0), (0xBF80, -1.0), (0x0001, 2.0 ** -133),
                    (0x8001, -(2.0 ** -133)), (0x7F7F, (2 - 2.0 ** -7) * 2.0 ** 127),
                    (0x7F80, float("inf"))):
        assert orc.f32(v) == want


def _exact_nearest_bf16(d: float) -> int:
    """Brute force with rationals for d >= 0: scan the bf16 patterns around
    d's binary32 neighbourhood, keep the nearest (ties: even pattern)."""
    x = fractions.Fraction(d)
    base = int(np.array([d], dtype=np.float32).view(np.uint32)[0] >> 16)
    best = None
    for b in range(max(base - 2, 0), min(base + 3, 0x7F81)):
        val = np.array([b << 16], dtype=np.uint32).view(np.float32)[0]
        cand = fractions.Fraction(2 ** 128) if not np.isfinite(val) else fractions.Fraction(float(val))
        key = (abs(cand - x), b & 1)
        if best is None or key < best[0]:
            best = (key, b)
    return best[1]


def test_bf16_rn_f64_direct_rounding(orc):
    rng = np.random.default_rng(11)
    ds = list(rng.standard_normal(300) * 10.0 ** rng.integers(-30, 30, 300))
    # a double just above a bf16 midpoint: a binary32 detour would first round
    # it onto the midpoint and then tie to even (down); direct rounding goes up
    mid = 1.0 + 2.0 ** -8
    ds += [mid + 2.0 ** -40, mid - 2.0 ** -40, -(mid + 2.0 ** -40), mid]
    for d in ds:
        assert orc.bf16_rn_f64(d) == _exact_nearest_bf16(abs(d)) | (0x8000 if d < 0 else 0), d
    assert orc.bf16_rn_f64(mid + 2.0 ** -40) == 0x3F81
    # binary32-representable inputs agree with the binary32 conversion
    f = stratified_f32()
    f = f[np.isfinite(f)]
    assert np.array_equal(orc.bf16_rn_f64_array(f.astype(np.float64)), orc.bf16_rn_array(f))
