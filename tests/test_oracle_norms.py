"""Pins of the oracle's row norms (a1, a2) and its reduction orders.

Sources: page "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.draft.context"
(ContextNorms, _ContextNormsKernel: hidden norm, BF16 rounding, per-layer
input norm, stack) and "...cutedsl.common.draft_boundary" (boundary_fragments:
the inverse RMS from fma(sum, 1/D, eps), then x * r, then * gamma).

Every expected value here comes from a closed form (the RMSNorm of a constant
or sparse row is sqrt(D) * x / ||x|| up to eps), an exact hand derivation
(tests/golden/sum_order_cases.json), or an invariant; none retypes the
oracle's loops.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

D = 8192
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sum_order_cases.json")


def bf16_bits(vals) -> np.ndarray:
    """Library rounding (torch) of float64 closed-form values to bf16 bits."""
    t = torch.tensor(np.asarray(vals, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_of(vals) -> np.ndarray:
    return np.asarray(vals, dtype=np.float32).view(np.uint32) >> 16


def rng_bf16(rng, shape, mu, sigma):
    a = (rng.standard_normal(shape) * sigma + mu).astype(np.float32)
    return bf16_bits(a.astype(np.float64))


def far_from_bf16_boundary(v: float, margin: float = 1e-3) -> bool:
    """True when v is not within `margin` (relative to the bf16 spacing) of a
    rounding boundary, so eps and binary32 noise cannot move its rounding."""
    if v == 0:
        return True
    e = math.floor(math.log2(abs(v)))
    q = 2.0 ** (e - 7)
    frac = (abs(v) / q) % 1.0
    return abs(frac - 0.5) > margin


def _row(case):
    v = np.full(case["width"], case["fill"], dtype=np.float32)
    for i, val in case["set"]:
        v[i] = val
    return v


def test_golden_row_orders(orc):
    cases = json.load(open(GOLDEN))["row_cases"]
    for case in cases:
        got = orc.row_sumsq(_row(case))
        assert got == np.float32(case["expected"]), case["name"]
        for name, other in case["other_orders"].items():
            assert np.float32(other) != got, (case["name"], name)


def test_golden_head_orders(orc):
    cases = json.load(open(GOLDEN))["head_cases"]
    for case in cases:
        got = orc.head_sumsq(_row(case))
        assert got == np.float32(case["expected"]), case["name"]


def test_constant_row_sum_is_exact(orc):
    for k in (-3, 0, 5):
        v = np.full(D, 2.0 ** k, dtype=np.float32)
        assert orc.row_sumsq(v) == np.float32(D * 4.0 ** k)


def test_inv_rms_scalar_closed_forms(orc):
    # S = D * 4^k, eps tiny: fma gives 4^k, sqrt 2^k, r = 2^-k exactly
    for k in (-4, 0, 3):
        assert orc.inv_rms(D * 4.0 ** k, 2.0 ** -13, 0.0) == np.float32(2.0 ** -k)
    # eps enters inside the root, added to the mean: mean 2^-25 + eps 2^-25 = 2^-24
    assert orc.inv_rms(2.0 ** -12, 2.0 ** -13, 2.0 ** -25) == np.float32(2.0 ** 12)
    # the head width: S = 64 * 9, eps 0 -> 1/3 correctly rounded
    assert orc.inv_rms(576.0, 2.0 ** -6, 0.0) == np.float32(1.0) / np.float32(3.0)


@pytest.mark.parametrize("k", [-3, 0, 5])
def test_constant_row_normalises_to_one_and_to_gain(orc, k):
    T, L = 3, 2
    x = np.full((T, D), bf16_bits([2.0 ** k])[0], dtype=np.uint16)
    out = orc.context_norms(x, None, None, L, 1e-6)
    assert np.all(out == 0x3F80)
    rng = np.random.default_rng(3)
    pre = rng_bf16(rng, (L, D), 1.0, 0.1)
    out = orc.context_norms(x, None, pre, L, 1e-6)
    assert np.array_equal(out, np.broadcast_to(pre[:, None, :], out.shape))
    # hidden gain 2 everywhere: z = 2, the layer norm brings it back to gamma
    hid = np.full(D, 0x4000, dtype=np.uint16)
    out = orc.context_norms(x, hid, pre, L, 1e-6)
    assert np.array_equal(out, np.broadcast_to(pre[:, None, :], out.shape))


def test_one_hot_row_is_sqrt_d(orc):
    rng = np.random.default_rng(5)
    cols = rng.choice(D, size=6, replace=False)
    T = len(cols)
    x = np.zeros((T, D), dtype=np.uint16)
    signs = np.where(np.arange(T) % 2 == 0, 1.0, -1.0)
    for t, c in enumerate(cols):
        x[t, c] = bf16_bits([16.0 * signs[t]])[0]
    out = orc.context_norms(x, None, None, 3, 1e-6)
    want = bf16_bits(np.sqrt(D) * signs)     # sqrt(8192) = 90.51 -> 90.5
    for t, c in enumerate(cols):
        row = out[:, t, :]
        assert np.all(row[:, c] == want[t])
        others = np.delete(row, c, axis=1)
        assert np.all(others == 0)


def test_two_sparse_row_closed_form(orc):
    # x = (3, 4) at two columns: each norm maps x to sqrt(D) * x / ||x||,
    # with the hidden result rounded to bf16 before the layer norm reads it
    x = np.zeros((1, D), dtype=np.uint16)
    a, b = 100, 5000
    x[0, a], x[0, b] = bf16_bits([3.0, 4.0])
    eps = 1e-6
    z = np.array([3.0, 4.0]) / np.sqrt(25.0 / D + eps)
    zb = bf16_bits(z).astype(np.uint32)
    zf = (zb << 16).view(np.float32).astype(np.float64)
    o = zf / np.sqrt(np.sum(zf ** 2) / D + eps)
    assert all(far_from_bf16_boundary(v) for v in np.concatenate([z, o]))
    out = orc.context_norms(x, None, None, 2, eps)
    assert np.all(out[:, 0, a] == bf16_bits([o[0]])[0])
    assert np.all(out[:, 0, b] == bf16_bits([o[1]])[0])


def test_hidden_output_is_rounded_before_layer_norm(orc):
    # x = (1, 3) with hidden gains (g1, g2): z = bf16(sqrt(D/10) * (g1, 3 g2)).
    # Search gains whose final bf16 result differs between a rounded and an
    # unrounded z, and check the oracle follows the rounded one.
    rng = np.random.default_rng(9)
    a, b = 17, 4099
    eps = 1e-6
    found = 0
    for _ in range(4000):
        g = bf16_bits(rng.uniform(0.5, 2.0, 2))
        gf = (g.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        y = np.array([1.0, 3.0]) / np.sqrt(10.0 / D + eps) * gf
        zr = (bf16_bits(y).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        o_r = zr / np.sqrt(np.sum(zr ** 2) / D + eps)
        o_u = y / np.sqrt(np.sum(y ** 2) / D + eps)
        if not all(far_from_bf16_boundary(v, 2e-3) for v in np.concatenate([y, o_r, o_u])):
            continue
        if np.array_equal(bf16_bits(o_r), bf16_bits(o_u)):
            continue
        x = np.zeros((1, D), dtype=np.uint16)
        x[0, a], x[0, b] = bf16_bits([1.0, 3.0])
        hid = np.full(D, 0x3F80, dtype=np.uint16)
        hid[a], hid[b] = g
        out = orc.context_norms(x, hid, None, 1, eps)
        assert out[0, 0, a] == bf16_bits([o_r[0]])[0]
        assert out[0, 0, b] == bf16_bits([o_r[1]])[0]
        found += 1
        if found == 5:
            break
    assert found == 5


def test_zero_row_keeps_sign_of_zero(orc):
    x = np.zeros((2, D), dtype=np.uint16)
    x[1, ::3] = 0x8000
    rng = np.random.default_rng(1)
    pre = np.abs(rng_bf16(rng, (2, D), 1.0, 0.1).view(np.int16)).view(np.uint16)
    out = orc.context_norms(x, None, pre, 2, 1e-6)
    assert np.array_equal(out, np.broadcast_to(x[None], out.shape))


def test_power_of_two_scaling_invariance_with_zero_eps(orc):
    rng = np.random.default_rng(2)
    x = rng_bf16(rng, (4, D), 0.0, 1.0)
    hid = rng_bf16(rng, (D,), 1.0, 0.1)
    pre = rng_bf16(rng, (2, D), 1.0, 0.1)
    base = orc.context_norms(x, hid, pre, 2, 0.0)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    for s in (8.0, 2.0 ** -3):
        xs = bf16_bits((xf * s).astype(np.float64))
        assert np.array_equal(orc.context_norms(xs, hid, pre, 2, 0.0), base)


def test_layer_norm_scalar_is_shared_across_layers(orc):
    rng = np.random.default_rng(4)
    x = rng_bf16(rng, (3, D), 0.0, 2.0)
    hid = rng_bf16(rng, (D,), 1.0, 0.1)
    g = rng_bf16(rng, (D,), 1.0, 0.1)
    g2 = rng_bf16(rng, (D,), 1.0, 0.1)
    pre = np.stack([g, g2, g])
    out = orc.context_norms(x, hid, pre, 3, 1e-5)
    assert np.array_equal(out[0], out[2])
    assert not np.array_equal(out[0], out[1])


def test_rms_of_output_is_one(orc):
    # the weightless norm output has mean square 1 up to bf16 rounding
    rng = np.random.default_rng(6)
    x = rng_bf16(rng, (8, D), 0.0, 3.0)
    out = orc.context_norms(x, None, None, 1, 1e-6)
    of = (out.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ms = np.mean(of ** 2, axis=-1)
    assert np.all(np.abs(ms - 1.0) < 2.0 ** -7)


def test_hidden_gain_multiplies_after_the_inverse_rms(orc):
    # z_c = bf16((x_c * r) * g_c): the row is scaled by its inverse RMS, then
    # by the gain.  (x_c * g_c) * r rounds differently now and then; among
    # two-sparse rows (one rounding in their sum of squares, so r is
    # unambiguous) find some where the two orders give different outputs and
    # check the oracle follows the first.
    eps = np.float32(1e-6)
    rng = np.random.default_rng(21)
    n = 1 << 20
    f = lambda bits: (bits.astype(np.uint32) << 16).view(np.float32)
    x = f(rng_bf16(rng, (n, 2), 0.0, 1.0))
    g = f(rng_bf16(rng, (n, 2), 1.0, 0.1))
    keep = np.all(np.abs(x) >= 0.25, axis=1)
    x, g = x[keep], g[keep]
    S = x[:, 0] * x[:, 0] + x[:, 1] * x[:, 1]
    # fma(S, 2^-13, eps): exact in float64 for these S, then one rounding
    v = (S.astype(np.float64) * 2.0 ** -13 + np.float64(eps)).astype(np.float32)
    r = np.float32(1.0) / np.sqrt(v)
    rn = lambda a: bf16_bits(a.astype(np.float64)).reshape(a.shape)   # bf16 of float32, RNE
    first = rn((x * r[:, None]) * g)
    other = rn((x * g) * r[:, None])
    hits = np.flatnonzero(np.any(first != other, axis=1))
    a, b = 100, 5000
    checked = 0
    for i in hits:
        expect = []
        for z_bits in (first[i], other[i]):
            z = f(z_bits.astype(np.uint16))
            r2 = orc.inv_rms(z[0] * z[0] + z[1] * z[1], 2.0 ** -13, eps)
            expect.append(rn(z * np.float32(r2)))
        if np.array_equal(expect[0], expect[1]):
            continue                     # the layer norm hides the difference
        assert orc.inv_rms(S[i], 2.0 ** -13, eps) == r[i]
        row = np.zeros((1, D), dtype=np.uint16)
        row[0, a], row[0, b] = bits_of(x[i])
        hid = np.full(D, 0x3F80, dtype=np.uint16)
        hid[a], hid[b] = bits_of(g[i])
        out = orc.context_norms(row, hid, None, 1, float(eps))
        assert out[0, 0, a] == expect[0][0] and out[0, 0, b] == expect[0][1]
        checked += 1
    assert checked >= 2
