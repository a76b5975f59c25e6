"""Pins of the oracle's norm variants (FP32 weights, input-scale weights,
gain centers, separate hidden and layer eps) and of per-layer slot lengths.

Sources: page "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.draft.context"
(ContextNormConstants: weight dtype per norm and whether each weight scales
the input; ContextNorms: hidden_eps, pre_eps and the gain centers;
_ContextNormsKernel: the gain center added to each weight element), page
"...cutedsl.common.draft_boundary" (boundary_fragments: an input-scale weight
multiplies the input before the sum of squares and nothing after it) and
page "...runtime.draft" (_slot_groups: each layer inserts the first
len(slots[l]) rows).

Expected values are closed forms of the RMSNorm (sqrt(D) * u / ||u|| up to
eps), exact power-of-two identities, or invariants; none retypes the
oracle's loops.
"""
import math

import numpy as np
import torch

import workloads

D = 8192


def bf16_bits(vals) -> np.ndarray:
    t = torch.tensor(np.asarray(vals, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_of(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def far_from_bf16_boundary(v: float, margin: float = 1e-2) -> bool:
    e = math.floor(math.log2(abs(v)))
    frac = (abs(v) / 2.0 ** (e - 7)) % 1.0
    return abs(frac - 0.5) > margin


def norms(orc, x, L, **kw):
    kw.setdefault("hidden_eps", 0.0)
    kw.setdefault("pre_eps", 0.0)
    return orc.context_norms_ex(np.ascontiguousarray(x), L, **kw)


def rows_of(rng, T, sigma=1.0):
    return bf16_bits(rng.standard_normal((T, D)) * sigma)


def test_defaults_equal_plain_norms(orc):
    # the variant entry with bf16 output-scale weights, center 0 and one eps
    # is the plain chain (both pinned elsewhere for that case)
    rng = np.random.default_rng(1)
    x = rows_of(rng, 5)
    hw = bf16_bits(1 + 0.1 * rng.standard_normal(D))
    pw = bf16_bits(1 + 0.1 * rng.standard_normal((3, D)))
    a = orc.context_norms(x, hw, pw, 3, 1e-5)
    b = norms(orc, x, 3, hidden_w=hw, pre_w=pw, hidden_eps=1e-5, pre_eps=1e-5)
    assert np.array_equal(a, b)


def test_input_scale_constant_row_is_one(orc):
    # x == 2^k, gamma == 2^j: an input-scale norm sees u == 2^(j+k), so with
    # eps = 0 its output is exactly 1; an output-scale norm gives gamma
    x = np.full((2, D), bf16_bits([4.0])[0], dtype=np.uint16)
    g = np.full(D, bf16_bits([2.0])[0], dtype=np.uint16)
    gl = np.stack([np.full(D, bf16_bits([2.0 ** l])[0], dtype=np.uint16) for l in range(3)])
    one, two = bf16_bits([1.0])[0], bf16_bits([2.0])[0]
    out = norms(orc, x, 3, hidden_w=g, hidden_input_scale=True)
    assert np.all(out == one)
    out = norms(orc, x, 3, hidden_w=g, hidden_input_scale=False)
    assert np.all(out == one)                     # z == 2, layer norm -> 1
    # per-layer gains 2^l: input-scale -> every layer 1.0 (each layer its own
    # inverse RMS); output-scale -> 2^l
    out = norms(orc, x, 3, pre_w=gl, pre_input_scale=True)
    assert np.all(out == one)
    out = norms(orc, x, 3, pre_w=gl, pre_input_scale=False)
    for l in range(3):
        assert np.all(out[l] == bf16_bits([2.0 ** l])[0])
    assert two == bf16_bits([2.0])[0]


def test_input_scale_single_nonzero(orc):
    # one non-zero x_c = a, gamma_c = 2, eps = 0: input scale gives
    # u_c * r = +-sqrt(8192) = +-90.51 -> bf16 90.5; output scale gives
    # +-sqrt(8192) * 2 = 181.02 -> 181 (the scale side is visible)
    x = np.zeros((1, D), dtype=np.uint16)
    x[0, 77] = bf16_bits([-3.0])[0]
    g = np.full(D, bf16_bits([2.0])[0], dtype=np.uint16)
    i = norms(orc, x, 1, hidden_w=g, hidden_input_scale=True)
    o = norms(orc, x, 1, hidden_w=g, hidden_input_scale=False)
    # the layer norm (weightless) of a single non-zero z is again +-90.5
    assert bf16_of(i[0, 0, 77:78])[0] == -90.5
    assert bf16_of(o[0, 0, 77:78])[0] == -90.5
    # seen through the layer norm with an output-scale layer gain of 2:
    pw = np.full((1, D), bf16_bits([2.0])[0], dtype=np.uint16)
    o2 = norms(orc, x, 1, pre_w=pw, pre_input_scale=False)
    i2 = norms(orc, x, 1, pre_w=pw, pre_input_scale=True)
    assert bf16_of(o2[0, 0, 77:78])[0] == -181.0
    assert bf16_of(i2[0, 0, 77:78])[0] == -90.5
    others = np.delete(np.arange(D), 77)
    for out in (i, o, o2, i2):
        assert np.all((out[0, 0, others] & 0x7FFF) == 0)


def test_input_scale_weight_shapes_the_row(orc):
    # two non-zero inputs 1 and 1 at columns 5 and 900, gains 1 and 2 there,
    # eps = 0: an input-scale weight makes u = (1, 2), so the norm's output
    # is (1, 2) * sqrt(8192 / 5) = (40.48, 80.95) -> bf16 (40.5, 81.0); a
    # weight that were dropped would leave (64, 64).  Seen through either
    # norm (the other weightless; a weightless layer norm of a row shaped
    # (1, 2) gives the same (1, 2) * sqrt(8192 / 5) again).
    x = np.zeros((1, D), dtype=np.uint16)
    x[0, [5, 900]] = bf16_bits([1.0, 1.0])
    g = np.full(D, bf16_bits([1.0])[0], dtype=np.uint16)
    g[900] = bf16_bits([2.0])[0]
    want = np.array([1.0, 2.0]) * math.sqrt(8192.0 / 5.0)
    assert all(far_from_bf16_boundary(v) for v in want)
    hidden = norms(orc, x, 1, hidden_w=g, hidden_input_scale=True)
    layer = norms(orc, x, 1, pre_w=g[None, :], pre_input_scale=True)
    for out in (hidden, layer):
        assert np.array_equal(out[0, 0, [5, 900]], bf16_bits(want))
        others = np.delete(np.arange(D), [5, 900])
        assert np.all((out[0, 0, others] & 0x7FFF) == 0)


def test_pre_input_scale_layers_equal_weightless(orc):
    # gamma_l == 2^l scales u by 2^l and r by 2^-l: with eps = 0 every
    # layer's output equals the weightless norm's, bit for bit (exact)
    rng = np.random.default_rng(2)
    x = rows_of(rng, 6)
    gl = np.stack([np.full(D, bf16_bits([2.0 ** (l - 1)])[0], dtype=np.uint16) for l in range(4)])
    base = norms(orc, x, 1)
    out = norms(orc, x, 4, pre_w=gl, pre_input_scale=True)
    for l in range(4):
        assert np.array_equal(out[l], base[0])


def test_separate_eps(orc):
    # x == 1, weightless: hidden eps 3 -> r = 1/sqrt(1 + 3) = 0.5, z == 0.5;
    # layer eps 0 -> z's norm is 1.0.  Swapped: z == 1, layer r = 0.5.
    x = np.full((3, D), bf16_bits([1.0])[0], dtype=np.uint16)
    a = norms(orc, x, 2, hidden_eps=3.0, pre_eps=0.0)
    b = norms(orc, x, 2, hidden_eps=0.0, pre_eps=3.0)
    assert np.all(a == bf16_bits([1.0])[0])
    assert np.all(b == bf16_bits([0.5])[0])


def test_gain_center(orc):
    rng = np.random.default_rng(3)
    x = rows_of(rng, 4, 2.0)
    # center 1 and zero weights: gamma == 1 -> the weightless norm, bit exact
    zero_h = np.zeros(D, dtype=np.uint16)
    zero_p = np.zeros((2, D), dtype=np.uint16)
    base = norms(orc, x, 2, hidden_eps=1e-6, pre_eps=1e-6)
    for inp in (False, True):
        c = norms(orc, x, 2, hidden_w=zero_h, pre_w=zero_p, hidden_center=1.0, pre_center=1.0,
                  hidden_eps=1e-6, pre_eps=1e-6, hidden_input_scale=inp, pre_input_scale=inp)
        assert np.array_equal(c, base)
    # center 1 and bf16 weights in [0.5, 1): w + 1 is exact in binary32, so
    # the centered bf16 weight equals the FP32 weight w + 1 with center 0
    w_h = bf16_bits(rng.uniform(0.5, 1.0, D))
    w_p = bf16_bits(rng.uniform(0.5, 1.0, (2, D)))
    f_h = (bf16_of(w_h).astype(np.float64) + 1.0).astype(np.float32)
    f_p = (bf16_of(w_p).astype(np.float64) + 1.0).astype(np.float32)
    c = norms(orc, x, 2, hidden_w=w_h, pre_w=w_p, hidden_center=1.0, pre_center=1.0)
    f = norms(orc, x, 2, hidden_w=f_h, pre_w=f_p)
    assert np.array_equal(c, f)
    # and it differs from the uncentered weights
    u = norms(orc, x, 2, hidden_w=w_h, pre_w=w_p)
    assert not np.array_equal(c, u)


def test_center_zero_keeps_negative_zero_weight(orc):
    # center 0 leaves a -0.0 weight as it is: its column is -0 times the
    # normed value, so the sign bit follows -sign(x); adding 0 would give +0
    x = np.full((1, D), bf16_bits([1.0])[0], dtype=np.uint16)
    w = np.full(D, bf16_bits([1.0])[0], dtype=np.uint16)
    w[5] = 0x8000
    out = norms(orc, x, 1, hidden_w=w)
    assert out[0, 0, 5] == 0x8000


def test_fp32_weights(orc):
    rng = np.random.default_rng(4)
    x = rows_of(rng, 4)
    # bf16-representable FP32 weights give the bf16-weight result exactly
    w_h = bf16_bits(1 + 0.1 * rng.standard_normal(D))
    w_p = bf16_bits(1 + 0.1 * rng.standard_normal((2, D)))
    for inp in (False, True):
        a = norms(orc, x, 2, hidden_w=w_h, pre_w=w_p, hidden_input_scale=inp, pre_input_scale=inp)
        b = norms(orc, x, 2, hidden_w=bf16_of(w_h).copy(), pre_w=bf16_of(w_p).copy(),
                  hidden_input_scale=inp, pre_input_scale=inp)
        assert np.array_equal(a, b)


def test_fp32_weight_bits_below_bf16_matter(orc):
    # three equal non-zeros: the norm is sqrt(8192/3) = 52.2566 times gamma.
    # gamma = 1 + 3*2^-10 is exact in FP32 and rounds to 1.0 in bf16:
    # 52.2566 * gamma = 52.4097 -> bf16 52.5, while 52.2566 -> 52.25
    g = np.float32(1 + 3 * 2.0 ** -10)
    x = np.zeros((1, D), dtype=np.uint16)
    x[0, [10, 2000, 4100]] = bf16_bits([1.0])[0]
    pw = np.full((1, D), g, dtype=np.float32)
    out = norms(orc, x, 1, pre_w=pw)
    expect = math.sqrt(8192 / 3) * float(g)
    assert far_from_bf16_boundary(expect)
    assert np.array_equal(out[0, 0, [10, 2000, 4100]], bf16_bits([expect] * 3))
    out_bf16 = norms(orc, x, 1, pre_w=bf16_bits(pw.astype(np.float64)))
    assert np.all(bf16_of(out_bf16[0, 0, [10, 2000, 4100]]) == 52.25)
    # the hidden FP32 weight on one of the three columns: z = (52.5, 52.25,
    # 52.25), whose layer norm at column 10 is 52.5 * sqrt(8192 / (52.5^2 +
    # 2 * 52.25^2)) in closed form
    hw = np.ones(D, dtype=np.float32)
    hw[10] = g
    out = norms(orc, x, 1, hidden_w=hw)
    z0 = 52.5
    expect0 = z0 * math.sqrt(8192 / (z0 ** 2 + 2 * 52.25 ** 2))
    expect1 = 52.25 * math.sqrt(8192 / (z0 ** 2 + 2 * 52.25 ** 2))
    assert far_from_bf16_boundary(expect0) and far_from_bf16_boundary(expect1)
    assert np.array_equal(out[0, 0, [10, 2000]], bf16_bits([expect0, expect1]))


def test_store_per_layer_rows(orc):
    # each layer writes exactly the first rows_l rows' slots; every other
    # cache entry keeps the sentinel ([rt] _slot_groups)
    case = workloads.random_case(11, T=40, L=3, H=2, max_position=64, num_blocks=8,
                                 block_size=8, neg_frac=0.0)
    H = 2
    rng = np.random.default_rng(5)
    kv = bf16_bits(rng.standard_normal((3, 40, 128 * H)))
    rows = [40, 17, 0]
    caches = [np.full(case["cache_shape"], 0x5A5A, dtype=np.uint16) for _ in range(3)]
    err = orc.kv_store_from_projection(kv, H, case["positions"], case["slots"], case["cos_sin"],
                                       caches, case["eps"], rows)
    assert err == 0
    for l in range(3):
        written = np.zeros(case["cache_shape"][0] * case["cache_shape"][2], dtype=bool)
        for t in range(rows[l]):
            written[case["slots"][l][t]] = True
        c = caches[l]
        bs = case["cache_shape"][2]
        for s in range(written.size):
            entry = c[s // bs, :, s % bs, :]
            if written[s]:
                # V is a bit copy of the row that owns the slot
                t = int(np.nonzero(case["slots"][l][:rows[l]] == s)[0][0])
                assert np.array_equal(entry[:, 64:], kv[l, t, 64 * H:].reshape(H, 64))
            else:
                assert np.all(entry == 0x5A5A)
