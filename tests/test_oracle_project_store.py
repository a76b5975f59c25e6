"""Pins of the oracle's projection (a3) and store chain (a5-a7).

Sources: page "vllm.models.muse_spark.nvidia.specialized_decode.runtime.draft"
(ContextKV._project: torch.bmm of the stacked norms with the K/V weight;
ContextKV.store: K = the first 64H columns, V the next 64H) and
"...cutedsl.draft.context" (ContextKvStore, _ContextKvStoreKernel: weightless
K-norm, BF16 key, GPT-J RoPE with cos in columns 0..31 and sin in 32..63,
insert at [slot // block_size, h, slot % block_size], negative slot skips).
"""
import numpy as np
import pytest
import torch

HD = 64


def bf16_bits(vals) -> np.ndarray:
    t = torch.tensor(np.asarray(vals, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def to_f64(bits) -> np.ndarray:
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rnd_bf16(rng, shape, sigma=1.0, mu=0.0):
    return bf16_bits(rng.standard_normal(shape) * sigma + mu)


# ------------------------------------------------------------- projection

@pytest.mark.parametrize("w_nd", [False, True])
def test_projection_one_hot_weight_selects_columns(orc, w_nd):
    rng = np.random.default_rng(0)
    L, T, D, N = 2, 5, 256, 128
    a = rnd_bf16(rng, (L, T, D))
    perm = rng.integers(0, D, size=(L, N))
    W = np.zeros((L, D, N), dtype=np.uint16)
    for l in range(L):
        W[l, perm[l], np.arange(N)] = 0x3F80
    Wx = np.ascontiguousarray(W.transpose(0, 2, 1)) if w_nd else W
    out, ab = orc.kv_project(a, Wx, w_nd=w_nd)
    for l in range(L):
        assert np.array_equal(out[l], to_f64(a[l][:, perm[l]]))
        assert np.array_equal(ab[l], np.abs(to_f64(a[l][:, perm[l]])))


@pytest.mark.parametrize("w_nd", [False, True])
def test_projection_matches_library_matmul(orc, w_nd):
    rng = np.random.default_rng(1)
    L, T, D, N = 3, 7, 192, 256
    a = rnd_bf16(rng, (L, T, D))
    W = rnd_bf16(rng, (L, D, N), 0.02)
    Wx = np.ascontiguousarray(W.transpose(0, 2, 1)) if w_nd else W
    rows = np.array([6, 0, 3], dtype=np.int64)
    out, ab = orc.kv_project(a, Wx, rows=rows, w_nd=w_nd)
    af, wf = to_f64(a), to_f64(W)
    ref = np.einsum("ltk,lkn->ltn", af[:, rows], wf)
    refab = np.einsum("ltk,lkn->ltn", np.abs(af[:, rows]), np.abs(wf))
    assert np.allclose(out, ref, rtol=0, atol=1e-12 * refab.max())
    assert np.allclose(ab, refab, rtol=1e-13)


# ------------------------------------------------------------------ store

def _store(orc, kv, H, positions, slots, cos_sin, caches, eps=1e-6, rows=None):
    L, T, N = kv.shape
    return orc.kv_store_from_projection(kv, H, positions, slots, cos_sin, caches, eps,
                                        T if rows is None else rows)


def _caches(L, nb, H, bs, fill=0x5A5A):
    return [np.full((nb, H, bs, 2 * HD), fill, dtype=np.uint16) for _ in range(L)]


def test_insert_layout_and_untouched_slots(orc):
    rng = np.random.default_rng(2)
    L, T, H, nb, bs = 2, 6, 4, 5, 8
    kv = rnd_bf16(rng, (L, T, 2 * H * HD))
    slots = [np.array([37, -1, 0, 31, 5, -7], dtype=np.int64),
             np.array([1, 2, -1, 3, 30, 17], dtype=np.int64)]
    caches = _caches(L, nb, H, bs)
    before = [c.copy() for c in caches]
    err = _store(orc, kv, H, None, slots, None, caches)
    assert err == 0
    for l in range(L):
        written = np.zeros((nb, bs), dtype=bool)
        for t, s in enumerate(slots[l]):
            if s < 0:
                continue
            b, p = divmod(int(s), bs)
            written[b, p] = True
            for h in range(H):
                v = kv[l, t, H * HD + h * HD: H * HD + (h + 1) * HD]
                assert np.array_equal(caches[l][b, h, p, HD:], v)     # V bit copy
                assert not np.array_equal(caches[l][b, h, p, :HD], before[l][b, h, p, :HD])
        # every (block, page) not named by a non-negative slot is untouched
        for b in range(nb):
            for p in range(bs):
                if not written[b, p]:
                    assert np.array_equal(caches[l][b, :, p], before[l][b, :, p])
        changed = np.any(caches[l] != before[l], axis=-1)   # [nb, H, bs]
        assert changed.sum() == H * int(np.sum(slots[l] >= 0))


def test_knorm_constant_and_one_hot_heads(orc):
    H, L, T = 2, 1, 4
    kv = np.zeros((L, T, 2 * H * HD), dtype=np.uint16)
    # row 0: head 0 constant 3.0, head 1 constant -0.5 -> +-1/sqrt(1 + eps/a^2) -> +-1
    kv[0, 0, :HD] = bf16_bits([3.0])[0]
    kv[0, 0, HD:2 * HD] = bf16_bits([-0.5])[0]
    # row 1: one-hot a=1 at element 9 of head 0 -> a / sqrt(a^2/64 + eps) = 7.99974 -> 8
    kv[0, 1, 9] = 0x3F80
    # row 2: one-hot a=-2 at element 62 of head 1 -> -8
    kv[0, 2, HD + 62] = bf16_bits([-2.0])[0]
    slots = [np.arange(T, dtype=np.int64)]
    caches = _caches(L, 1, H, 4)
    _store(orc, kv, H, None, slots, None, caches)
    c = caches[0][0]
    assert np.all(c[0, 0, :HD] == 0x3F80) and np.all(c[1, 0, :HD] == 0xBF80)
    exp = np.zeros(HD, dtype=np.uint16)
    exp[9] = bf16_bits([1.0 / np.sqrt(1.0 / 64 + 1e-6)])[0]
    assert exp[9] == bf16_bits([8.0])[0]
    assert np.array_equal(c[0, 1, :HD], exp)
    exp = np.zeros(HD, dtype=np.uint16)
    exp[62] = bf16_bits([-8.0])[0]
    assert np.array_equal(c[1, 2, :HD], exp)
    # row 3: all zero -> zero key
    assert np.all(c[:, 3, :HD] == 0)


def test_knorm_unit_mean_square(orc):
    rng = np.random.default_rng(3)
    H, L, T = 8, 1, 64
    kv = rnd_bf16(rng, (L, T, 2 * H * HD), 0.7)
    slots = [np.arange(T, dtype=np.int64)]
    caches = _caches(L, 4, H, 16)
    _store(orc, kv, H, None, slots, None, caches)
    k = to_f64(np.concatenate([caches[0][b, :, :, :HD] for b in range(4)], axis=1))
    ms = np.mean(k ** 2, axis=-1)
    assert np.all(np.abs(ms - 1.0) <= 2.0 ** -7)


def _table(max_pos, cos, sin):
    tab = np.zeros((max_pos, HD), dtype=np.uint16)
    tab[:, :32] = bf16_bits(cos)
    tab[:, 32:] = bf16_bits(sin)
    return tab


def test_rope_identity_quarter_turn_and_norm(orc):
    rng = np.random.default_rng(4)
    H, L, T = 4, 1, 3
    kv = rnd_bf16(rng, (L, T, 2 * H * HD))
    slots = [np.arange(T, dtype=np.int64)]
    plain = _caches(L, 1, H, 4)
    _store(orc, kv, H, None, slots, None, plain)
    # table row 0: cos 1, sin 0 -> identity (values; the sign of a zero may flip)
    # table row 1: cos 0, sin 1 -> (x, y) -> (-y, x) exactly
    # table row 2: a generic angle per pair
    ang = rng.uniform(0, 2 * np.pi, 32)
    tab = np.zeros((3, HD), dtype=np.uint16)
    tab[0] = _table(1, np.ones(32), np.zeros(32))[0]
    tab[1] = _table(1, np.zeros(32), np.ones(32))[0]
    tab[2] = _table(1, np.cos(ang), np.sin(ang))[0]
    positions = np.array([0, 1, 2], dtype=np.int64)
    roped = _caches(L, 1, H, 4)
    _store(orc, kv, H, positions, slots, tab, roped)
    n = to_f64(plain[0][0, :, :, :HD])          # [H, page, 64]
    r = to_f64(roped[0][0, :, :, :HD])
    assert np.array_equal(r[:, 0], n[:, 0])
    assert np.array_equal(r[:, 1, 0::2], -n[:, 1, 1::2])
    assert np.array_equal(r[:, 1, 1::2], n[:, 1, 0::2])
    c, s = to_f64(tab[2, :32]), to_f64(tab[2, 32:])
    pn = n[:, 2, 0::2] ** 2 + n[:, 2, 1::2] ** 2
    pr = r[:, 2, 0::2] ** 2 + r[:, 2, 1::2] ** 2
    assert np.all(np.abs(pr - (c ** 2 + s ** 2) * pn) <= 4 * 2.0 ** -8 * pn + 1e-30)
    # V is never rotated
    assert np.array_equal(roped[0][..., HD:], plain[0][..., HD:])


def test_rope_follows_each_rows_position(orc):
    # the rotation of row t comes from table row positions[t], not from t:
    # positions [1, 2, 0] give row 0 the quarter turn and row 2 the identity;
    # and permuting the rows with their positions and slots stores the same
    # cache bits
    rng = np.random.default_rng(14)
    H, L, T = 2, 1, 3
    kv = rnd_bf16(rng, (L, T, 2 * H * HD))
    slots = [np.arange(T, dtype=np.int64)]
    plain = _caches(L, 1, H, 4)
    _store(orc, kv, H, None, slots, None, plain)
    ang = rng.uniform(0, 2 * np.pi, 32)
    tab = np.zeros((3, HD), dtype=np.uint16)
    tab[0] = _table(1, np.ones(32), np.zeros(32))[0]
    tab[1] = _table(1, np.zeros(32), np.ones(32))[0]
    tab[2] = _table(1, np.cos(ang), np.sin(ang))[0]
    positions = np.array([1, 2, 0], dtype=np.int64)
    roped = _caches(L, 1, H, 4)
    _store(orc, kv, H, positions, slots, tab, roped)
    n = to_f64(plain[0][0, :, :, :HD])
    r = to_f64(roped[0][0, :, :, :HD])
    assert np.array_equal(r[:, 0, 0::2], -n[:, 0, 1::2]) and np.array_equal(r[:, 0, 1::2], n[:, 0, 0::2])
    assert np.array_equal(r[:, 2], n[:, 2])
    perm = np.array([2, 0, 1])
    again = _caches(L, 1, H, 4)
    _store(orc, np.ascontiguousarray(kv[:, perm]), H, positions[perm], [slots[0][perm]], tab, again)
    assert np.array_equal(again[0], roped[0])


def test_store_separate_k_and_v_strides(orc):
    # K from a packed [L, T, 64H] buffer and V from the middle third of a
    # [L, T, 192H] buffer (different row and layer strides) store the same
    # cache bits as the [K | V] rows of the projection
    rng = np.random.default_rng(15)
    H, L, T, P = 2, 2, 5, 4
    kv = rnd_bf16(rng, (L, T, 2 * H * HD))
    slots = [rng.permutation(8)[:T].astype(np.int64) for _ in range(L)]
    positions = rng.integers(0, P, T).astype(np.int64)
    inv = 10000.0 ** (-np.arange(32) / 32.0)
    tab = np.concatenate([_table(1, np.cos(p * inv), np.sin(p * inv)) for p in range(P)])
    ref = _caches(L, 2, H, 4)
    assert _store(orc, kv, H, positions, slots, tab, ref) == 0
    k = np.ascontiguousarray(kv[..., :H * HD]).reshape(-1)
    wide = np.zeros((L, T, 3 * H * HD), dtype=np.uint16)
    wide[..., H * HD:2 * H * HD] = kv[..., H * HD:]
    v = wide.reshape(-1)[H * HD:]
    got = _caches(L, 2, H, 4)
    err = orc.kv_store(k, v, T * H * HD, H * HD, T * 3 * H * HD, 3 * H * HD, positions, slots,
                       tab, got, H, 1e-6, T)
    assert err == 0
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)


def test_rope_reads_cos_then_sin_per_pair(orc):
    # pair j gets cos from column j and sin from column 32 + j: a table whose
    # pair j rotates by a quarter turn only for even j tells them apart
    H, L, T = 1, 1, 1
    kv = np.zeros((L, T, 2 * H * HD), dtype=np.uint16)
    kv[0, 0, :HD] = bf16_bits(np.arange(1, HD + 1) / 16.0)
    slots = [np.zeros(1, dtype=np.int64)]
    plain = _caches(L, 1, H, 1)
    _store(orc, kv, H, None, slots, None, plain)
    even = (np.arange(32) % 2 == 0)
    tab = _table(1, np.where(even, 0.0, 1.0), np.where(even, 1.0, 0.0))
    roped = _caches(L, 1, H, 1)
    _store(orc, kv, H, np.zeros(1, dtype=np.int64), slots, tab, roped)
    n = to_f64(plain[0][0, 0, 0, :HD]).reshape(32, 2)
    r = to_f64(roped[0][0, 0, 0, :HD]).reshape(32, 2)
    assert np.array_equal(r[even, 0], -n[even, 1]) and np.array_equal(r[even, 1], n[even, 0])
    assert np.array_equal(r[~even], n[~even])


def test_rope_scalar_closed_forms(orc):
    assert orc.rope(3.0, 5.0, 0.0, 1.0) == (np.float32(-5.0), np.float32(3.0))
    assert orc.rope(3.0, 5.0, 1.0, 0.0) == (np.float32(3.0), np.float32(5.0))
    # a rotation by pi: (x, y) -> (-x, -y)
    assert orc.rope(0.75, -2.5, -1.0, 0.0) == (np.float32(-0.75), np.float32(2.5))


def test_rope_uses_fused_multiply_adds(orc):
    # x' = fma(x, c, -(y s)) and y' = fma(y, c, x s): x c enters unrounded.
    # For random pairs where rounding x c (or y c) first changes the float32
    # result, the oracle gives the fused one, computed here exactly.
    from fractions import Fraction
    rng = np.random.default_rng(22)
    n = 4096
    x, y, c, s = (rng.uniform(0.5, 2.0, n).astype(np.float32) for _ in range(4))
    f64 = lambda a: a.astype(np.float64)
    ys, xs = (f64(y) * f64(s)).astype(np.float32), (f64(x) * f64(s)).astype(np.float32)
    ex, ey = f64(x) * f64(c) - f64(ys), f64(y) * f64(c) + f64(xs)    # exact (checked below)
    fused_x, fused_y = ex.astype(np.float32), ey.astype(np.float32)
    split_x, split_y = (x * c) - ys, (y * c) + xs
    hits = np.flatnonzero((fused_x != split_x) | (fused_y != split_y))
    assert len(hits) >= 20
    for i in hits[:20]:
        fr = lambda v: Fraction(float(v))
        assert fr(x[i]) * fr(c[i]) - fr(ys[i]) == Fraction(float(ex[i]))
        assert fr(y[i]) * fr(c[i]) + fr(xs[i]) == Fraction(float(ey[i]))
        assert orc.rope(x[i], y[i], c[i], s[i]) == (fused_x[i], fused_y[i])


def test_out_of_range_rows_are_counted_not_written(orc):
    rng = np.random.default_rng(5)
    H, L, T, nb, bs = 2, 2, 5, 2, 4
    kv = rnd_bf16(rng, (L, T, 2 * H * HD))
    slots = [np.array([0, 8, 100, -1, 7], dtype=np.int64),     # 8 and 100 >= nb*bs
             np.array([1, 2, 3, 4, 5], dtype=np.int64)]
    positions = np.array([0, 1, 2, 3, 99], dtype=np.int64)      # 99 >= max_position
    tab = _table(4, np.ones((4, 32)), np.zeros((4, 32)))
    caches = _caches(L, nb, H, bs)
    before = [c.copy() for c in caches]
    err = _store(orc, kv, H, positions, slots, tab, caches)
    # layer 0: slots 8, 100 out of range, row 4 position out of range -> 3
    # layer 1: row 4 position out of range -> 1
    assert err == 4
    assert np.array_equal(caches[0][1, :, 3], before[0][1, :, 3])     # slot 7 (row 4) not written
    assert np.array_equal(caches[1][1, :, 1], before[1][1, :, 1])     # slot 5 (row 4) not written
    assert not np.array_equal(caches[1][0, :, 1], before[1][0, :, 1])  # slot 1 written


def test_rows_prefix_and_skipped_layer(orc):
    rng = np.random.default_rng(6)
    H, L, T = 2, 3, 6
    kv = rnd_bf16(rng, (L, T, 2 * H * HD))
    slots = [np.arange(T, dtype=np.int64), None, np.arange(T, dtype=np.int64)[::-1].copy()]
    caches = _caches(L, 1, H, 8)
    before = [c.copy() for c in caches]
    _store(orc, kv, H, None, slots, None, caches, rows=4)
    assert np.array_equal(caches[1], before[1])                    # no slots: untouched
    changed0 = np.any(caches[0] != before[0], axis=-1)[0, 0]       # pages of layer 0
    assert list(np.nonzero(changed0)[0]) == [0, 1, 2, 3]
    changed2 = np.any(caches[2] != before[2], axis=-1)[0, 0]
    assert list(np.nonzero(changed2)[0]) == [2, 3, 4, 5]
