"""Pins of the oracle's decode QKV front (the page "...runtime.draft":
_fused_qkv_projection, _attention's split of its output into [Q | K | V |
O-gate], may_fuse_qkv_front; the per-head norm and RoPE are the context
K-norm's, pinned in test_oracle_project_store).

Expected values: constant heads norm to +-1 exactly (closed form), a table
row with cos = 0.75 and sin = 0.5 rotates (1, 1) to (0.25, 1.25) exactly,
V and the gate are bit copies, and the cache holds exactly the rows whose
slot is valid (sentinel elsewhere).
"""
import numpy as np
import torch

SENT = 0x5A5A


def bf16_bits(vals) -> np.ndarray:
    t = torch.tensor(np.asarray(vals, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_of(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def constant_heads(rng, M, nh, nkv):
    """Raw rows whose every 64-wide head is one constant (sign random,
    magnitude in [0.5, 4)); returns (raw bits, per-head constants)."""
    heads = 2 * nh + 2 * nkv
    c = rng.uniform(0.5, 4.0, (M, heads)) * rng.choice([-1.0, 1.0], (M, heads))
    cb = bf16_of(bf16_bits(c))
    raw = bf16_bits(np.repeat(cb, 64, axis=1))
    return raw, cb


def table(rows, c=0.75, s=0.5):
    t = np.zeros((rows, 64), dtype=np.uint16)
    t[:, :32] = bf16_bits([1.0])[0]              # row 0..: cos 1, sin 0 (identity)
    t[1, :32] = bf16_bits([c])[0]
    t[1, 32:] = bf16_bits([s])[0]
    return t


def test_routing_norm_and_rope(orc):
    rng = np.random.default_rng(1)
    M, nh, nkv = 4, 3, 2
    raw, cb = constant_heads(rng, M, nh, nkv)
    pos = np.array([0, 1, 1, 0], dtype=np.int64)
    cs = table(8)
    out, err = orc.qkv_front_post(raw, nh, nkv, pos, cs, None, None, 1e-6)
    assert err == 0
    sign = np.sign(cb)
    for m in range(M):
        for h in range(nh + nkv):                  # Q heads, then K heads
            head = bf16_of(out[m, 64 * h:64 * (h + 1)])
            if pos[m] == 0:
                assert np.all(head == sign[m, h])
            else:
                # (n0, n1) = (s, s), s = +-1: (fma(s, .75, -(s*.5)), fma(s, .75, s*.5))
                assert np.all(head[0::2] == 0.25 * sign[m, h])
                assert np.all(head[1::2] == 1.25 * sign[m, h])
    # V and the gate: bit copies
    q, kv = 64 * nh, 64 * nkv
    assert np.array_equal(out[:, q + kv:], raw[:, q + kv:])


def test_no_table_is_norm_only(orc):
    rng = np.random.default_rng(2)
    raw, cb = constant_heads(rng, 2, 1, 1)
    out, err = orc.qkv_front_post(raw, 1, 1, None, None, None, None, 1e-6)
    assert err == 0
    for h in range(2):
        assert np.all(bf16_of(out[:, 64 * h:64 * (h + 1)]) == np.sign(cb[:, h])[:, None])


def test_cache_insert_and_skips(orc):
    rng = np.random.default_rng(3)
    M, nh, nkv, nb, bs = 7, 2, 4, 3, 4
    raw = bf16_bits(rng.standard_normal((M, 64 * (2 * nh + 2 * nkv))))
    # row 3: slot past the cache (12); row 4: position past the table; row 6: both
    pos = np.array([0, 1, 2, 3, 99, 5, 100], dtype=np.int64)
    slots = np.array([7, -1, 0, 12, 3, 11, 13], dtype=np.int64)
    cs = table(8)
    cache = np.full((nb, nkv, bs, 128), SENT, dtype=np.uint16)
    out, err = orc.qkv_front_post(raw, nh, nkv, pos, cs, slots, cache, 1e-5)
    assert err == 3                                # one per bad row: 3, 4 and 6
    q, kv = 64 * nh, 64 * nkv
    written = {}
    for m in (0, 2, 5):                            # valid slots
        s = slots[m]
        written[s] = m
        for h in range(nkv):
            entry = cache[s // bs, h, s % bs]
            assert np.array_equal(entry[:64], out[m, q + 64 * h:q + 64 * (h + 1)])
            assert np.array_equal(entry[64:], raw[m, q + kv + 64 * h:q + kv + 64 * (h + 1)])
    for s in range(nb * bs):
        if s not in written:
            assert np.all(cache[s // bs, :, s % bs] == SENT)
    # row 4 (bad position): Q and K normed, not rotated -> same as with no table
    ref, _ = orc.qkv_front_post(raw[4:5].copy(), nh, nkv, None, None, None, None, 1e-5)
    assert np.array_equal(out[4], ref[0])
    # rows with a valid position are rotated (differ from the unrotated norm)
    ref1, _ = orc.qkv_front_post(raw[1:2].copy(), nh, nkv, None, None, None, None, 1e-5)
    assert not np.array_equal(out[1, :q + kv], ref1[0, :q + kv])


def test_projection_against_numpy(orc):
    # the float64 projection equals a library float64 matmul to rounding
    rng = np.random.default_rng(4)
    M, D, N = 5, 256, 384
    h = bf16_bits(rng.standard_normal((M, D)))
    W = bf16_bits(0.02 * rng.standard_normal((N, D)))
    got, ab = orc.qkv_project(h, W)
    ref = bf16_of(h).astype(np.float64) @ bf16_of(W).astype(np.float64).T
    assert np.all(np.abs(got - ref) <= 1e-12 * ab + 1e-300)
    assert np.allclose(ab, np.abs(bf16_of(h).astype(np.float64)) @ np.abs(bf16_of(W).astype(np.float64)).T)
