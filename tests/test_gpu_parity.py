"""CUDA path vs the oracle, element by element, through the C ABI.

Norms and store are bit-exact (the store fed the GPU's own projection, the
whole sentinel-filled cache compared); the projection is within the 2-ulp
rule of tests/parity.py.  Small fuzz shapes span several tiles with ragged
tails; the five workloads run at full size (projection checked on sampled
rows beyond the first two).
"""
import numpy as np
import pytest
import torch

import oracle
import rope_chain_gb300 as rc
import workloads
from tests import parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    from rope_chain_gb300 import _build
    _build.build()
    oracle.build()
    rc.read_device_faults(clear=True)
    yield
    assert rc.read_device_faults(clear=True) == 0, "a projection wait timed out"


def bits_to_dev(a):
    return parity.dev_bf16(a, DEV)


# ------------------------------------------------------------------ norms

@pytest.mark.parametrize("T,L,hw,pw", [(1, 1, True, True), (3, 2, False, True),
                                       (129, 3, True, False), (257, 9, False, False)])
def test_norms_bit_exact(T, L, hw, pw):
    case = workloads.random_case(100 + T, T=T, L=L, H=1, hidden_weighted=hw, pre_weighted=pw,
                                 num_blocks=32, block_size=16)
    x = bits_to_dev(case["x"])
    out = rc.context_norms(x, bits_to_dev(case["hidden_w"]), bits_to_dev(case["pre_w"]), L, 1e-5)
    ref = oracle.context_norms(case["x"], case["hidden_w"], case["pre_w"], L, 1e-5)
    assert np.array_equal(parity.host_bits(out), ref)


def test_norms_special_values():
    rng = np.random.default_rng(3)
    x = workloads.normal_bf16(rng, (6, 8192), 0.0, 1.0)
    x[0] = 0                                   # zero row
    x[1, ::2] = 0x8000                         # -0.0 entries
    x[2, ::7] = rng.integers(1, 128, x[2, ::7].shape).astype(np.uint16)   # subnormals
    x[3] = rng.integers(1, 128, 8192).astype(np.uint16) | 0x8000           # all subnormal
    x[4] = workloads.to_bf16_bits(np.full(8192, 3.0e38, np.float32))       # huge: sum overflows
    x[5, 17] = 0x4580                          # one large entry
    hw = workloads.normal_bf16(rng, (8192,), 1.0, 0.1)
    pw = workloads.normal_bf16(rng, (2, 8192), 1.0, 0.1)
    for eps in (1e-6, 0.0):
        out = rc.context_norms(bits_to_dev(x), bits_to_dev(hw), bits_to_dev(pw), 2, eps)
        ref = oracle.context_norms(x, hw, pw, 2, eps)
        got = parity.host_bits(out)
        finite = (ref & 0x7F80) != 0x7F80
        assert np.array_equal(got[finite], ref[finite])
        # NaN results (the row of 3e38 with eps=0 overflows): both sides NaN
        nan_ref = ((ref & 0x7F80) == 0x7F80) & ((ref & 0x7F) != 0)
        nan_got = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
        assert np.array_equal(nan_ref, nan_got)


def test_norms_nan_encoding():
    """Reading R4: which bf16 NaN the GPU's conversion produces."""
    x = np.zeros((1, 8192), dtype=np.uint16)
    x[0, 5] = 0x7FC0                             # a NaN input makes the whole row NaN
    out = parity.host_bits(rc.context_norms(bits_to_dev(x), None, None, 1, 1e-6))
    ref = oracle.context_norms(x, None, None, 1, 1e-6)
    assert np.array_equal(out, ref), (hex(out[0, 0, 0]), hex(ref[0, 0, 0]))


# ------------------------------------------------------------- projection

@pytest.mark.parametrize("T,L,D,H", [(1, 1, 8192, 8), (100, 2, 512, 1), (129, 1, 1024, 2),
                                     (300, 2, 8192, 16), (64, 3, 8192, 8)])
@pytest.mark.parametrize("layout", [rc.RC_W_KN, rc.RC_W_NK])
@pytest.mark.parametrize("split", [True, False])
def test_projection_within_two_ulp(T, L, D, H, layout, split):
    rng = np.random.default_rng(T * 7 + L)
    N = 128 * H
    a = workloads.normal_bf16(rng, (L, T, D), 0.0, 1.0)
    W = workloads.normal_bf16(rng, (L, D, N), 0.0, 0.02)
    Wl = W if layout == rc.RC_W_KN else np.ascontiguousarray(W.transpose(0, 2, 1))
    ws = None
    if split:
        nbytes = rc.workspace_size(L, T, D, N)
        ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=DEV)
    out = rc.kv_project(bits_to_dev(a), bits_to_dev(Wl), w_layout=layout, workspace=ws)
    ref, ab = oracle.kv_project(a, W)
    parity.assert_projection_close(parity.host_bits(out), ref, ab)


@pytest.mark.parametrize("L,T,H,layout", [(3, 100, 1, rc.RC_W_KN),    # single CTA, workspace
                                           (3, 512, 8, rc.RC_W_NK),    # CTA pairs, cluster split-K
                                           (1, 64, 8, rc.RC_W_KN)])    # single CTA, 16 splits
def test_projection_repeated_calls_identical(L, T, H, layout):
    # one workspace (when the plan uses one), three calls in a row: identical
    # results within the 2-ulp rule, i.e. nothing a call leaves behind
    # changes the next one
    rng = np.random.default_rng(21 + T)
    D, N = 8192, 128 * H
    a = workloads.normal_bf16(rng, (L, T, D), 0.0, 1.0)
    W = workloads.normal_bf16(rng, (L, D, N), 0.0, 0.02)
    Wl = W if layout == rc.RC_W_KN else np.ascontiguousarray(W.transpose(0, 2, 1))
    ws = rc.new_workspace(L, T, D, N, DEV)
    a_d, w_d = bits_to_dev(a), bits_to_dev(Wl)
    ref, ab = oracle.kv_project(a, W)
    outs = [parity.host_bits(rc.kv_project(a_d, w_d, w_layout=layout, workspace=ws))
            for _ in range(3)]
    parity.assert_projection_close(outs[0], ref, ab)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_projection_one_hot_is_exact():
    # W selects one input column per output: every product but one is zero,
    # so the tensor-core result is exact whatever the summation order
    rng = np.random.default_rng(8)
    L, T, D, N = 2, 200, 8192, 256
    a = workloads.normal_bf16(rng, (L, T, D), 0.0, 1.0)
    perm = rng.integers(0, D, size=(L, N))
    W = np.zeros((L, D, N), dtype=np.uint16)
    for l in range(L):
        W[l, perm[l], np.arange(N)] = 0x3F80
    for layout in (rc.RC_W_KN, rc.RC_W_NK):
        Wl = W if layout == rc.RC_W_KN else np.ascontiguousarray(W.transpose(0, 2, 1))
        nbytes = rc.workspace_size(L, T, D, N)
        ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=DEV)
        out = parity.host_bits(rc.kv_project(bits_to_dev(a), bits_to_dev(Wl), w_layout=layout,
                                             workspace=ws))
        for l in range(L):
            assert np.array_equal(out[l], a[l][:, perm[l]])


# ------------------------------------------------------------------ store

@pytest.mark.parametrize("H", [1, 2, 4, 8, 16, 32])
@pytest.mark.parametrize("rope", [True, False])
def test_store_bit_exact_all_heads(H, rope):
    L, T = 2, 70
    case = workloads.random_case(200 + H, T=T, L=L, H=H, rope=rope, max_position=128,
                                 num_blocks=8, block_size=16)
    rng = np.random.default_rng(H)
    kv = workloads.normal_bf16(rng, (L, T, 128 * H), 0.0, 0.5)
    _compare_store(case, kv, rows=T)


def _compare_store(case, kv, rows, slots=None):
    L, T, N = kv.shape
    H = N // 128
    slots = case["slots"] if slots is None else slots
    caches_d = [bits_to_dev(c) for c in parity.make_caches(case, L, parity.SENTINEL)]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    rc.kv_store_from_projection(bits_to_dev(kv), H, torch.from_numpy(case["positions"]).to(DEV),
                                [None if s is None else torch.from_numpy(s).to(DEV) for s in slots],
                                bits_to_dev(case["cos_sin"]), caches_d, case["eps"], rows=rows,
                                err=err)
    caches = parity.make_caches(case, L, parity.SENTINEL)
    e = oracle.kv_store_from_projection(kv, H, case["positions"], slots, case["cos_sin"], caches,
                                        case["eps"], rows)
    for g, r in zip(caches_d, caches):
        assert np.array_equal(parity.host_bits(g), r)
    assert int(err.item()) == e
    return e


@pytest.mark.parametrize("H", [1, 8, 32])
@pytest.mark.parametrize("rope", [True, False])
def test_store_unaligned_views(H, rope):
    """K and V views that are only 4-byte aligned (row stride 128 H + 6
    elements, K starting 2 elements in) take the lane-per-pair kernel; the
    aligned views of the other store tests take the lane-per-head kernel.
    Both must write the oracle's bits."""
    L, T = 2, 45
    case = workloads.random_case(260 + H, T=T, L=L, H=H, rope=rope, max_position=96,
                                 num_blocks=8, block_size=16)
    rng = np.random.default_rng(31 + H)
    kv = workloads.normal_bf16(rng, (L, T, 128 * H), 0.0, 0.7)
    buf = np.zeros((L, T, 128 * H + 6), dtype=np.uint16)
    buf[:, :, 2:2 + 128 * H] = kv
    bd = bits_to_dev(buf)
    k = bd[:, :, 2:2 + 64 * H].unflatten(2, (H, 64))
    v = bd[:, :, 2 + 64 * H:2 + 128 * H].unflatten(2, (H, 64))
    assert k.data_ptr() % 16 != 0
    caches_d = [bits_to_dev(c) for c in parity.make_caches(case, L, parity.SENTINEL)]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots = case["slots"]
    rc.kv_store(k, v, torch.from_numpy(case["positions"]).to(DEV),
                [torch.from_numpy(s).to(DEV) for s in slots], bits_to_dev(case["cos_sin"]),
                caches_d, case["eps"], rows=T, err=err)
    caches = parity.make_caches(case, L, parity.SENTINEL)
    e = oracle.kv_store_from_projection(kv, H, case["positions"], slots, case["cos_sin"], caches,
                                        case["eps"], T)
    for g, r in zip(caches_d, caches):
        assert np.array_equal(parity.host_bits(g), r)
    assert int(err.item()) == e


@pytest.mark.parametrize("L", [9, 17])
def test_store_layer_chunks_null_layers_and_rows_prefix(L):
    T, H = 50, 4
    case = workloads.random_case(300 + L, T=T, L=L, H=H, max_position=64, num_blocks=4,
                                 block_size=16)
    slots = list(case["slots"])
    slots[3] = None
    slots[L - 1] = None
    rng = np.random.default_rng(L)
    kv = workloads.normal_bf16(rng, (L, T, 128 * H), 0.0, 1.0)
    _compare_store(case, kv, rows=37, slots=slots)


def test_store_out_of_range_rows_counted():
    T, H, L = 40, 8, 2
    case = workloads.random_case(400, T=T, L=L, H=H, max_position=32, num_blocks=4, block_size=16)
    slots = [s.copy() for s in case["slots"]]
    slots[0][3] = 64             # == capacity
    slots[0][4] = 1 << 40        # far past the cache
    slots[1][5] = -(1 << 62)     # negative: plain skip
    pos = case["positions"].copy()
    pos[7] = 32                  # == max_position
    pos[8] = -3
    case = dict(case, positions=pos)
    rng = np.random.default_rng(4)
    kv = workloads.normal_bf16(rng, (L, T, 128 * H), 0.0, 1.0)
    e = _compare_store(case, kv, rows=T, slots=slots)
    assert e >= 2
