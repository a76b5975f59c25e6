"""The decode QKV front (rc_qkv_front) against the oracle: the projection
(raw_out) within the 2-ulp rule of the float64 sum, the output row and the
cache bit-exact against the oracle's front fed that projection, the skip
count equal.  Covers one CTA per column tile and the K split across a
cluster of two, 1 to 16 tokens, ragged small D, no table, no slots, and
out-of-range slots and positions."""
import numpy as np
import pytest
import torch

import oracle
import rope_chain_gb300 as rc
import workloads
from tests import parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SENT = 0x5A5A


@pytest.fixture(scope="module", autouse=True)
def built():
    from rope_chain_gb300 import _build
    _build.build()
    oracle.build()
    rc.read_device_faults(clear=True)
    yield
    assert rc.read_device_faults(clear=True) == 0


def make_case(seed, M, D, nh, nkv, *, rope=True, with_slots=True, nb=8, bs=16, max_pos=4096):
    rng = np.random.default_rng(seed)
    N = 64 * (2 * nh + 2 * nkv)
    hidden = workloads.to_bf16_bits(rng.standard_normal((M, D)).astype(np.float32))
    W = workloads.to_bf16_bits((0.02 * rng.standard_normal((N, D))).astype(np.float32))
    pos = rng.integers(0, max_pos, M).astype(np.int64)
    cs = workloads.cos_sin_table(max_pos) if rope else None
    slots = None
    if with_slots:
        slots = rng.permutation(nb * bs)[:M].astype(np.int64)
        slots[rng.random(M) < 0.2] = -1
    return dict(hidden=hidden, W=W, pos=pos, cs=cs, slots=slots, nh=nh, nkv=nkv, nb=nb, bs=bs,
                eps=1e-6)


def run(case, *, raw=True):
    M = case["hidden"].shape[0]
    N = case["W"].shape[0]
    cache = None
    if case["slots"] is not None:
        cache = parity.dev_bf16(np.full((case["nb"], case["nkv"], case["bs"], 128), SENT,
                                        dtype=np.uint16), DEV)
    raw_t = torch.empty((M, N), dtype=torch.bfloat16, device=DEV) if raw else None
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = rc.qkv_front(parity.dev_bf16(case["hidden"], DEV), parity.dev_bf16(case["W"], DEV),
                       case["nh"], case["nkv"], torch.from_numpy(case["pos"]).to(DEV),
                       parity.dev_bf16(case["cs"], DEV),
                       None if case["slots"] is None else torch.from_numpy(case["slots"]).to(DEV),
                       cache, case["eps"], raw_out=raw_t, err=err)
    torch.cuda.synchronize()
    return dict(out=parity.host_bits(out), raw=None if raw_t is None else parity.host_bits(raw_t),
                cache=None if cache is None else parity.host_bits(cache), err=int(err.item()))


def check(case, got):
    ref64, ab = oracle.qkv_project(case["hidden"], case["W"])
    parity.assert_projection_close(got["raw"], ref64, ab, what="QKV projection")
    cache = None
    if case["slots"] is not None:
        cache = np.full((case["nb"], case["nkv"], case["bs"], 128), SENT, dtype=np.uint16)
    out, err = oracle.qkv_front_post(got["raw"], case["nh"], case["nkv"],
                                     case["pos"] if case["cs"] is not None else None, case["cs"],
                                     case["slots"], cache, case["eps"])
    assert np.array_equal(got["out"], out)
    if cache is not None:
        assert np.array_equal(got["cache"], cache)
    assert got["err"] == err


@pytest.mark.parametrize("M,D,nh,nkv", [
    (1, 8192, 128, 8),       # 136 column tiles: one CTA each
    (16, 8192, 128, 8),
    (7, 8192, 8, 2),         # 10 tiles: K split over a cluster of two
    (3, 1024, 4, 4),
    (16, 128, 1, 1),         # two K blocks, one per CTA of the pair
    (5, 64, 2, 1),           # one K block: no split
    (12, 8192, 64, 8),
])
def test_front_against_oracle(M, D, nh, nkv):
    case = make_case(M * 1000 + nh + nkv + D, M, D, nh, nkv)
    got = run(case)
    check(case, got)
    # without raw_out the output and the cache are the same bits
    again = run(case, raw=False)
    assert np.array_equal(again["out"], got["out"])
    assert np.array_equal(again["cache"], got["cache"])


def test_front_no_table_no_slots():
    case = make_case(5, 9, 2048, 16, 4, rope=False, with_slots=False)
    check(case, run(case))


def test_front_bad_slots_and_positions():
    case = make_case(6, 8, 8192, 8, 2, nb=2, bs=16, max_pos=64)
    case["slots"][:] = np.arange(8)
    case["slots"][1] = 32            # == capacity
    case["slots"][2] = -5
    case["slots"][3] = 1 << 40
    case["pos"][4] = 64              # == max_position
    case["pos"][5] = -1
    got = run(case)
    assert got["err"] == 4
    check(case, got)


def test_front_repeatable():
    case = make_case(7, 16, 8192, 32, 8)
    a, b = run(case), run(case)
    for k in ("out", "raw", "cache"):
        assert np.array_equal(a[k], b[k])
