"""The norm variants (rc_context_norms_ex) and per-layer row counts
(rc_kv_store_rows, rc_kv_project_store_rows) against the oracle.

Norms: bit-exact over every element for every combination of weight dtype
(none, bf16, FP32) and scale side per norm, with and without gain centers,
with separate hidden and layer eps.  Stores: the whole caches bit-exact
against the oracle's store fed the same projection, layer l inserting its
first rows_l rows.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
import rope_chain_gb300 as rc
import workloads
from tests import parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
D = 8192


@pytest.fixture(scope="module", autouse=True)
def built():
    from rope_chain_gb300 import _build
    _build.build()
    oracle.build()
    rc.read_device_faults(clear=True)
    yield
    assert rc.read_device_faults(clear=True) == 0


def _weight(rng, kind, shape):
    if kind == "none":
        return None
    vals = 1 + 0.1 * rng.standard_normal(shape)
    if kind == "bf16":
        return workloads.to_bf16_bits(vals.astype(np.float32))
    return vals.astype(np.float32)          # FP32 bits below bf16 precision included


def _dev_w(w):
    if w is None:
        return None
    if w.dtype == np.uint16:
        return parity.dev_bf16(w, DEV)
    return torch.from_numpy(w).to(DEV)


NORM_KINDS = [("none", False), ("bf16", False), ("bf16", True), ("f32", False), ("f32", True)]


@pytest.mark.parametrize("hidden,pre", list(itertools.product(NORM_KINDS, NORM_KINDS)))
def test_norm_variants_bit_exact(hidden, pre):
    (hk, hin), (pk, pin) = hidden, pre
    seed = 100 + 10 * NORM_KINDS.index(hidden) + NORM_KINDS.index(pre)
    rng = np.random.default_rng(seed)
    T, L = 37, 3
    x = workloads.to_bf16_bits((rng.standard_normal((T, D)) * 1.5).astype(np.float32))
    hw = _weight(rng, hk, (D,))
    pw = _weight(rng, pk, (L, D))
    centered = seed % 2 == 1
    kw = dict(hidden_eps=1e-5, pre_eps=3e-4,
              hidden_center=0.5 if centered else 0.0, pre_center=-0.25 if centered else 0.0,
              hidden_input_scale=hin, pre_input_scale=pin)
    ref = oracle.context_norms_ex(x, L, hidden_w=hw, pre_w=pw, **kw)
    out = rc.context_norms_ex(parity.dev_bf16(x, DEV), L, hidden_w=_dev_w(hw), pre_w=_dev_w(pw),
                              **kw)
    torch.cuda.synchronize()
    got = parity.host_bits(out)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} elements differ"


@pytest.mark.parametrize("T,L", [(1, 1), (129, 9), (300, 2)])
def test_norm_variants_shapes(T, L):
    rng = np.random.default_rng(T + L)
    x = workloads.to_bf16_bits((rng.standard_normal((T, D)) * 2).astype(np.float32))
    hw = _weight(rng, "f32", (D,))
    pw = _weight(rng, "bf16", (L, D))
    kw = dict(hidden_eps=1e-6, pre_eps=1e-5, pre_center=1.0, hidden_input_scale=True,
              pre_input_scale=True)
    ref = oracle.context_norms_ex(x, L, hidden_w=hw, pre_w=pw, **kw)
    out = rc.context_norms_ex(parity.dev_bf16(x, DEV), L, hidden_w=_dev_w(hw), pre_w=_dev_w(pw),
                              **kw)
    torch.cuda.synchronize()
    assert np.array_equal(parity.host_bits(out), ref)


@pytest.mark.parametrize("T", [4099, 16387])
@pytest.mark.parametrize("hidden,pre,center", [
    (("f32", True), ("f32", False), 1.0),     # one r for every layer, FP32 gains staged
    (("bf16", False), ("f32", True), 0.0),    # input-scale layer weight: r per layer
    (("none", False), ("bf16", False), -0.5),
    (("none", False), ("none", False), 0.0),
])
def test_norm_variants_many_rows(T, hidden, pre, center):
    # row counts that take the kernels holding several rows per CTA (odd,
    # and 3 mod 4: the last CTA is ragged)
    (hk, hin), (pk, pin) = hidden, pre
    rng = np.random.default_rng(T + int(8 * center))
    L = 3
    x = workloads.to_bf16_bits(rng.standard_normal((T, D)).astype(np.float32))
    hw = _weight(rng, hk, (D,))
    pw = _weight(rng, pk, (L, D))
    kw = dict(hidden_eps=1e-6, pre_eps=1e-5, pre_center=center, hidden_input_scale=hin,
              pre_input_scale=pin)
    ref = oracle.context_norms_ex(x, L, hidden_w=hw, pre_w=pw, **kw)
    out = rc.context_norms_ex(parity.dev_bf16(x, DEV), L, hidden_w=_dev_w(hw), pre_w=_dev_w(pw),
                              **kw)
    torch.cuda.synchronize()
    got = parity.host_bits(out)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} elements differ"


def test_plain_options_equal_context_norms():
    # bf16 output-scale weights without a center and with one eps: the same
    # bits as rc_context_norms
    w = workloads.WORKLOADS[2]
    case = workloads.make_inputs(w)
    x = parity.dev_bf16(case["x"], DEV)
    hw, pw = parity.dev_bf16(case["hidden_w"], DEV), parity.dev_bf16(case["pre_w"], DEV)
    a = rc.context_norms(x, hw, pw, w.L, w.eps)
    b = rc.context_norms_ex(x, w.L, hidden_w=hw, pre_w=pw, hidden_eps=w.eps, pre_eps=w.eps)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_separate_eps_default_kernel():
    # bf16 output-scale weights and two eps values take the default kernel
    rng = np.random.default_rng(7)
    T, L = 64, 2
    x = workloads.to_bf16_bits(rng.standard_normal((T, D)).astype(np.float32) * 1e-3)
    hw = _weight(rng, "bf16", (D,))
    pw = _weight(rng, "bf16", (L, D))
    kw = dict(hidden_eps=1e-2, pre_eps=1e-7)      # eps large against the row's mean square
    ref = oracle.context_norms_ex(x, L, hidden_w=hw, pre_w=pw, **kw)
    out = rc.context_norms_ex(parity.dev_bf16(x, DEV), L, hidden_w=_dev_w(hw), pre_w=_dev_w(pw),
                              **kw)
    torch.cuda.synchronize()
    assert np.array_equal(parity.host_bits(out), ref)


def test_norm_variant_rejections():
    x = torch.zeros((4, D), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(TypeError):
        rc.context_norms_ex(x, 1, hidden_w=torch.ones(D, dtype=torch.float16, device=DEV),
                            hidden_eps=1e-6, pre_eps=1e-6)
    with pytest.raises(ValueError):
        rc.context_norms_ex(x, 2, pre_w=torch.ones((3, D), device=DEV), hidden_eps=1e-6,
                            pre_eps=1e-6)
    bad = torch.ones(D + 4, dtype=torch.float32, device=DEV)[2:]   # 8-byte aligned only
    h = rc._norm_params(bad, False, 0.0, 1e-6, "hidden_w")
    p = rc._norm_params(None, False, 0.0, 1e-6, "pre_w")
    import ctypes
    out = torch.empty((1, 4, D), dtype=torch.bfloat16, device=DEV)
    st = rc.lib().rc_context_norms_ex(x.data_ptr(), 4, D, ctypes.byref(h), ctypes.byref(p), 1,
                                      out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == rc.RC_ERR_INVALID_ARG


# ----------------------------------------------------------- slot lengths

def _store_case(seed, T, L, H, rows):
    case = workloads.random_case(seed, T=T, L=L, H=H, max_position=512,
                                 num_blocks=(T + 15) // 16 + 3, block_size=16)
    # each layer's slot mapping cut to its own length ([rt] _slot_groups)
    slots = [None if r is None else s[:r].copy() for s, r in zip(case["slots"], rows)]
    return dict(case, slots=slots)


def _oracle_caches(case, kv, rows):
    L = len(case["slots"])
    H = case["cache_shape"][1]
    ref = parity.make_caches(case, L, parity.SENTINEL)
    err = oracle.kv_store_from_projection(kv, H, case["positions"], case["slots"], case["cos_sin"],
                                          ref, case["eps"], [0 if r is None else r for r in rows])
    return ref, err


@pytest.mark.parametrize("T,L,H,rows", [
    (100, 4, 8, [100, 17, None, 0]),
    (300, 9, 2, [300, 299, 1, 150, 0, 64, 65, 300, 7]),     # two launches of <= 8 layers
    (64, 3, 32, [5, 64, 33]),
])
def test_store_per_layer_rows(T, L, H, rows):
    case = _store_case(31 + T + L, T, L, H, rows)
    rng = np.random.default_rng(T)
    kv = workloads.to_bf16_bits(rng.standard_normal((L, T, 128 * H)).astype(np.float32))
    caches = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    rc.kv_store_from_projection(parity.dev_bf16(kv, DEV), H, torch.from_numpy(case["positions"]).to(DEV),
                                [None if s is None else torch.from_numpy(s).to(DEV) for s in case["slots"]],
                                parity.dev_bf16(case["cos_sin"], DEV), caches, case["eps"], err=err)
    torch.cuda.synchronize()
    ref, ref_err = _oracle_caches(case, kv, rows)
    for g, r in zip(caches, ref):
        assert np.array_equal(parity.host_bits(g), r)
    assert int(err.item()) == ref_err


@pytest.mark.parametrize("T,L,H,workspace,rows", [
    (300, 3, 8, False, [300, 120, 0]),       # CTA pairs, epilogue store
    (300, 9, 2, False, [300, 299, 1, 150, 0, 64, 65, 300, 7]),   # persistent pairs, 9 layers
    (512, 3, 8, True, [1, 512, 400]),        # CTA pairs, split-K, reduce-and-store
    (100, 2, 1, False, [100, 3]),            # single CTAs: kv_out, then the store kernel
    (257, 10, 2, True, [257, 0, 5, 256, 100, 1, 2, 3, 250, 257]),
    # persistent pairs with a tail split (rows 512-999 of the last layer):
    # the last layer stores its first 700 rows, so the tail stores 188
    (1000, 10, 4, True, [1000, 999, 0, 500, 1000, 3, 1000, 256, 1000, 700]),
])
def test_project_store_per_layer_rows(T, L, H, workspace, rows):
    case = _store_case(77 + T + L, T, L, H, rows)
    normed = oracle.context_norms(case["x"], case["hidden_w"], case["pre_w"], L, case["eps"])
    kv = torch.empty((L, T, 128 * H), dtype=torch.bfloat16, device=DEV)
    caches = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = rc.new_workspace(L, T, D, 128 * H, DEV) if workspace else None
    rc.kv_project_store(parity.dev_bf16(normed, DEV), parity.dev_bf16(case["W"], DEV), H,
                        torch.from_numpy(case["positions"]).to(DEV),
                        [None if s is None else torch.from_numpy(s).to(DEV) for s in case["slots"]],
                        parity.dev_bf16(case["cos_sin"], DEV), caches, case["eps"], err=err,
                        kv_out=kv, workspace=ws)
    torch.cuda.synchronize()
    kv_h = parity.host_bits(kv)
    ref, ref_err = _oracle_caches(case, kv_h, rows)
    for g, r in zip(caches, ref):
        assert np.array_equal(parity.host_bits(g), r)
    assert int(err.item()) == ref_err
    ref64, ab = oracle.kv_project(normed, case["W"])
    parity.assert_projection_close(kv_h, ref64, ab)
