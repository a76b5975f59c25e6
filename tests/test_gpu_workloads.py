"""The five workloads at full size, in the launch configuration bench.py
times: the whole chain through the C ABI, compared with the oracle.

  * norms: every element, bit-exact;
  * projection: every row for workloads 1-2, a seeded sample of rows (with
    the first and last row, i.e. the ragged tail) for 3-5, 2-ulp rule;
  * store: the whole cache of every layer, bit-exact, the oracle fed the
    GPU's projection; the skip counter equal;
  * end to end on the sampled rows: V in the cache within the projection
    rule, K within 2 ulp of its pair's magnitude (see _check_end_to_end).
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
SAMPLE_ROWS = 256


@pytest.fixture(scope="module", autouse=True)
def built():
    from rope_chain_gb300 import _build
    _build.build()
    oracle.build()
    rc.read_device_faults(clear=True)
    yield
    assert rc.read_device_faults(clear=True) == 0


def _sample_rows(T, seed):
    if T <= 512:
        return None
    rng = np.random.default_rng(seed)
    rows = rng.choice(T, size=SAMPLE_ROWS - 2, replace=False)
    return np.unique(np.concatenate([[0, T - 1], rows])).astype(np.int64)


def _check_end_to_end(case, got, ref, rows):
    """K and V in the cache for the sampled rows, against the oracle store
    fed bf16(ref64).  K's tolerance: 2 ulp of the pair magnitude
    |(x', y')| of the oracle's result, or of what a projection error of the
    projection rule's size can move through the K-norm (r * tol_k)."""
    L = len(case["slots"])
    H = case["cache_shape"][1]
    T = case["x"].shape[0]
    rows = np.arange(T) if rows is None else rows
    kv_ref = oracle.bf16_rn_f64_array(ref["kv64"])               # [L, R, N]
    sub_slots = [s[rows].copy() for s in case["slots"]]
    sub = dict(case, slots=sub_slots, positions=case["positions"][rows].copy())
    caches = parity.make_caches(case, L, parity.SENTINEL)
    oracle.kv_store_from_projection(kv_ref, H, sub["positions"], sub_slots, case["cos_sin"],
                                    caches, case["eps"], len(rows))
    bs = case["cache_shape"][2]
    cap = case["cache_shape"][0] * bs
    worst_k = 0.0
    k_err, k_pair, k_tol, v_bits, v_ref, v_abs = [], [], [], [], [], []
    for l in range(L):
        for i, t in enumerate(rows):
            s = int(case["slots"][l][t])
            if s < 0 or s >= cap:
                continue
            b, p = divmod(s, bs)
            g = got["caches"][l][b, :, p]                      # [H, 128]
            r = caches[l][b, :, p]
            gk = (g[:, :64].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            rk = (r[:, :64].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            pair = np.sqrt(rk[:, 0::2] ** 2 + rk[:, 1::2] ** 2)
            pair = np.repeat(pair, 2, axis=1)
            # what the K-norm does to a projection error of the 2-ulp rule
            k64 = ref["kv64"][l, i, :64 * H].reshape(H, 64)
            kab = ref["kvabs"][l, i, :64 * H].reshape(H, 64)
            ktol = 2 * parity.ulp_bf16(np.maximum(np.abs(k64), 2.0 ** -12 * kab))
            rms = np.sqrt(np.mean(k64 ** 2, axis=1, keepdims=True) + case["eps"])
            scale = np.maximum(pair, np.repeat(
                np.sqrt((ktol[:, 0::2] / rms) ** 2 + (ktol[:, 1::2] / rms) ** 2), 2, axis=1))
            tol = 2 * parity.ulp_bf16(np.where(scale > 0, scale, 2.0 ** -133))
            err = np.abs(gk - rk)
            assert np.all(err <= tol), (l, t, float(np.max(err / tol)))
            worst_k = max(worst_k, float(np.max(err / tol)))
            k_err.append(err.reshape(-1))
            k_pair.append(pair.reshape(-1))
            k_tol.append(scale.reshape(-1))
            gv = g[:, 64:].reshape(-1)
            parity.assert_projection_close(gv, ref["kv64"][l, i, 64 * H:], ref["kvabs"][l, i, 64 * H:],
                                           what="end-to-end V")
            v_bits.append(gv)
            v_ref.append(ref["kv64"][l, i, 64 * H:])
            v_abs.append(ref["kvabs"][l, i, 64 * H:])
    if k_err:
        e = np.concatenate(k_err)
        k = parity.ulp_stats(e, np.concatenate(k_pair))
        k["at_rule_scale"] = parity.ulp_stats(e, np.concatenate(k_tol))
        v = parity.projection_ulp_stats(np.concatenate(v_bits), np.concatenate(v_ref),
                                        np.concatenate(v_abs))
        return worst_k, k, v
    return worst_k, None, None


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_workload_parity(index):
    w = workloads.WORKLOADS[index]
    case = workloads.make_inputs(w)
    got = parity.run_gpu_chain(case, DEV)
    ref_normed = oracle.context_norms(case["x"], case["hidden_w"], case["pre_w"], w.L, w.eps)
    assert np.array_equal(got["normed"], ref_normed), "norms"
    rows = _sample_rows(w.T, w.seed)
    ref = parity.run_oracle_chain(case, got["kv"], rows=rows, normed=ref_normed)
    kv_rows = got["kv"] if rows is None else got["kv"][:, rows]
    parity.assert_projection_close(kv_rows, ref["kv64"], ref["kvabs"])
    for l, (g, r) in enumerate(zip(got["caches"], ref["caches"])):
        assert np.array_equal(g, r), f"store, layer {l}"
    assert got["err"] == ref["err"] == 0
    _, k_stats, v_stats = _check_end_to_end(case, got, ref, rows)
    # the error itself, not only pass/fail: max ulps and a histogram per
    # workload for the projection and the end-to-end K and V
    parity.report(f"workload {index} projection",
                  parity.projection_ulp_stats(kv_rows, ref["kv64"], ref["kvabs"]))
    parity.report(f"workload {index} end-to-end K (ulps of the pair magnitude)", k_stats)
    parity.report(f"workload {index} end-to-end V", v_stats)


def test_workload_parity_nk_layout_and_no_workspace():
    # workload 2 with the nn.Linear weight layout and without split-K
    w = workloads.WORKLOADS[2]
    case = workloads.make_inputs(w)
    got = parity.run_gpu_chain(case, DEV, w_layout=rc.RC_W_NK, use_workspace=False)
    ref = parity.run_oracle_chain(case, got["kv"])
    assert np.array_equal(got["normed"], ref["normed"])
    parity.assert_projection_close(got["kv"], ref["kv64"], ref["kvabs"])
    for g, r in zip(got["caches"], ref["caches"]):
        assert np.array_equal(g, r)
