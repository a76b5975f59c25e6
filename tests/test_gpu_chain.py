"""rc_context_kv (the whole chain in one call, norms fused into the
projection) against the three-call chain and the oracle.

The projection's operand is formed in shared memory from the hidden-norm
output; it must equal rc_context_norms' output bit for bit, so with an equal
split plan kv_out is bit-identical to rc_kv_project's output and the caches
to the unfused chain's.  The caches are also compared bit-exactly with the
oracle's store fed kv_out, and kv_out with the oracle's projection of the
oracle's norms (2-ulp rule).
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
    assert rc.read_device_faults(clear=True) == 0


def run_whole(case, *, layout=rc.RC_W_KN, full_workspace=True):
    L = len(case["slots"])
    H = case["cache_shape"][1]
    T = case["x"].shape[0]
    W = case["W"] if layout == rc.RC_W_KN else np.ascontiguousarray(case["W"].transpose(0, 2, 1))
    ws = rc.context_kv_workspace(L, T, H, DEV)
    if not full_workspace:                      # only the fixed part: no split-K
        fixed = ((T * 8192 * 2 + 255) // 256) * 256 + ((T * 4 + 255) // 256) * 256
        ws = ws[:fixed]
    caches = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
    kv = torch.empty((L, T, 128 * H), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    rc.context_kv(parity.dev_bf16(case["x"], DEV), parity.dev_bf16(case["hidden_w"], DEV),
                  parity.dev_bf16(case["pre_w"], DEV), parity.dev_bf16(W, DEV), H,
                  torch.from_numpy(case["positions"]).to(DEV),
                  [None if s is None else torch.from_numpy(s).to(DEV) for s in case["slots"]],
                  parity.dev_bf16(case["cos_sin"], DEV), caches, case["eps"], ws, err=err,
                  kv_out=kv, w_layout=layout)
    torch.cuda.synchronize()
    return dict(kv=parity.host_bits(kv), caches=[parity.host_bits(c) for c in caches],
                err=int(err.item()))


def check_against_oracle(case, got, normed=None, sample=None):
    L = len(case["slots"])
    H = case["cache_shape"][1]
    T = case["x"].shape[0]
    ref_caches = parity.make_caches(case, L, parity.SENTINEL)
    ref_err = oracle.kv_store_from_projection(got["kv"], H, case["positions"], case["slots"],
                                              case["cos_sin"], ref_caches, case["eps"], T)
    for g, r in zip(got["caches"], ref_caches):
        assert np.array_equal(g, r)
    assert got["err"] == ref_err
    if normed is None:
        normed = oracle.context_norms(case["x"], case["hidden_w"], case["pre_w"], L, case["eps"])
    ref64, ab = oracle.kv_project(normed, case["W"], rows=sample)
    parity.assert_projection_close(got["kv"] if sample is None else got["kv"][:, sample], ref64, ab)


@pytest.mark.parametrize("T,L,H,rope,hw,pw", [
    (300, 2, 2, True, True, True),       # K and V heads in one tile
    (512, 3, 8, True, True, True),
    (200, 2, 16, False, True, True),
    (257, 9, 4, True, False, True),      # 9 layers, weightless hidden norm
    (400, 2, 8, True, True, False),      # weightless layer norms
    (64, 2, 8, True, True, True),        # T <= 128: norms in the workspace, single CTAs
    (100, 2, 1, True, True, True),       # N = 128
])
@pytest.mark.parametrize("layout", [rc.RC_W_KN, rc.RC_W_NK])
def test_whole_chain_equals_unfused_and_oracle(T, L, H, rope, hw, pw, layout):
    case = workloads.random_case(900 + T + L + H, T=T, L=L, H=H, rope=rope, max_position=512,
                                 num_blocks=(T + 15) // 16 + 3, block_size=16,
                                 hidden_weighted=hw, pre_weighted=pw)
    got = run_whole(case, layout=layout)
    ref = parity.run_gpu_chain(case, DEV, w_layout=layout)
    assert np.array_equal(got["kv"], ref["kv"]), "the fused operand differs from the norms kernel's"
    for a, b in zip(got["caches"], ref["caches"]):
        assert np.array_equal(a, b)
    assert got["err"] == ref["err"]
    check_against_oracle(case, got, normed=ref["normed"])


@pytest.mark.parametrize("T,H", [(512, 8), (300, 2)])
def test_whole_chain_without_split(T, H):
    # a workspace with room for z and r only: no split-K, the epilogue stores
    case = workloads.random_case(950 + T, T=T, L=3, H=H, max_position=512,
                                 num_blocks=(T + 15) // 16 + 3, block_size=16)
    got = run_whole(case, full_workspace=False)
    check_against_oracle(case, got)


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_whole_chain_workloads(index):
    w = workloads.WORKLOADS[index]
    case = workloads.make_inputs(w)
    got = run_whole(case)
    # the unfused chain under the whole chain's plan: split-K where the
    # tiles need fewer CTAs than there are SMs; otherwise persistent pairs
    # over every tile (no workspace, so no tail launch of the last rows)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    pair_ctas = 2 * w.L * ((w.T + 255) // 256) * (w.N // 256)
    persistent = w.T > 128 and w.N % 256 == 0 and pair_ctas >= sms
    ref = parity.run_gpu_chain(case, DEV, use_workspace=not persistent)
    assert np.array_equal(got["kv"], ref["kv"])
    for a, b in zip(got["caches"], ref["caches"]):
        assert np.array_equal(a, b)
    assert got["err"] == ref["err"]
    T = w.T
    sample = None if T <= 512 else np.unique(np.r_[0, T - 1, np.linspace(0, T - 1, 256).astype(int)])
    check_against_oracle(case, got, normed=ref["normed"], sample=sample)


@pytest.mark.parametrize("hw,pw", [(True, True), (False, True), (True, False)])
def test_two_phase_rows_then_projection(hw, pw):
    T, L, H = 384, 3, 8
    case = workloads.random_case(4242, T=T, L=L, H=H, max_position=512, num_blocks=(T + 15) // 16 + 3,
                                 block_size=16, hidden_weighted=hw, pre_weighted=pw)
    x = parity.dev_bf16(case["x"], DEV)
    z, r2 = rc.context_rows(x, parity.dev_bf16(case["hidden_w"], DEV), case["eps"])
    torch.cuda.synchronize()
    # (z, r2) reproduce the oracle's normed rows: bf16((z * r2) * gamma_l) in
    # binary32, one rounding per operation, as the layer step is defined
    zf = (parity.host_bits(z).astype(np.uint32) << 16).view(np.float32)
    r2h = r2.cpu().numpy().astype(np.float32)
    ref = oracle.context_norms(case["x"], case["hidden_w"], case["pre_w"], L, case["eps"])
    for l in range(L):
        y = zf * r2h[:, None]
        if pw:
            y = y * ((case["pre_w"][l].astype(np.uint32) << 16).view(np.float32))[None, :]
        assert np.array_equal(workloads.to_bf16_bits(y), ref[l])
    # rows + from_rows == the one-call chain
    whole = run_whole(case)
    caches = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
    kv = torch.empty((L, T, 128 * H), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = rc.new_workspace(L, T, 8192, 128 * H, DEV)
    rc.context_kv_from_rows(z, r2, parity.dev_bf16(case["pre_w"], DEV), parity.dev_bf16(case["W"], DEV),
                            H, torch.from_numpy(case["positions"]).to(DEV),
                            [torch.from_numpy(s).to(DEV) for s in case["slots"]],
                            parity.dev_bf16(case["cos_sin"], DEV), caches, case["eps"], err=err,
                            kv_out=kv, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(parity.host_bits(kv), whole["kv"])
    for a, b in zip(caches, whole["caches"]):
        assert np.array_equal(parity.host_bits(a), b)
    assert int(err.item()) == whole["err"]
