"""rc_kv_project_store (projection and store in one pass) against the
oracle: the caches bit-exact against the oracle's store fed the projection
the same call wrote to kv_out, kv_out within the projection rule, the skip
count equal; and the caches identical with and without kv_out and to the
unfused calls.  Covers the three ways the call runs: the CTA-pair epilogue
store (no split), the reduce-and-store pass (split-K), and projection to
kv_out then the store kernel (single CTAs, no split)."""
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


def _dev(case):
    H = case["cache_shape"][1]
    L = len(case["slots"])
    return dict(
        positions=torch.from_numpy(case["positions"]).to(DEV),
        slots=[None if s is None else torch.from_numpy(s).to(DEV) for s in case["slots"]],
        cs=parity.dev_bf16(case["cos_sin"], DEV),
        caches=[parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)],
        err=torch.zeros(1, dtype=torch.int32, device=DEV), H=H, L=L)


def run_fused(case, normed_d, W_d, *, workspace, kv_out, rows=None, layout=rc.RC_W_KN):
    d = _dev(case)
    T = normed_d.shape[1]
    kv = torch.empty((d["L"], T, 128 * d["H"]), dtype=torch.bfloat16, device=DEV) if kv_out else None
    ws = rc.new_workspace(d["L"], T, 8192 if normed_d.shape[2] == 8192 else normed_d.shape[2],
                          128 * d["H"], DEV) if workspace else None
    rc.kv_project_store(normed_d, W_d, d["H"], d["positions"], d["slots"], d["cs"], d["caches"],
                        case["eps"], rows=rows, err=d["err"], kv_out=kv, w_layout=layout,
                        workspace=ws)
    torch.cuda.synchronize()
    return ([parity.host_bits(c) for c in d["caches"]],
            None if kv is None else parity.host_bits(kv), int(d["err"].item()))


def check(case, normed, W, *, workspace, rows=None, layout=rc.RC_W_KN, slots=None):
    if slots is not None:
        case = dict(case, slots=slots)
    Wl = W if layout == rc.RC_W_KN else np.ascontiguousarray(W.transpose(0, 2, 1))
    nd, wd = parity.dev_bf16(normed, DEV), parity.dev_bf16(Wl, DEV)
    caches, kv, err = run_fused(case, nd, wd, workspace=workspace, kv_out=True, rows=rows,
                                layout=layout)
    T = normed.shape[1]
    rows_ = T if rows is None else rows
    ref_caches = parity.make_caches(case, len(case["slots"]), parity.SENTINEL)
    ref_err = oracle.kv_store_from_projection(kv, case["cache_shape"][1], case["positions"],
                                              case["slots"], case["cos_sin"], ref_caches,
                                              case["eps"], rows_)
    for g, r in zip(caches, ref_caches):
        assert np.array_equal(g, r)
    assert err == ref_err
    sample = None if T <= 512 else np.unique(np.r_[0, T - 1, np.linspace(0, T - 1, 200).astype(int)])
    ref64, ab = oracle.kv_project(normed, W, rows=sample)
    parity.assert_projection_close(kv if sample is None else kv[:, sample], ref64, ab)
    return caches, nd, wd


@pytest.mark.parametrize("T,L,H,workspace,rope", [
    (300, 2, 2, False, True),      # CTA pairs, epilogue store, K and V heads in one tile
    (512, 3, 8, False, True),      # CTA pairs, epilogue store
    (512, 3, 8, True, True),       # CTA pairs, split-K, reduce-and-store
    (256, 3, 8, True, True),       # CTA pairs, 6 splits
    (200, 1, 2, True, False),      # CTA pairs, 16 splits of 8 K blocks, ragged rows
    (200, 2, 16, False, False),    # CTA pairs, epilogue store, no RoPE
    (1000, 10, 4, False, True),    # persistent pairs: 80 tiles over at most 76 pairs (both accumulators)
    (1000, 10, 4, True, True),     # persistent pairs over 76 tiles, then the last layer's last two
                                   # row blocks (rows 512-999) split 16 ways and reduced and stored
    (129, 1, 32, True, True),      # H = 32, ragged rows
    (64, 2, 8, True, True),        # single CTAs, split-K, reduce-and-store
    (100, 2, 1, False, True),      # N = 128: single CTAs without split, kv_out then store
    (100, 3, 4, True, False),      # single CTAs (T <= 128), split, no RoPE
])
def test_fused_store_bit_exact(T, L, H, workspace, rope):
    case = workloads.random_case(500 + T + H, T=T, L=L, H=H, rope=rope, max_position=512,
                                 num_blocks=(T + 15) // 16 + 4, block_size=16)
    normed = oracle.context_norms(case["x"], case["hidden_w"], case["pre_w"], L, case["eps"])
    caches, nd, wd = check(case, normed, case["W"], workspace=workspace)
    # without kv_out (where the plan allows) the caches are the same bits
    if not (H == 1 and not workspace):
        c2, kv2, e2 = run_fused(case, nd, wd, workspace=workspace, kv_out=False)
        for a, b in zip(caches, c2):
            assert np.array_equal(a, b)


def test_fused_rows_prefix_null_layer_and_bad_rows():
    T, L, H = 300, 3, 8
    case = workloads.random_case(777, T=T, L=L, H=H, max_position=64, num_blocks=24, block_size=16)
    slots = [s.copy() for s in case["slots"]]
    slots[1] = None
    slots[0][5] = 24 * 16           # == capacity
    slots[2][7] = 1 << 40
    pos = case["positions"].copy()
    pos[9] = 64                     # == max_position
    case = dict(case, positions=pos)
    normed = oracle.context_norms(case["x"], case["hidden_w"], case["pre_w"], L, case["eps"])
    for ws in (False, True):
        check(case, normed, case["W"], workspace=ws, rows=250, slots=slots)


@pytest.mark.parametrize("layout", [rc.RC_W_KN, rc.RC_W_NK])
def test_fused_matches_unfused_chain(layout):
    # the caches of the fused call equal those of kv_project + kv_store
    w = workloads.WORKLOADS[2]
    case = workloads.make_inputs(w)
    got = parity.run_gpu_chain(case, DEV, w_layout=layout)
    normed = got["normed"]
    W = case["W"]
    Wl = W if layout == rc.RC_W_KN else np.ascontiguousarray(W.transpose(0, 2, 1))
    caches, kv, err = run_fused(case, parity.dev_bf16(normed, DEV), parity.dev_bf16(Wl, DEV),
                                workspace=True, kv_out=True, layout=layout)
    assert np.array_equal(kv, got["kv"])
    for a, b in zip(caches, got["caches"]):
        assert np.array_equal(a, b)
    assert err == got["err"]


@pytest.mark.parametrize("layout", [rc.RC_W_KN, rc.RC_W_NK])
def test_tail_split_projection(layout):
    # 80 tiles of 256 x 256 over 76 CTA pairs: the persistent kernel takes
    # 76, and the last layer's final row block (rows 2304-2499, ragged) runs
    # as a split-K launch of its own when a workspace is given
    T, L, H = 2500, 2, 8
    N = 128 * H
    case = workloads.random_case(4242, T=T, L=L, H=H, max_position=512,
                                 num_blocks=(T + 15) // 16 + 4, block_size=16)
    assert rc.workspace_size(L, T, 8192, N) > 0, "no tail split planned on this device"
    normed = oracle.context_norms(case["x"], case["hidden_w"], case["pre_w"], L, case["eps"])
    Wl = case["W"] if layout == rc.RC_W_KN else np.ascontiguousarray(case["W"].transpose(0, 2, 1))
    nd, wd = parity.dev_bf16(normed, DEV), parity.dev_bf16(Wl, DEV)
    ws = rc.new_workspace(L, T, 8192, N, DEV)
    tailed = parity.host_bits(rc.kv_project(nd, wd, w_layout=layout, workspace=ws))
    plain = parity.host_bits(rc.kv_project(nd, wd, w_layout=layout))
    sample = np.unique(np.r_[0, 2303, 2304, 2305, T - 1, np.linspace(0, T - 1, 120).astype(int),
                             np.arange(2304, T, 9)])
    ref64, ab = oracle.kv_project(normed, case["W"], rows=sample)
    parity.assert_projection_close(tailed[:, sample], ref64, ab, "projection with the tail split")
    parity.assert_projection_close(plain[:, sample], ref64, ab, "projection without it")
    # rows outside the tail come from the same persistent kernel either way
    assert np.array_equal(tailed[0], plain[0]) and np.array_equal(tailed[1, :2304], plain[1, :2304])
    caches, kv, err = run_fused(case, nd, wd, workspace=True, kv_out=True, layout=layout)
    assert np.array_equal(kv, tailed), "the fused call's projection differs from rc_kv_project's"
    ref_caches = parity.make_caches(case, L, parity.SENTINEL)
    ref_err = oracle.kv_store_from_projection(kv, H, case["positions"], case["slots"],
                                              case["cos_sin"], ref_caches, case["eps"], T)
    for g, r in zip(caches, ref_caches):
        assert np.array_equal(g, r)
    assert err == ref_err


@pytest.mark.parametrize("last_rows", [2000, 2304, 2400])
def test_tail_split_with_layer_row_counts(last_rows):
    # the last layer stores its first last_rows rows: none of the tail's rows
    # (2304-2499) when last_rows <= 2304, some of them otherwise
    T, L, H = 2500, 2, 8
    case = workloads.random_case(4343, T=T, L=L, H=H, max_position=512,
                                 num_blocks=(T + 15) // 16 + 4, block_size=16)
    case = dict(case, slots=[case["slots"][0], np.ascontiguousarray(case["slots"][1][:last_rows])])
    normed = oracle.context_norms(case["x"], case["hidden_w"], case["pre_w"], L, case["eps"])
    nd, wd = parity.dev_bf16(normed, DEV), parity.dev_bf16(case["W"], DEV)
    caches, kv, err = run_fused(case, nd, wd, workspace=True, kv_out=True)
    ref_caches = parity.make_caches(case, L, parity.SENTINEL)
    ref_err = oracle.kv_store_from_projection(kv, H, case["positions"], case["slots"],
                                              case["cos_sin"], ref_caches, case["eps"],
                                              np.array([T, last_rows]))
    for g, r in zip(caches, ref_caches):
        assert np.array_equal(g, r)
    assert err == ref_err
    sample = np.array([0, 2303, 2304, 2400, T - 1])
    ref64, ab = oracle.kv_project(normed, case["W"], rows=sample)
    parity.assert_projection_close(kv[:, sample], ref64, ab)


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_fused_workloads(index):
    w = workloads.WORKLOADS[index]
    case = workloads.make_inputs(w)
    normed = oracle.context_norms(case["x"], case["hidden_w"], case["pre_w"], w.L, w.eps)
    check(case, normed, case["W"], workspace=True)



@pytest.mark.parametrize("L,T,D,H,layout,tail", [(4, 8192, 1024, 16, rc.RC_W_KN, False),
                                                 (4, 8192, 1024, 16, rc.RC_W_NK, False),
                                                 (8, 8192, 4096, 8, rc.RC_W_KN, True)])
def test_dynamic_tile_order_repeats_and_graph_replays(L, T, D, H, layout, tail):
    # persistent pairs over eight rounds of tiles or more (1024 tiles of 256 x
    # 256): given a workspace the pairs take tiles from a counter in it (the
    # last shape also splits its final row blocks into a tail launch).  Each
    # tile's arithmetic is the fixed-order kernel's, so every call (back to
    # back on one workspace, with other inputs in between, and as CUDA-graph
    # replays) must match the fixed order outside the tail bit for bit.
    N = 128 * H
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    nbytes = rc.workspace_size(L, T, D, N)
    plan = rc.project_plan(L, T, D, N, sms, nbytes)
    assert plan["kernel"] == "persistent CTA pairs" and plan["dynamic_tiles"], plan
    assert (plan["tail_splits"] > 0) == tail, plan
    assert not rc.project_plan(L, T, D, N, sms, 0)["dynamic_tiles"]
    rng = np.random.default_rng(4242 + D)
    ins, raw = [], []
    for _ in range(2):
        a = workloads.normal_bf16(rng, (L, T, D), 0.0, 1.0)
        W = workloads.normal_bf16(rng, (L, D, N), 0.0, 0.02)
        Wl = W if layout == rc.RC_W_KN else np.ascontiguousarray(W.transpose(0, 2, 1))
        ins.append((parity.dev_bf16(a, DEV), parity.dev_bf16(Wl, DEV)))
        raw.append((a, W))
    fixed = [parity.host_bits(rc.kv_project(a_d, w_d, w_layout=layout)) for a_d, w_d in ins]
    # the tail's rows (the last layer's final row blocks) use another split
    # and so another summation order: those are checked against float64
    rows_fixed = plan["tail_row0"]
    tail_rows = np.arange(rows_fixed, T)

    def check(got, i, what):
        if not tail:
            assert np.array_equal(got, fixed[i]), what
            return
        assert np.array_equal(got[:L - 1], fixed[i][:L - 1]), what
        assert np.array_equal(got[L - 1, :rows_fixed], fixed[i][L - 1, :rows_fixed]), what
        sample = tail_rows[:: max(1, len(tail_rows) // 16)]
        ref64, ab = oracle.kv_project(raw[i][0][L - 1:], raw[i][1][L - 1:], rows=sample)
        parity.assert_projection_close(got[L - 1:, sample], ref64, ab, what + " (tail rows)")

    ws = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device=DEV)    # any initial contents
    for i in (0, 1, 0, 0, 1):
        check(parity.host_bits(rc.kv_project(ins[i][0], ins[i][1], w_layout=layout, workspace=ws)),
              i, f"call on input {i}")
    # as CUDA-graph replays
    outs = [torch.empty((L, T, N), dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    s = torch.cuda.Stream(DEV)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(2):
            rc.kv_project(ins[i][0], ins[i][1], out=outs[i], w_layout=layout, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(2):
            rc.kv_project(ins[i][0], ins[i][1], out=outs[i], w_layout=layout, workspace=ws)
    for _ in range(3):
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for i in range(2):
            check(parity.host_bits(outs[i]), i, f"graph replay, input {i}")
    assert rc.read_device_faults(clear=True) == 0
