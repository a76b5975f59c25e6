"""rc_context_kv_chunked (norms, projection and store by row chunks, each
chunk's norms running beside the previous chunk's projection) against the
unfused three-call chain.

A chunk's rows are normed by the same kernel arithmetic and projected by
the same persistent CTA-pair kernel with the same K order as the unchunked
call without a workspace (chunks start on 256-row tile boundaries), so every
cache must be bit-identical to the unfused chain's, whose caches the oracle
tests pin; the error count must match too.  Cases: ragged last chunks, rows
below T, layers without a slot map, no RoPE, weightless norms, both weight
layouts, a repeated call and a graph replay (each chunk's tile counter is
zeroed per call), and workload 5 at full size.
"""
import ctypes

import numpy as np
import pytest
import torch

import rope_chain_gb300 as rc
import workloads
from tests import parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    from rope_chain_gb300 import _build
    _build.build()
    rc.read_device_faults(clear=True)
    yield
    assert rc.read_device_faults(clear=True) == 0


def _operands(case, layout):
    W = case["W"] if layout == rc.RC_W_KN else np.ascontiguousarray(case["W"].transpose(0, 2, 1))
    return dict(x=parity.dev_bf16(case["x"], DEV), hw=parity.dev_bf16(case["hidden_w"], DEV),
                pw=parity.dev_bf16(case["pre_w"], DEV), W=parity.dev_bf16(W, DEV),
                positions=torch.from_numpy(case["positions"]).to(DEV),
                slots=[None if s is None else torch.from_numpy(s).to(DEV) for s in case["slots"]],
                cs=parity.dev_bf16(case["cos_sin"], DEV))


def run_chunked(case, chunks, *, layout=rc.RC_W_KN, rows=None, ops=None, calls=1):
    L = len(case["slots"])
    H = case["cache_shape"][1]
    T = case["x"].shape[0]
    ops = ops or _operands(case, layout)
    ws = rc.context_kv_chunked_workspace(L, T, H, DEV, chunks=chunks)
    out = []
    for _ in range(calls):                       # each call into fresh sentinel caches
        caches = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        rc.context_kv_chunked(ops["x"], ops["hw"], ops["pw"], ops["W"], H, ops["positions"],
                              ops["slots"], ops["cs"], caches, case["eps"], ws, rows=rows, err=err,
                              chunks=chunks, w_layout=layout)
        torch.cuda.synchronize()
        out.append(dict(caches=[parity.host_bits(c) for c in caches], err=int(err.item())))
    return out if calls > 1 else out[0]


def run_reference(case, *, layout=rc.RC_W_KN, rows=None, use_workspace=False, kv_out=False):
    """rc_context_norms + rc_kv_project_store, the default step's two calls."""
    L = len(case["slots"])
    H = case["cache_shape"][1]
    T = case["x"].shape[0]
    ops = _operands(case, layout)
    caches = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    normed = rc.context_norms(ops["x"], ops["hw"], ops["pw"], L, case["eps"])
    ws = rc.new_workspace(L, T, 8192, 128 * H, DEV) if use_workspace else None
    kv = torch.empty((L, T, 128 * H), dtype=torch.bfloat16, device=DEV) if kv_out else None
    rc.kv_project_store(normed, ops["W"], H, ops["positions"], ops["slots"], ops["cs"], caches,
                        case["eps"], rows=rows, err=err, workspace=ws, w_layout=layout, kv_out=kv)
    torch.cuda.synchronize()
    return dict(caches=[parity.host_bits(c) for c in caches], err=int(err.item()))


def assert_same(got, ref):
    for l, (a, b) in enumerate(zip(got["caches"], ref["caches"])):
        diff = np.argwhere(a != b)
        assert diff.size == 0, f"layer {l}: {len(diff)} cache elements differ, first {tuple(diff[0])}"
    assert got["err"] == ref["err"]


SMS = None


def sms():
    global SMS
    if SMS is None:
        SMS = torch.cuda.get_device_properties(DEV).multi_processor_count
    return SMS


@pytest.mark.parametrize("T,L,H,chunks,rope,hw,pw", [
    (1024, 3, 8, 2, True, True, True),       # chunks of 256 and 768 rows
    (1300, 2, 4, 3, True, True, True),       # 256, 768 and a ragged 276
    (2304, 4, 8, 4, True, True, True),       # 256, 768, 768, 512
    (800, 2, 16, 3, False, True, True),      # no RoPE, 16 heads (256 and 544)
    (1536, 3, 2, 2, True, False, True),      # weightless hidden norm, K and V heads in one tile
    (1000, 2, 8, 2, True, True, False),      # weightless layer norms (256 and 744)
    (1024, 9, 2, 2, True, True, True),       # 9 layers: past 8 layers per store launch
])
@pytest.mark.parametrize("layout", [rc.RC_W_KN, rc.RC_W_NK])
def test_chunked_equals_unfused(T, L, H, chunks, rope, hw, pw, layout):
    assert rc.context_kv_chunks(L, T, H, sms(), chunks) >= 2
    case = workloads.random_case(1700 + T + L + H, T=T, L=L, H=H, rope=rope, max_position=512,
                                 num_blocks=(T + 15) // 16 + 3, block_size=16,
                                 hidden_weighted=hw, pre_weighted=pw)
    got = run_chunked(case, chunks, layout=layout)
    ref = run_reference(case, layout=layout)
    assert_same(got, ref)


def test_chunked_rows_null_layer_and_out_of_range():
    T, L, H = 1536, 3, 8
    case = workloads.random_case(1777, T=T, L=L, H=H, max_position=512,
                                 num_blocks=(T + 15) // 16 + 3, block_size=16)
    case["slots"][1] = None                      # a layer without a slot map stores nothing
    case["slots"][2] = case["slots"][2].copy()
    case["slots"][2][::97] = (T + 15) // 16 * 16 + 3 * 16 + 5     # past the cache: counted
    case["positions"] = case["positions"].copy()
    case["positions"][5::211] = 9999             # past the table: counted
    assert rc.context_kv_chunk_rows(L, T, H, sms(), 3) == [0, 256, 1024, 1536]
    for rows in (T, 1000, 200, 0):               # rows ending in the 3rd, 2nd, 1st chunk, none
        got = run_chunked(case, 3, rows=rows)
        ref = run_reference(case, rows=rows)
        assert_same(got, ref)
        if rows == T:
            assert got["err"] > 0


def test_chunked_repeated_calls_and_graph_replay():
    T, L, H = 2048, 3, 8
    case = workloads.random_case(1788, T=T, L=L, H=H, max_position=512,
                                 num_blocks=(T + 15) // 16 + 3, block_size=16)
    ref = run_reference(case)
    first, second = run_chunked(case, 4, calls=2)
    assert_same(first, ref)
    assert_same(second, ref)
    # the same call captured once and replayed into fresh sentinel caches
    ops = _operands(case, rc.RC_W_KN)
    ws = rc.context_kv_chunked_workspace(L, T, H, DEV, chunks=4)
    caches = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    fresh = [c.clone() for c in caches]
    s = torch.cuda.Stream(device=DEV)
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            rc.context_kv_chunked(ops["x"], ops["hw"], ops["pw"], ops["W"], H, ops["positions"],
                                  ops["slots"], ops["cs"], caches, case["eps"], ws, err=err,
                                  chunks=4)
    torch.cuda.synchronize()
    for _ in range(2):
        for c, f in zip(caches, fresh):
            c.copy_(f)
        err.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_same(dict(caches=[parity.host_bits(c) for c in caches], err=int(err.item())), ref)


@pytest.mark.parametrize("chunks", [0, 3])
def test_chunked_x_in_host_memory(chunks):
    # x in page-locked host memory: each chunk's norms read their rows over
    # the host link, and the chunk plan is the host one; the bits do not
    # depend on the chunks
    T, L, H = 2048, 3, 8
    case = workloads.random_case(1822, T=T, L=L, H=H, max_position=512,
                                 num_blocks=(T + 15) // 16 + 3, block_size=16)
    ops = _operands(case, rc.RC_W_KN)
    ops["x"] = ops["x"].cpu().pin_memory()
    want = rc.context_kv_chunks(L, T, H, sms(), chunks, x_on_host=True)
    assert want == (2 if chunks == 0 else 3)
    got = run_chunked(case, chunks, ops=ops)
    ref = run_reference(case) if want > 1 else run_reference(case, use_workspace=True)
    assert_same(got, ref)


@pytest.mark.parametrize("T,L,H", [(2560, 8, 1), (100, 5, 32)])
def test_chunked_single_ctas_without_split(T, L, H):
    # N = 128 at 2560 rows, or 100 rows of 32 heads: single CTAs and enough
    # tiles for no K split, so the store reads a bf16 copy of the
    # projection, which the chunked call keeps in its workspace
    assert rc.context_kv_chunks(L, T, H, sms(), 0) == 1
    p = rc.project_plan(L, T, 8192, 128 * H, sms(), rc.workspace_size_for(L, T, 8192, 128 * H, sms()))
    assert p["kernel"] == "single CTAs" and p["splits"] == 1
    case = workloads.random_case(1833 + T, T=T, L=L, H=H, max_position=512,
                                 num_blocks=(T + 15) // 16 + 3, block_size=16)
    got = run_chunked(case, 0)
    ref = run_reference(case, use_workspace=True, kv_out=True)
    assert_same(got, ref)


def test_chunked_one_chunk_uses_the_full_plan():
    # too few tiles per chunk for the automatic choice: one chunk, the
    # projection's full-workspace plan (split-K here), as the default step
    T, L, H = 512, 3, 8
    assert rc.context_kv_chunks(L, T, H, sms(), 0) == 1
    case = workloads.random_case(1799, T=T, L=L, H=H, max_position=512,
                                 num_blocks=(T + 15) // 16 + 3, block_size=16)
    got = run_chunked(case, 0)
    ref = run_reference(case, use_workspace=True)
    assert_same(got, ref)


def test_chunked_refusals():
    T, L, H = 1024, 2, 8
    case = workloads.random_case(1811, T=T, L=L, H=H, max_position=512,
                                 num_blocks=(T + 15) // 16 + 3, block_size=16)
    ops = _operands(case, rc.RC_W_KN)
    caches = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
    before = [parity.host_bits(c) for c in caches]
    ws = rc.context_kv_chunked_workspace(L, T, H, DEV, chunks=2)
    call = lambda w, **kw: rc.context_kv_chunked(ops["x"], ops["hw"], ops["pw"], ops["W"], H,
                                                 ops["positions"], ops["slots"], ops["cs"], caches,
                                                 case["eps"], w, chunks=2, **kw)
    need = (L * T * 8192 * 2 + 255) // 256 * 256 + 2 * 256     # normed rows + 2 counters
    assert ws.numel() >= need
    with pytest.raises(rc.RopeChainError, match="workspace needs"):
        call(ws[:need - 256])                    # no room for the second chunk's counter
    # a workspace holding x
    buf = torch.empty(ws.numel() + T * 8192 * 2, dtype=torch.uint8, device=DEV)
    xv = buf[:T * 8192 * 2].view(torch.bfloat16).view(T, 8192)
    xv.copy_(ops["x"])
    with pytest.raises(rc.RopeChainError, match="overlaps"):
        rc.context_kv_chunked(xv, ops["hw"], ops["pw"], ops["W"], H, ops["positions"], ops["slots"],
                              ops["cs"], caches, case["eps"], buf, chunks=2)
    torch.cuda.synchronize()
    for a, b in zip(caches, before):
        assert np.array_equal(parity.host_bits(a), b)


@pytest.mark.parametrize("index", [4, 5])
@pytest.mark.parametrize("host", [False, True])
def test_chunked_workload_full_size(index, host):
    # the default step (x in device memory: 2 chunks at workload 4, 4 at
    # workload 5) and the end-to-end step (x in pinned host memory: the host
    # plan's 6 and 7 chunks) at full size
    w = workloads.WORKLOADS[index]
    case = workloads.make_inputs(w)
    chunks = rc.context_kv_chunks(w.L, w.T, w.H, sms(), 0, x_on_host=host)
    assert chunks >= 2
    ops = _operands(case, rc.RC_W_KN)
    if host:
        ops["x"] = ops["x"].cpu().pin_memory()
    got = run_chunked(case, 0, ops=ops)
    ref = run_reference(case)
    assert_same(got, ref)


def _options(case, L, kind):
    """Norm options of the _ex call: FP32 gains with the hidden weight on the
    input and a layer gain centre of 1; bf16 gains with centres; none."""
    f32 = lambda a: None if a is None else torch.from_numpy(
        (a.astype(np.uint32) << 16).view(np.float32)).to(DEV)
    eps = case["eps"]
    if kind == "fp32":
        return dict(hidden_w=f32(case["hidden_w"]), pre_w=f32(case["pre_w"]), hidden_eps=eps,
                    pre_eps=10 * eps, hidden_input_scale=True, pre_center=1.0)
    if kind == "centred":
        return dict(hidden_w=parity.dev_bf16(case["hidden_w"], DEV),
                    pre_w=parity.dev_bf16(case["pre_w"], DEV), hidden_eps=2 * eps, pre_eps=eps,
                    hidden_center=-0.5, pre_center=0.25)
    return dict(hidden_w=None, pre_w=None, hidden_eps=eps, pre_eps=eps)


@pytest.mark.parametrize("T,L,H,chunks,kind,layout,per_layer,host", [
    (1536, 3, 8, 3, "fp32", rc.RC_W_KN, True, False),
    (1536, 3, 8, 2, "centred", rc.RC_W_NK, False, False),
    (2048, 2, 4, 2, "none", rc.RC_W_KN, True, True),
    (512, 3, 8, 0, "fp32", rc.RC_W_KN, True, False),     # one chunk: the full plan
])
def test_chunked_ex_equals_norms_ex_and_rows_store(T, L, H, chunks, kind, layout, per_layer, host):
    case = workloads.random_case(1900 + T + L, T=T, L=L, H=H, max_position=512,
                                 num_blocks=(T + 15) // 16 + 3, block_size=16)
    ops = _operands(case, layout)
    opts = _options(case, L, kind)
    rows = [T - l * (T // (2 * L)) for l in range(L)] if per_layer else T
    n = rc.context_kv_chunks(L, T, H, sms(), chunks, x_on_host=host)
    assert (n >= 2) == (chunks != 0)
    # the reference: the option norms, then the projection + store with a
    # row count per layer (no workspace where chunks run, as they do)
    caches_r = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
    err_r = torch.zeros(1, dtype=torch.int32, device=DEV)
    normed = rc.context_norms_ex(ops["x"], L, **opts)
    ws_r = None if n >= 2 else rc.new_workspace(L, T, 8192, 128 * H, DEV)
    rc.kv_project_store(normed, ops["W"], H, ops["positions"], ops["slots"], ops["cs"], caches_r,
                        case["eps"], rows=rows, err=err_r, workspace=ws_r, w_layout=layout)
    # the chunked call
    caches = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    x = ops["x"].cpu().pin_memory() if host else ops["x"]
    ws = rc.context_kv_chunked_workspace(L, T, H, DEV, chunks=chunks)
    rc.context_kv_chunked_ex(x, ops["W"], H, ops["positions"], ops["slots"], ops["cs"], caches,
                             case["eps"], ws, rows=rows, err=err, chunks=chunks, w_layout=layout,
                             **opts)
    torch.cuda.synchronize()
    assert_same(dict(caches=[parity.host_bits(c) for c in caches], err=int(err.item())),
                dict(caches=[parity.host_bits(c) for c in caches_r], err=int(err_r.item())))


@pytest.mark.parametrize("host", [False, True])
def test_chunked_ex_automatic_count_with_options(host):
    # at a size the plain call splits (2 chunks), FP32 gains keep one chunk
    # with x in device memory (the option kernel beside the projection costs
    # more than the overlap) and take the host plan with x in host memory;
    # the bits are the same either way
    T, L, H = 16384, 8, 8
    assert rc.context_kv_chunks(L, T, H, sms(), 0) >= 2
    assert rc.context_kv_chunks(L, T, H, sms(), 0, x_on_host=True) >= 2
    case = workloads.random_case(1950, T=T, L=L, H=H, max_position=512,
                                 num_blocks=(T + 15) // 16 + 3, block_size=16)
    ops = _operands(case, rc.RC_W_KN)
    opts = _options(case, L, "fp32")
    caches_r = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
    err_r = torch.zeros(1, dtype=torch.int32, device=DEV)
    normed = rc.context_norms_ex(ops["x"], L, **opts)
    rc.kv_project_store(normed, ops["W"], H, ops["positions"], ops["slots"], ops["cs"], caches_r,
                        case["eps"], err=err_r, workspace=rc.new_workspace(L, T, 8192, 128 * H, DEV))
    del normed
    caches = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    x = ops["x"].cpu().pin_memory() if host else ops["x"]
    rc.context_kv_chunked_ex(x, ops["W"], H, ops["positions"], ops["slots"], ops["cs"], caches,
                             case["eps"], rc.context_kv_chunked_workspace(L, T, H, DEV), err=err,
                             **opts)
    torch.cuda.synchronize()
    assert_same(dict(caches=[parity.host_bits(c) for c in caches], err=int(err.item())),
                dict(caches=[parity.host_bits(c) for c in caches_r], err=int(err_r.item())))


def test_chunked_ex_refusals():
    T, L, H = 1024, 2, 8
    case = workloads.random_case(1961, T=T, L=L, H=H, max_position=512,
                                 num_blocks=(T + 15) // 16 + 3, block_size=16)
    ops = _operands(case, rc.RC_W_KN)
    caches = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
    before = [parity.host_bits(c) for c in caches]
    ws = rc.context_kv_chunked_workspace(L, T, H, DEV)
    slot_arr, cache_arr, nb, bs, _ = rc._store_operands(H, ops["slots"], caches, ops["positions"],
                                                        ops["cs"], T)
    ok = rc.NormParams(None, rc.RC_NORM_NONE, 0, 0.0, case["eps"])
    bad_dtype = rc.NormParams(None, 7, 0, 0.0, case["eps"])
    stray = rc.NormParams(ops["pw"].data_ptr(), rc.RC_NORM_NONE, 0, 0.0, case["eps"])
    rows = (ctypes.c_int64 * L)(*([T] * L))

    def call(h, p):
        return rc.lib().rc_context_kv_chunked_ex(
            ops["x"].data_ptr(), T, 8192, h, p, L, ops["W"].data_ptr(), rc.RC_W_KN, H,
            ops["positions"].data_ptr(), slot_arr, ops["cs"].data_ptr(), ops["cs"].shape[0],
            cache_arr, nb, bs, case["eps"], rows, None, 0, ws.data_ptr(), ws.numel(),
            torch.cuda.current_stream().cuda_stream)

    assert call(None, ctypes.byref(ok)) == rc.RC_ERR_INVALID_ARG
    assert call(ctypes.byref(bad_dtype), ctypes.byref(ok)) == rc.RC_ERR_INVALID_ARG
    assert "weight_dtype" in rc.lib().rc_last_error().decode()
    assert call(ctypes.byref(ok), ctypes.byref(stray)) == rc.RC_ERR_INVALID_ARG
    assert "NULL exactly" in rc.lib().rc_last_error().decode()
    torch.cuda.synchronize()
    for a, b in zip(caches, before):
        assert np.array_equal(parity.host_bits(a), b)


def test_chunked_ex_workload5_variants_host_x():
    # the variants' end-to-end step at full size: FP32 gains with the hidden
    # gain on the input, a layer gain centre of 1, separate eps and layer l
    # storing T - l * T / (2 L) rows, x in pinned host memory (the host
    # plan's chunks); against the option norms + the per-layer store
    w = workloads.WORKLOADS[5]
    case = workloads.make_inputs(w)
    L, T, H = w.L, w.T, w.H
    assert rc.context_kv_chunks(L, T, H, sms(), 0, x_on_host=True) >= 2
    ops = _operands(case, rc.RC_W_KN)
    opts = _options(case, L, "fp32")
    rows = [T - l * (T // (2 * L)) for l in range(L)]
    caches_r = [torch.zeros(case["cache_shape"], dtype=torch.bfloat16, device=DEV) for _ in range(L)]
    err_r = torch.zeros(1, dtype=torch.int32, device=DEV)
    normed = rc.context_norms_ex(ops["x"], L, **opts)
    rc.kv_project_store(normed, ops["W"], H, ops["positions"], ops["slots"], ops["cs"], caches_r,
                        case["eps"], rows=rows, err=err_r,
                        workspace=rc.new_workspace(L, T, 8192, 128 * H, DEV))
    del normed
    caches = [torch.zeros(case["cache_shape"], dtype=torch.bfloat16, device=DEV) for _ in range(L)]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    rc.context_kv_chunked_ex(ops["x"].cpu().pin_memory(), ops["W"], H, ops["positions"],
                             ops["slots"], ops["cs"], caches, case["eps"],
                             rc.context_kv_chunked_workspace(L, T, H, DEV), rows=rows, err=err,
                             **opts)
    torch.cuda.synchronize()
    assert_same(dict(caches=[parity.host_bits(c) for c in caches], err=int(err.item())),
                dict(caches=[parity.host_bits(c) for c in caches_r], err=int(err_r.item())))
