"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, and rejects malformed calls on the host before any CUDA
call (so these run on a machine with no GPU at all)."""
import ctypes
import os
import re

import pytest

import rope_chain_gb300 as rc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rope_chain.h")


@pytest.fixture(scope="module")
def lib():
    from rope_chain_gb300 import _build
    _build.build()
    return rc.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rc_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_are_exported(lib):
    names = declared_functions()
    assert {"rc_context_norms", "rc_kv_project", "rc_kv_store", "rc_last_error"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(rc.SIGNATURES)


def test_version(lib):
    assert lib.rc_version() == 100


def A(v):
    """A fake, suitably aligned device address: never dereferenced, because
    every call below is rejected (or is empty) before anything is launched."""
    return ctypes.c_void_p(v)


def last(lib):
    return lib.rc_last_error().decode()


def test_norms_rejections(lib):
    x, o = 0x10000, 0x200000
    assert lib.rc_context_norms(A(x), 4, 4096, None, None, 1, 1e-6, A(o), None) == rc.RC_ERR_UNSUPPORTED
    assert "8192" in last(lib)
    assert lib.rc_context_norms(None, 4, 8192, None, None, 1, 1e-6, A(o), None) == rc.RC_ERR_INVALID_ARG
    assert lib.rc_context_norms(A(x + 2), 4, 8192, None, None, 1, 1e-6, A(o), None) == rc.RC_ERR_INVALID_ARG
    assert "aligned" in last(lib)
    assert lib.rc_context_norms(A(x), 4, 8192, A(0x8), None, 1, 1e-6, A(o), None) == rc.RC_ERR_INVALID_ARG
    assert lib.rc_context_norms(A(x), 4, 8192, None, None, 0, 1e-6, A(o), None) == rc.RC_ERR_INVALID_ARG
    assert lib.rc_context_norms(A(x), -1, 8192, None, None, 1, 1e-6, A(o), None) == rc.RC_ERR_INVALID_ARG
    # out overlapping x
    assert lib.rc_context_norms(A(x), 4, 8192, None, None, 1, 1e-6, A(x + 16), None) == rc.RC_ERR_INVALID_ARG
    assert "overlaps" in last(lib)
    # T == 0 launches nothing and succeeds
    assert lib.rc_context_norms(A(x), 0, 8192, None, None, 2, 1e-6, A(o), None) == rc.RC_OK
    assert last(lib) == ""


def test_project_rejections(lib):
    a, w, o = 0x100000, 0x4000000, 0x8000000
    call = lambda *kw: lib.rc_kv_project(*kw)
    assert call(A(a), A(w), 0, A(o), 1, 8, 8192, 100, None, 0, None) == rc.RC_ERR_UNSUPPORTED
    assert call(A(a), A(w), 0, A(o), 1, 8, 8100, 1024, None, 0, None) == rc.RC_ERR_UNSUPPORTED
    assert call(A(a), A(w), 2, A(o), 1, 8, 8192, 1024, None, 0, None) == rc.RC_ERR_INVALID_ARG
    assert call(A(a), A(w), 0, A(o), 0, 8, 8192, 1024, None, 0, None) == rc.RC_ERR_INVALID_ARG
    assert call(A(a), A(w), 0, A(o), 1, 65535 * 128 + 1, 8192, 1024, None, 0, None) == rc.RC_ERR_INVALID_ARG
    assert call(A(a + 8), A(w), 0, A(o), 1, 8, 8192, 1024, None, 0, None) == rc.RC_ERR_INVALID_ARG
    assert call(None, A(w), 0, A(o), 1, 8, 8192, 1024, None, 0, None) == rc.RC_ERR_INVALID_ARG
    assert call(A(a), A(w), 0, A(o), 1, 0, 8192, 1024, None, 0, None) == rc.RC_OK
    assert lib.rc_kv_project_workspace_size(1, 8, 8192, 100) == 0


def _store(lib, **over):
    arg = dict(k=A(0x1000), v=A(0x1080), kls=1024, krs=128, vls=1024, vrs=128, positions=A(0x4000),
               slots=[A(0x8000)], cos=None, maxpos=0, caches=[A(0x100000)], nb=4, bs=16, H=8,
               L=1, eps=1e-6, rows=4, err=None)
    arg.update(over)
    L = arg["L"]
    slots = (ctypes.c_void_p * max(L, 1))(*arg["slots"][:L])
    caches = (ctypes.c_void_p * max(L, 1))(*arg["caches"][:L])
    return lib.rc_kv_store(arg["k"], arg["v"], arg["kls"], arg["krs"], arg["vls"], arg["vrs"],
                           arg["positions"], slots, arg["cos"], arg["maxpos"], caches, arg["nb"],
                           arg["bs"], arg["H"], L, arg["eps"], arg["rows"], arg["err"], None)


def test_store_rejections(lib):
    assert _store(lib, H=3) == rc.RC_ERR_UNSUPPORTED
    assert _store(lib, H=64) == rc.RC_ERR_UNSUPPORTED
    assert _store(lib, k=A(0x1002)) == rc.RC_ERR_INVALID_ARG
    assert _store(lib, krs=127) == rc.RC_ERR_INVALID_ARG
    assert _store(lib, vls=-2) == rc.RC_ERR_INVALID_ARG
    assert _store(lib, nb=1 << 20, bs=1 << 11) == rc.RC_ERR_INVALID_ARG   # 2^31 slots
    assert _store(lib, nb=0) == rc.RC_ERR_INVALID_ARG
    assert _store(lib, rows=-1) == rc.RC_ERR_INVALID_ARG
    assert _store(lib, cos=A(0x9000), maxpos=0) == rc.RC_ERR_INVALID_ARG
    assert _store(lib, cos=A(0x9000), maxpos=16, positions=None) == rc.RC_ERR_INVALID_ARG
    assert _store(lib, slots=[A(0x8004)]) == rc.RC_ERR_INVALID_ARG
    assert _store(lib, caches=[None]) == rc.RC_ERR_INVALID_ARG
    assert "caches[0]" in last(lib)
    # a layer without slots needs no cache; rows == 0 launches nothing
    assert _store(lib, slots=[None], caches=[None], rows=0) == rc.RC_OK
    assert _store(lib, rows=0) == rc.RC_OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(rc, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(rc, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        rc.lib()


def _norm(weight=None, dtype=0, input_scale=0, center=0.0, eps=1e-6):
    return rc.NormParams(weight, dtype, input_scale, center, eps)


def test_norms_ex_rejections(lib):
    x, o = 0x10000, 0x200000
    call = lambda h, p, D=8192, T=4, L=1: lib.rc_context_norms_ex(
        A(x), T, D, None if h is None else ctypes.byref(h), None if p is None else ctypes.byref(p),
        L, A(o), None)
    none = _norm()
    assert call(none, none, D=4096) == rc.RC_ERR_UNSUPPORTED
    assert call(None, none) == rc.RC_ERR_INVALID_ARG
    assert call(_norm(dtype=5), none) == rc.RC_ERR_INVALID_ARG
    assert "weight_dtype" in last(lib)
    assert call(_norm(dtype=rc.RC_NORM_BF16), none) == rc.RC_ERR_INVALID_ARG     # dtype, no weight
    assert call(none, _norm(weight=0x4000)) == rc.RC_ERR_INVALID_ARG             # weight, no dtype
    assert call(none, _norm(weight=0x4008, dtype=rc.RC_NORM_F32)) == rc.RC_ERR_INVALID_ARG
    assert "aligned" in last(lib)
    assert call(none, none, L=0) == rc.RC_ERR_INVALID_ARG
    # input_scale and a center on a weightless norm are ignored; T == 0 is empty
    assert call(_norm(input_scale=1, center=1.0), _norm(weight=0x4000, dtype=rc.RC_NORM_F32),
                T=0) == rc.RC_OK


def _store_rows(lib, layer_rows, **over):
    arg = dict(k=A(0x1000), v=A(0x1080), kls=1024, krs=128, vls=1024, vrs=128, positions=A(0x4000),
               slots=[A(0x8000), A(0x9000)], cos=None, maxpos=0,
               caches=[A(0x100000), A(0x200000)], nb=4, bs=16, H=8, L=2, eps=1e-6, err=None)
    arg.update(over)
    L = arg["L"]
    slots = (ctypes.c_void_p * L)(*arg["slots"][:L])
    caches = (ctypes.c_void_p * L)(*arg["caches"][:L])
    rows = None if layer_rows is None else (ctypes.c_int64 * L)(*layer_rows)
    return lib.rc_kv_store_rows(arg["k"], arg["v"], arg["kls"], arg["krs"], arg["vls"],
                                arg["vrs"], arg["positions"], slots, arg["cos"], arg["maxpos"],
                                caches, arg["nb"], arg["bs"], arg["H"], L, arg["eps"], rows,
                                arg["err"], None)


def test_store_rows_rejections(lib):
    assert _store_rows(lib, None) == rc.RC_ERR_INVALID_ARG
    assert "layer_rows" in last(lib)
    assert _store_rows(lib, [4, -1]) == rc.RC_ERR_INVALID_ARG
    assert "layer 1" in last(lib)
    assert _store_rows(lib, [4, 1 << 31]) == rc.RC_ERR_INVALID_ARG
    assert _store_rows(lib, [4, 2], H=5) == rc.RC_ERR_UNSUPPORTED
    assert _store_rows(lib, [0, 0]) == rc.RC_OK            # nothing to insert: no launch


def test_project_store_rows_rejections(lib):
    a, w = 0x100000, 0x4000000
    slots = (ctypes.c_void_p * 2)(A(0x8000), A(0x9000))
    caches = (ctypes.c_void_p * 2)(A(0x1000000), A(0x2000000))
    call = lambda rows, T=8: lib.rc_kv_project_store_rows(
        A(a), A(w), 0, 2, T, 8192, 8, None, slots, None, 0, caches, 4, 16, 1e-6,
        None if rows is None else (ctypes.c_int64 * 2)(*rows), None, None, None, 0, None)
    assert call(None) == rc.RC_ERR_INVALID_ARG
    assert call([8, 9]) == rc.RC_ERR_INVALID_ARG
    assert "outside [0, T]" in last(lib)
    assert call([-1, 0]) == rc.RC_ERR_INVALID_ARG
    assert call([0, 0], T=0) == rc.RC_OK


def test_qkv_front_rejections(lib):
    h, w, o = 0x10000, 0x1000000, 0x8000000
    call = lambda M=4, D=8192, nh=4, nkv=2, hidden=A(h), W=A(w), out=A(o), raw=None, slots=None, \
        cache=None, cos=None, pos=None, maxpos=0, nb=0, bs=0: lib.rc_qkv_front(
        hidden, M, D, W, nh, nkv, pos, cos, maxpos, slots, cache, nb, bs, 1e-6, out, raw, None, None)
    assert call(M=17) == rc.RC_ERR_UNSUPPORTED
    assert "16" in last(lib)
    assert call(D=100) == rc.RC_ERR_UNSUPPORTED
    assert call(nh=0) == rc.RC_ERR_INVALID_ARG
    assert call(hidden=None) == rc.RC_ERR_INVALID_ARG
    assert call(out=A(o + 8)) == rc.RC_ERR_INVALID_ARG
    assert call(cos=A(0x4000), maxpos=8) == rc.RC_ERR_INVALID_ARG          # no positions
    assert call(slots=A(0x5000)) == rc.RC_ERR_INVALID_ARG                  # no cache
    assert call(slots=A(0x5000), cache=A(0x6000), nb=1 << 20, bs=1 << 11) == rc.RC_ERR_INVALID_ARG
    assert call(out=A(w + 64)) == rc.RC_ERR_INVALID_ARG                    # out overlaps W
    assert "overlaps" in last(lib)
    assert call(M=0) == rc.RC_OK


def test_device_address_rejections(lib):
    # NULL arguments are refused before any CUDA call; without a GPU (or for
    # pageable memory) the runtime cannot address a host buffer: an error
    # status, dev left untouched
    d = ctypes.c_void_p(0x1234)
    assert lib.rc_device_address(None, ctypes.byref(d)) == rc.RC_ERR_INVALID_ARG
    assert "must not be NULL" in last(lib) and d.value == 0x1234
    buf = ctypes.create_string_buffer(64)
    assert lib.rc_device_address(ctypes.addressof(buf), None) == rc.RC_ERR_INVALID_ARG
    assert lib.rc_device_address(ctypes.addressof(buf), ctypes.byref(d)) == rc.RC_ERR_INVALID_ARG
    assert "rc_device_address" in last(lib) and d.value == 0x1234


def test_no_alloc_rejections(lib):
    """rc_kv_project_no_alloc refuses on the host, before any CUDA call,
    what rc_kv_project refuses: sizes, layout, NULL, misalignment, and out
    overlapping normed or W."""
    a, w, o = 0x100000, 0x4000000, 0x8000000
    call = lambda *args: lib.rc_kv_project_no_alloc(*args)
    assert call(A(a), A(w), 0, A(o), 1, 8, 8192, 100, None) == rc.RC_ERR_UNSUPPORTED
    assert call(A(a), A(w), 0, A(o), 1, 8, 8100, 1024, None) == rc.RC_ERR_UNSUPPORTED
    assert call(A(a), A(w), 7, A(o), 1, 8, 8192, 1024, None) == rc.RC_ERR_INVALID_ARG
    assert "layout" in last(lib) and "rc_kv_project_no_alloc" in last(lib)
    assert call(A(a), A(w), 0, A(o), 0, 8, 8192, 1024, None) == rc.RC_ERR_INVALID_ARG
    assert call(A(a), A(w), 0, A(o), 1, -1, 8192, 1024, None) == rc.RC_ERR_INVALID_ARG
    assert call(A(a), A(w), 0, A(o + 2), 1, 8, 8192, 1024, None) == rc.RC_ERR_INVALID_ARG
    assert "aligned" in last(lib)
    assert call(None, A(w), 0, A(o), 1, 8, 8192, 1024, None) == rc.RC_ERR_INVALID_ARG
    assert call(A(a), None, 0, A(o), 1, 8, 8192, 1024, None) == rc.RC_ERR_INVALID_ARG
    # out overlapping normed ([1, 8, 8192] bf16 = 128 KiB from a) or W
    assert call(A(a), A(w), 0, A(a + 4096), 1, 8, 8192, 1024, None) == rc.RC_ERR_INVALID_ARG
    assert "overlaps" in last(lib)
    assert call(A(a), A(w), 0, A(w + 4096), 1, 8, 8192, 1024, None) == rc.RC_ERR_INVALID_ARG
    # T == 0 succeeds without touching a device
    assert call(A(a), A(w), 0, A(o), 1, 0, 8192, 1024, None) == rc.RC_OK
    assert last(lib) == ""


NO_ALLOC_SCRATCH = 24 << 20     # RC_NO_ALLOC_SCRATCH_BYTES


def test_no_alloc_scratch_covers_every_plan_on_a_gb300():
    """Every projection plan a 152-SM GB300 makes for the workload shapes
    (and a sweep of T around them) fits the no-alloc call's static scratch,
    so none of them is refused."""
    from rope_chain_gb300 import _build
    _build.build()
    assert "RC_NO_ALLOC_SCRATCH_BYTES ((size_t)24 << 20)" in open(HEADER).read()
    shapes = [(1, 8192, 1024), (3, 8192, 1024), (4, 8192, 1024), (5, 8192, 2048),
              (8, 8192, 1024), (1, 8192, 128), (2, 1024, 128), (9, 8192, 1024), (1, 8192, 4096)]
    Ts = sorted({1, 2, 63, 64, 65, 100, 127, 128, 129, 255, 256, 257, 300, 384, 511, 512, 513,
                 1000, 1024, 2047, 2048, 3000, 4096, 6000, 8192, 10000, 16384, 20000, 32768,
                 65536, 131072})
    worst = 0
    for L, D, N in shapes:
        for T in Ts:
            nbytes = rc.workspace_size_for(L, T, D, N, 152)
            worst = max(worst, nbytes)
            assert nbytes <= NO_ALLOC_SCRATCH, (L, T, D, N, nbytes)
    assert worst > 16 << 20        # the sweep reaches plans near the bound
    # the planner needs no device: 0 for invalid sizes or SM counts
    assert rc.workspace_size_for(1, 64, 8192, 100, 152) == 0
    assert rc.workspace_size_for(1, 64, 8192, 1024, 0) == 0


def test_project_plan_describes_the_workloads():
    """rc_kv_project_plan, host-only: on a 152-SM GB300 the workloads run
    split-K single CTAs (1), split-K CTA pairs (2), persistent pairs with a
    tail launch (3) and persistent pairs taking tiles from a counter (4, 5);
    without a workspace nothing splits and the tile order is fixed."""
    from rope_chain_gb300 import _build
    _build.build()
    import workloads
    want = {1: ("single CTAs", 16, 0, False), 2: ("CTA pairs", 3, 0, False),
            3: ("persistent CTA pairs", 1, 2, False), 4: ("persistent CTA pairs", 1, 0, True),
            5: ("persistent CTA pairs", 1, 0, True)}
    for i, w in workloads.WORKLOADS.items():
        ws = rc.workspace_size_for(w.L, w.T, w.D, w.N, 152)
        p = rc.project_plan(w.L, w.T, w.D, w.N, 152, ws)
        assert (p["kernel"], p["splits"], p["tail_splits"], p["dynamic_tiles"]) == want[i], (i, p)
        assert p["workspace_bytes"] == ws
        assert p["tail_row0"] == (w.T if p["tail_splits"] == 0 else 2304)
        bare = rc.project_plan(w.L, w.T, w.D, w.N, 152, 0)
        assert bare["splits"] == 1 and bare["tail_splits"] == 0 and not bare["dynamic_tiles"]
        assert bare["workspace_bytes"] == 0
        # a workspace one byte short of the counter keeps the fixed order
        if p["dynamic_tiles"]:
            assert not rc.project_plan(w.L, w.T, w.D, w.N, 152, ws - 1)["dynamic_tiles"]
    # T = 0 launches nothing (the planner must not divide by its zero tiles)
    empty = rc.project_plan(2, 0, 8192, 1024, 152, 1 << 30)
    assert empty["kernel"] == "single CTAs" and empty["splits"] == 1
    assert empty["tail_splits"] == 0 and not empty["dynamic_tiles"] and empty["workspace_bytes"] == 0
    assert rc.workspace_size_for(2, 0, 8192, 1024, 152) == 0
    with pytest.raises(rc.RopeChainError):
        rc.project_plan(1, 64, 8192, 100, 152, 0)
    with pytest.raises(rc.RopeChainError):
        rc.project_plan(1, 64, 8192, 1024, 0, 0)


def test_chunked_chain_row_chunks():
    """rc_context_kv_chunks, host-only: the automatic choice gives each chunk
    after the first 12 rounds of tiles or more on 152 SMs (76 CTA pairs), at
    most 4 chunks, the first chunk about half the others (its norms run
    alone), and chunk sizes snapped to whole rounds of tiles (workload 5:
    8, 16, 16 and 13.9 rounds; workload 4: 2 chunks; workloads 1-3 one).
    Every boundary is a multiple of 256 rows, an explicit request is met
    down to chunks of one 256-row block, and every chunk's plan is persistent
    CTA pairs without workspace."""
    from rope_chain_gb300 import _build
    _build.build()
    import workloads
    want = {1: [0, 64], 2: [0, 512], 3: [0, 4096], 4: [0, 4864, 16384],
            5: [0, 4864, 14592, 24320, 32768]}
    for i, w in workloads.WORKLOADS.items():
        assert rc.context_kv_chunk_rows(w.L, w.T, w.H, 152) == want[i], i
        assert rc.context_kv_chunks(w.L, w.T, w.H, 152, 0) == len(want[i]) - 1
        assert rc.context_kv_chunks(w.L, w.T, w.H, 152, 1) == 1
        b = want[i]
        for c in range(1, len(b) - 1):          # the automatic chunks after the first
            rows = b[c + 1] - b[c]
            p = rc.project_plan(w.L, rows, w.D, w.N, 152, 256)
            assert p["dynamic_tiles"], (i, c)
    w5 = workloads.WORKLOADS[5]
    for n in (2, 3, 6, 8, 16):
        b = rc.context_kv_chunk_rows(w5.L, w5.T, w5.H, 152, n)
        assert 2 <= len(b) - 1 <= n and b[0] == 0 and b[-1] == w5.T
        assert all(r % 256 == 0 for r in b[:-1]) and all(x < y for x, y in zip(b, b[1:]))
        for x, y in zip(b, b[1:]):
            p = rc.project_plan(w5.L, y - x, w5.D, w5.N, 152, 256)
            assert p["kernel"] == "persistent CTA pairs" and p["splits"] == 1 and p["tail_splits"] == 0
            assert p["workspace_bytes"] <= 256
    assert rc.context_kv_chunks(3, 512, 8, 152, 4) == 2          # 256-row chunks at most
    assert rc.context_kv_chunks(2, 300, 1, 152, 4) == 1          # N = 128: no CTA pairs
    assert rc.context_kv_chunks(2, 256, 8, 152, 4) == 1          # one tile row: nothing to split
    assert rc.context_kv_chunks(2, 0, 8, 152, 4) == 0            # empty
    assert rc.context_kv_chunk_rows(2, 1024, 8, 152, 100) == [0, 256, 512, 768, 1024]
    assert rc.context_kv_chunks(2, 1024, 6, 152, 2) == 0         # H not a power of two
    assert rc.context_kv_chunks(2, 1024, 8, 1, 2) == 0           # no SMs to plan for
    assert rc.context_kv_chunks(65, 1024, 8, 152, 2) == 0        # more layers than a call stores
    # x in host memory: equal chunks, their count the least exposed first
    # chunk plus idle tile rounds (workload 5: 7 chunks of 19 blocks, whole
    # rounds; workload 4: 6; workload 3: 4 of 1024 rows; workload 2 one
    # chunk, its split-K projection leaving no round idle)
    host = {1: [0, 64], 2: [0, 512], 3: [0, 1024, 2048, 3072, 4096],
            4: [0, 2816, 5632, 8448, 11264, 14080, 16384],
            5: [4864 * i for i in range(7)] + [32768]}
    for i, w in workloads.WORKLOADS.items():
        assert rc.context_kv_chunk_rows(w.L, w.T, w.H, 152, x_on_host=True) == host[i], i
    assert rc.context_kv_chunk_rows(3, 2048, 8, 152, 3, x_on_host=True) == [0, 768, 1536, 2048]


def test_chunk_planner_fuzz():
    """Every size up to 64 blocks of 256 rows (and ragged ones), every chunk
    request and both x locations, on a few shapes and SM counts: the host
    planner returns chunks that cover the rows once, start on 256-row
    boundaries and number at most 16, and never fails on valid sizes."""
    from rope_chain_gb300 import _build
    _build.build()
    sizes = list(range(1, 2048, 37)) + [256 * b for b in range(1, 65)] + [256 * b + 1 for b in range(1, 65)]
    for L, H in ((1, 2), (3, 8), (8, 8), (5, 16), (2, 1)):
        for sms in (152, 148, 132):
            for T in sizes:
                for req in (0, 1, 2, 3, 5, 8, 16, 17, 100):
                    for host in (False, True):
                        b = rc.context_kv_chunk_rows(L, T, H, sms, req, x_on_host=host)
                        assert b and b[0] == 0 and b[-1] == T, (L, H, sms, T, req, host, b)
                        assert all(x < y for x, y in zip(b, b[1:])), b
                        assert all(r % 256 == 0 for r in b[:-1]), b
                        assert len(b) - 1 <= 16 and (req != 1 or len(b) == 2), b
