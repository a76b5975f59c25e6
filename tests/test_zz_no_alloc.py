"""rc_kv_project_no_alloc, the projection for callers that cannot allocate
device memory (its split-K scratch is a static array inside the library).

Called through the C ABI on two calls in a row, for shapes that use its
scratch (split-K partials, a tail launch's partials, or the counter from
which the persistent kernel's CTA pairs take tiles):
each output must be bit-identical to rc_kv_project given a full workspace
(the same plan and kernels), and within the projection tolerance the other
tests use of the oracle's float64 product.  Also: the Python wrapper, an
empty call, and refused calls that must leave `out` untouched.  This file is
collected last so a run that stops at the first failure has run every other
test first.
"""
import ctypes

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


def _call(a_d, w_d, layout, out, L, T, D, N):
    stream = torch.cuda.current_stream().cuda_stream
    return rc.lib().rc_kv_project_no_alloc(
        ctypes.c_void_p(a_d.data_ptr() if a_d is not None else 0),
        ctypes.c_void_p(w_d.data_ptr()), layout, ctypes.c_void_p(out.data_ptr()),
        L, T, D, N, ctypes.c_void_p(stream))


@pytest.mark.parametrize("L,T,D,H,layout", [(3, 512, 8192, 8, rc.RC_W_KN),
                                            (3, 128, 8192, 8, rc.RC_W_KN),
                                            (1, 64, 8192, 8, rc.RC_W_KN),
                                            (2, 100, 1024, 1, rc.RC_W_NK),
                                            (4, 4096, 8192, 8, rc.RC_W_KN),
                                            (4, 8192, 1024, 16, rc.RC_W_KN)])
def test_no_alloc_matches_workspace_path_twice(L, T, D, H, layout):
    N = 128 * H
    rng = np.random.default_rng(L * 1000 + T)
    a = workloads.normal_bf16(rng, (L, T, D), 0.0, 1.0)
    W = workloads.normal_bf16(rng, (L, D, N), 0.0, 0.02)
    Wl = W if layout == rc.RC_W_KN else np.ascontiguousarray(W.transpose(0, 2, 1))
    a_d, w_d = parity.dev_bf16(a, DEV), parity.dev_bf16(Wl, DEV)
    nbytes = rc.workspace_size(L, T, D, N)
    assert nbytes > 0, "this shape should use scratch (split-K partials or the tile counter)"
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    ref = rc.kv_project(a_d, w_d, w_layout=layout, workspace=ws)
    torch.cuda.synchronize()
    ref_bits = parity.host_bits(ref)
    # the oracle's float64 product, on every row (small T) or sampled rows
    rows = None if L * T <= 1536 else np.unique(np.r_[0, T - 1, np.linspace(0, T - 1, 64).astype(np.int64)])
    ref64, absum = oracle.kv_project(a, W, rows=rows)
    sel = (lambda x: x) if rows is None else (lambda x: x[:, rows])
    for call in range(2):
        out = torch.full((L, T, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        status = _call(a_d, w_d, layout, out, L, T, D, N)
        assert status == rc.RC_OK, rc.lib().rc_last_error().decode()
        torch.cuda.synchronize()
        bits = parity.host_bits(out)
        diff = np.argwhere(bits != ref_bits)
        assert diff.size == 0, (f"no-alloc call {call + 1} differs from rc_kv_project with a "
                                f"workspace at {len(diff)} elements, first {tuple(diff[0])}")
        parity.assert_projection_close(sel(bits), ref64, absum, what=f"no-alloc call {call + 1}")
    assert rc.read_device_faults(clear=True) == 0


def test_no_alloc_wrapper_empty_call_and_refusals():
    L, T, D, H = 2, 300, 1024, 2
    N = 128 * H
    rng = np.random.default_rng(77)
    a = workloads.normal_bf16(rng, (L, T, D), 0.0, 1.0)
    W = workloads.normal_bf16(rng, (L, D, N), 0.0, 0.02)
    a_d, w_d = parity.dev_bf16(a, DEV), parity.dev_bf16(W, DEV)
    ws = torch.zeros(max(rc.workspace_size(L, T, D, N), 16), dtype=torch.uint8, device=DEV)
    ref = parity.host_bits(rc.kv_project(a_d, w_d, workspace=ws))
    # the Python wrapper
    out = torch.full((L, T, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    assert rc.kv_project_no_alloc(a_d, w_d, out) is out
    torch.cuda.synchronize()
    assert np.array_equal(parity.host_bits(out), ref)
    with pytest.raises(ValueError):
        rc.kv_project_no_alloc(a_d, w_d, out[:, :T - 1])          # out of the wrong shape
    with pytest.raises(ValueError):
        rc.kv_project_no_alloc(a_d, w_d[:, :D // 2], out)          # W not [L, D, N]
    # refused calls and an empty call leave out untouched
    nan = torch.full((L, T, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    before = parity.host_bits(nan)
    flat = nan.view(-1)
    assert _call(None, w_d, rc.RC_W_KN, nan, L, T, D, N) == rc.RC_ERR_INVALID_ARG
    assert _call(a_d, w_d, 5, nan, L, T, D, N) == rc.RC_ERR_INVALID_ARG
    assert _call(a_d, w_d, rc.RC_W_KN, flat[1:], L, T, D, N) == rc.RC_ERR_INVALID_ARG   # misaligned
    assert _call(a_d, w_d, rc.RC_W_KN, nan, L, T, D, 100) == rc.RC_ERR_UNSUPPORTED
    assert _call(a_d, w_d, rc.RC_W_KN, nan, 0, T, D, N) == rc.RC_ERR_INVALID_ARG
    assert _call(a_d, w_d, rc.RC_W_KN, nan, L, 0, D, N) == rc.RC_OK                     # empty
    # out overlapping normed
    assert _call(a_d, w_d, rc.RC_W_KN, a_d, L, T, D, N) == rc.RC_ERR_INVALID_ARG
    assert "overlaps" in rc.lib().rc_last_error().decode()
    torch.cuda.synchronize()
    assert np.array_equal(parity.host_bits(nan), before)
    assert np.array_equal(parity.host_bits(a_d), a.view(np.uint16))
    assert rc.read_device_faults(clear=True) == 0
