"""rc_kv_project_no_alloc, the projection for callers that cannot allocate
device memory (its split-K scratch is a static array inside the library).

Called through the C ABI and compared with rc_kv_project (given a workspace
of its own) within the projection tolerance the other tests use, on two
calls in a row, for shapes that split K.  This file is collected last so a
run that stops at the first failure has run every other test first.
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


@pytest.mark.parametrize("L,T,D,H,layout", [(3, 512, 8192, 8, rc.RC_W_KN),
                                            (3, 128, 8192, 8, rc.RC_W_KN),
                                            (1, 64, 8192, 8, rc.RC_W_KN),
                                            (2, 100, 1024, 1, rc.RC_W_NK)])
def test_no_alloc_matches_workspace_path_twice(L, T, D, H, layout):
    N = 128 * H
    rng = np.random.default_rng(L * 1000 + T)
    a = workloads.normal_bf16(rng, (L, T, D), 0.0, 1.0)
    W = workloads.normal_bf16(rng, (L, D, N), 0.0, 0.02)
    Wl = W if layout == rc.RC_W_KN else np.ascontiguousarray(W.transpose(0, 2, 1))
    a_d, w_d = parity.dev_bf16(a, DEV), parity.dev_bf16(Wl, DEV)
    nbytes = rc.workspace_size(L, T, D, N)
    assert nbytes > 0, "this shape should split K"
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    ref = rc.kv_project(a_d, w_d, w_layout=layout, workspace=ws)
    torch.cuda.synchronize()
    ref_bits = parity.host_bits(ref)
    ref_f64 = (ref_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    _, absum = oracle.kv_project(a, W)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full((L, T, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        status = rc.lib().rc_kv_project_no_alloc(
            ctypes.c_void_p(a_d.data_ptr()), ctypes.c_void_p(w_d.data_ptr()), layout,
            ctypes.c_void_p(out.data_ptr()), L, T, D, N, ctypes.c_void_p(stream))
        assert status == rc.RC_OK, rc.lib().rc_last_error().decode()
        torch.cuda.synchronize()
        parity.assert_projection_close(parity.host_bits(out), ref_f64, absum,
                                       what=f"no-alloc call {call + 1}")
    assert rc.read_device_faults(clear=True) == 0
