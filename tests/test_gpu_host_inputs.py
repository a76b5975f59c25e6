"""Inputs read in place from pinned host memory (rc_device_address): the
norms, the norm options, the row pass and the whole chain given x as a
pinned CPU tensor equal their results from a device copy of x, bit for bit;
pageable host memory is refused before anything launches."""
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


def _pinned_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()


def test_device_address():
    d = torch.empty(64, dtype=torch.bfloat16, device=DEV)
    assert rc.device_address(d) == d.data_ptr()
    h = torch.empty(64, dtype=torch.bfloat16).pin_memory()
    assert rc.device_address(h) != 0
    with pytest.raises(TypeError):
        rc.device_address(torch.empty(64, dtype=torch.bfloat16))      # pageable
    # the C call itself refuses pageable memory with an error, not a fault
    buf = ctypes.create_string_buffer(64)
    out = ctypes.c_void_p(0)
    assert rc.lib().rc_device_address(ctypes.addressof(buf), ctypes.byref(out)) == rc.RC_ERR_INVALID_ARG
    assert out.value is None


@pytest.mark.parametrize("T,L", [(1, 1), (512, 3), (129, 9), (2000, 2)])
def test_norms_from_host_x(T, L):
    case = workloads.random_case(600 + T, T=T, L=L, H=1, num_blocks=(T + 15) // 16 + 1, block_size=16)
    hw, pw = parity.dev_bf16(case["hidden_w"], DEV), parity.dev_bf16(case["pre_w"], DEV)
    x_h = _pinned_bf16(case["x"])
    a = rc.context_norms(x_h.to(DEV), hw, pw, L, 1e-5)
    b = rc.context_norms(x_h, hw, pw, L, 1e-5)
    c = rc.context_norms_ex(x_h, L, hidden_w=hw.float(), pre_w=pw.float(), hidden_eps=1e-5,
                            pre_eps=1e-4, pre_center=1.0, hidden_input_scale=True)
    d = rc.context_norms_ex(x_h.to(DEV), L, hidden_w=hw.float(), pre_w=pw.float(), hidden_eps=1e-5,
                            pre_eps=1e-4, pre_center=1.0, hidden_input_scale=True)
    z1, r1 = rc.context_rows(x_h, hw, 1e-5)
    z2, r2 = rc.context_rows(x_h.to(DEV), hw, 1e-5)
    torch.cuda.synchronize()
    assert b.is_cuda and torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(c.view(torch.int16), d.view(torch.int16))
    assert torch.equal(z1.view(torch.int16), z2.view(torch.int16)) and torch.equal(r1, r2)


def test_whole_chain_from_host_x():
    w = workloads.WORKLOADS[2]
    case = workloads.make_inputs(w)
    x_h = _pinned_bf16(case["x"])
    hw, pw, W = (parity.dev_bf16(case[k], DEV) for k in ("hidden_w", "pre_w", "W"))
    cs = parity.dev_bf16(case["cos_sin"], DEV)
    pos = torch.from_numpy(case["positions"]).to(DEV)
    slots = [torch.from_numpy(s).to(DEV) for s in case["slots"]]
    ws = rc.context_kv_workspace(w.L, w.T, w.H, DEV)
    got = []
    for xs in (x_h.to(DEV), x_h):
        caches = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, w.L, parity.SENTINEL)]
        kv = torch.empty((w.L, w.T, w.N), dtype=torch.bfloat16, device=DEV)
        rc.context_kv(xs, hw, pw, W, w.H, pos, slots, cs, caches, w.eps, ws, kv_out=kv)
        torch.cuda.synchronize()
        got.append((parity.host_bits(kv), [parity.host_bits(c) for c in caches]))
    assert np.array_equal(got[0][0], got[1][0])
    for a, b in zip(got[0][1], got[1][1]):
        assert np.array_equal(a, b)


def test_slice_of_pinned_buffer():
    # a row range of a pinned x is read at its own offset
    case = workloads.random_case(640, T=300, L=2, H=1, num_blocks=24, block_size=16)
    hw, pw = parity.dev_bf16(case["hidden_w"], DEV), parity.dev_bf16(case["pre_w"], DEV)
    x_h = _pinned_bf16(case["x"])
    assert rc.device_address(x_h[100:]) == rc.device_address(x_h) + 100 * 8192 * 2
    a = rc.context_norms(x_h[100:230], hw, pw, 2, 1e-5)
    b = rc.context_norms(x_h.to(DEV)[100:230], hw, pw, 2, 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("T,L,H,n,mode", [(600, 3, 8, 3, "inplace"), (512, 3, 8, 2, "inplace"),
                                          (1000, 2, 16, 4, "inplace"), (600, 3, 8, 3, "copy"),
                                          (1000, 2, 16, 5, "copy"), (513, 3, 8, 2, "copy")])
def test_overlapped_ranges_from_host_x(T, L, H, n, mode):
    # bench.py's end-to-end pass: row range c + 1 of x crosses from pinned
    # host memory (copied by the copy engines into one of two device
    # buffers, or read in place by the norms kernel) while range c goes
    # through the chain.  Its caches equal those of the same calls made one
    # after another from device memory, and those match the oracle.
    import oracle
    import bench
    oracle.build()
    N = 128 * H
    case = workloads.random_case(700 + T + H, T=T, L=L, H=H, max_position=512,
                                 num_blocks=(T + 15) // 16 + 4, block_size=16)
    hw, pw, W = (parity.dev_bf16(case[k], DEV) for k in ("hidden_w", "pre_w", "W"))
    cs = parity.dev_bf16(case["cos_sin"], DEV)
    pos = torch.from_numpy(case["positions"]).to(DEV)
    slots = [torch.from_numpy(s).to(DEV) for s in case["slots"]]
    x_h = _pinned_bf16(case["x"])
    chunks = bench.row_chunks(T, n)
    assert len(chunks) == n

    caches_a = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
    err_a = torch.zeros(1, dtype=torch.int32, device=DEV)
    run = bench.OverlappedChain(L, T, 8192, N, chunks, DEV, mode)
    for _ in range(2):                     # a second pass rewrites the same bits
        run(x_h, hw, pw, W, H, pos, slots, cs, caches_a, case["eps"], err_a)
    torch.cuda.synchronize()

    caches_b = [parity.dev_bf16(c, DEV) for c in parity.make_caches(case, L, parity.SENTINEL)]
    err_b = torch.zeros(1, dtype=torch.int32, device=DEV)
    xd = x_h.to(DEV)
    kvs = []
    for r0, r1 in chunks:
        nc = rc.context_norms(xd[r0:r1], hw, pw, L, case["eps"])
        kv = torch.empty((L, r1 - r0, N), dtype=torch.bfloat16, device=DEV)
        rc.kv_project_store(nc, W, H, pos[r0:r1], [s[r0:r1] for s in slots], cs, caches_b,
                            case["eps"], err=err_b, kv_out=kv,
                            workspace=rc.new_workspace(L, r1 - r0, 8192, N, DEV))
        kvs.append(parity.host_bits(kv))
    torch.cuda.synchronize()
    for a, b in zip(caches_a, caches_b):
        assert np.array_equal(parity.host_bits(a), parity.host_bits(b))
    assert int(err_a.item()) == 2 * int(err_b.item())

    kv = np.concatenate(kvs, axis=1)
    normed = oracle.context_norms(case["x"], case["hidden_w"], case["pre_w"], L, case["eps"])
    edges = [r for c in chunks for r in c]
    sample = np.unique(np.r_[edges[:-1], [e - 1 for e in edges[1:]], np.linspace(0, T - 1, 60).astype(int)])
    ref64, ab = oracle.kv_project(normed, case["W"], rows=sample)
    parity.assert_projection_close(kv[:, sample], ref64, ab, "projection by row ranges")
    ref_caches = parity.make_caches(case, L, parity.SENTINEL)
    ref_err = oracle.kv_store_from_projection(kv, H, case["positions"], case["slots"],
                                              case["cos_sin"], ref_caches, case["eps"], T)
    for g, r in zip(caches_b, ref_caches):
        assert np.array_equal(parity.host_bits(g), r)
    assert int(err_b.item()) == ref_err
