"""Writes stay inside their buffers.  Every output of the C ABI (normed rows,
projection, caches, the QKV front's outputs) is a view in the middle of one
allocation with 4 KiB of sentinel-filled slack before and after it; after
the call the slack must be untouched.  rows = 0 inserts nothing."""
import numpy as np
import pytest
import torch

import rope_chain_gb300 as rc
import workloads
from tests import parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
PAD = 2048                         # bf16 elements (4 KiB) on each side


@pytest.fixture(scope="module", autouse=True)
def built():
    from rope_chain_gb300 import _build
    _build.build()
    rc.read_device_faults(clear=True)
    yield
    assert rc.read_device_faults(clear=True) == 0


class Guarded:
    """A bf16 view of ``shape`` inside a sentinel-filled allocation."""

    def __init__(self, shape, fill=parity.SENTINEL):
        self.n = int(np.prod(shape))
        self.whole = torch.full((self.n + 2 * PAD,), fill, dtype=torch.int16, device=DEV)
        self.view = self.whole[PAD:PAD + self.n].view(torch.bfloat16).view(shape)

    def check(self, what):
        head, tail = self.whole[:PAD], self.whole[PAD + self.n:]
        assert bool((head == parity.SENTINEL).all()), f"{what}: write before the buffer"
        assert bool((tail == parity.SENTINEL).all()), f"{what}: write after the buffer"


def _operands(T, L, H, seed):
    c = workloads.random_case(seed, T=T, L=L, H=H, max_position=256,
                              num_blocks=(T + 15) // 16 + 2, block_size=16)
    d = lambda a: parity.dev_bf16(a, DEV)
    return c, dict(x=d(c["x"]), hw=d(c["hidden_w"]), pw=d(c["pre_w"]), W=d(c["W"]),
                   cs=d(c["cos_sin"]), pos=torch.from_numpy(c["positions"]).to(DEV),
                   slots=[torch.from_numpy(s).to(DEV) for s in c["slots"]])


@pytest.mark.parametrize("T,L,H,split", [(129, 2, 8, False), (300, 3, 2, True),
                                         (1000, 2, 4, False), (64, 1, 8, True)])
def test_step_outputs_stay_in_bounds(T, L, H, split):
    c, o = _operands(T, L, H, 900 + T)
    N = 128 * H
    normed = Guarded((L, T, 8192))
    rc.context_norms(o["x"], o["hw"], o["pw"], L, c["eps"], out=normed.view)
    ws = rc.new_workspace(L, T, 8192, N, DEV) if split else None
    kv = Guarded((L, T, N))
    rc.kv_project(normed.view, o["W"], out=kv.view, workspace=ws)
    caches = [Guarded(c["cache_shape"]) for _ in range(L)]
    rc.kv_store_from_projection(kv.view, H, o["pos"], o["slots"], o["cs"],
                                [g.view for g in caches], c["eps"])
    kv2 = Guarded((L, T, N))
    caches2 = [Guarded(c["cache_shape"]) for _ in range(L)]
    rc.kv_project_store(normed.view, o["W"], H, o["pos"], o["slots"], o["cs"],
                        [g.view for g in caches2], c["eps"], kv_out=kv2.view, workspace=ws)
    torch.cuda.synchronize()
    for g, what in [(normed, "normed"), (kv, "kv"), (kv2, "kv_out")]:
        g.check(what)
    for l in range(L):
        caches[l].check(f"cache {l}")
        caches2[l].check(f"fused cache {l}")
        assert torch.equal(caches2[l].whole, caches[l].whole)
    assert torch.equal(kv2.view, kv.view)


def test_whole_chain_and_front_stay_in_bounds():
    T, L, H = 300, 2, 8
    c, o = _operands(T, L, H, 31)
    caches = [Guarded(c["cache_shape"]) for _ in range(L)]
    kv = Guarded((L, T, 128 * H))
    ws = rc.context_kv_workspace(L, T, H, DEV)
    rc.context_kv(o["x"], o["hw"], o["pw"], o["W"], H, o["pos"], o["slots"], o["cs"],
                  [g.view for g in caches], c["eps"], ws, kv_out=kv.view)
    f = workloads.front_case(77, 7, num_heads=4, num_kv_heads=2, max_position=256,
                             num_blocks=4, block_size=16)
    Nq = 64 * (2 * 4 + 2 * 2)
    d = lambda a: parity.dev_bf16(a, DEV)
    cache = Guarded(f["cache_shape"])
    out, raw = Guarded((7, Nq)), Guarded((7, Nq))
    rc.qkv_front(d(f["hidden"]), d(f["W"]), 4, 2, torch.from_numpy(f["positions"]).to(DEV),
                 d(f["cos_sin"]), torch.from_numpy(f["slots"]).to(DEV), cache.view, f["eps"],
                 out=out.view, raw_out=raw.view)
    torch.cuda.synchronize()
    kv.check("kv_out")
    for l in range(L):
        caches[l].check(f"cache {l}")
    for g, what in [(cache, "front cache"), (out, "front out"), (raw, "front raw_out")]:
        g.check(what)


@pytest.mark.parametrize("call", ["store", "project_store", "context_kv"])
def test_rows_zero_inserts_nothing(call):
    T, L, H = 300, 2, 4
    c, o = _operands(T, L, H, 55)
    caches = [Guarded(c["cache_shape"]) for _ in range(L)]
    cv = [g.view for g in caches]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    normed = rc.context_norms(o["x"], o["hw"], o["pw"], L, c["eps"])
    split_ws = rc.new_workspace(L, T, 8192, 128 * H, DEV)     # the plan context_kv takes
    kv = rc.kv_project(normed, o["W"], workspace=split_ws)
    kv2 = torch.zeros_like(kv)
    if call == "store":
        rc.kv_store_from_projection(kv, H, o["pos"], o["slots"], o["cs"], cv, c["eps"], rows=0,
                                    err=err)
    elif call == "project_store":
        rc.kv_project_store(normed, o["W"], H, o["pos"], o["slots"], o["cs"], cv, c["eps"],
                            rows=0, err=err, kv_out=kv2, workspace=split_ws)
    else:
        ws = rc.context_kv_workspace(L, T, H, DEV)
        rc.context_kv(o["x"], o["hw"], o["pw"], o["W"], H, o["pos"], o["slots"], o["cs"], cv,
                      c["eps"], ws, rows=0, err=err, kv_out=kv2)
    torch.cuda.synchronize()
    for l in range(L):
        assert bool((caches[l].whole == parity.SENTINEL).all()), f"cache {l} written"
    assert int(err.item()) == 0
    if call != "store":
        assert torch.equal(kv2, kv)            # the projection itself is still written
