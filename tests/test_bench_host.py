"""bench.py's host-side arithmetic on CPU: the algorithmic byte and FLOP
counts behind the roofline figures, the clock summary behind the
throttle check, and the L2 flush sizes.  The counts are checked against
sums taken element by element over the operands, not against the formulas
themselves."""
import numpy as np

import bench
import workloads

L2_BYTES = 129 * 10**6        # GB300's L2


def test_norm_and_projection_counts_by_operand():
    for w in workloads.WORKLOADS.values():
        c = bench.algorithmic_counts(w, splits=1)
        # norms: x read once, L rows written, and each gain vector read once
        operands = [(w.T, w.D)] + [(w.T, w.D)] * w.L
        if w.hidden_weighted:
            operands.append((w.D,))
        if w.pre_weighted:
            operands += [(w.D,)] * w.L
        assert c["k1_bytes"] == sum(2 * int(np.prod(s)) for s in operands)
        # projection: one multiply and one add per (layer, row, k, column)
        assert c["k2_flops"] == 2 * w.L * w.T * w.D * w.N
        assert c["k2_bytes"] == 2 * (w.L * w.T * w.D + w.L * w.D * w.N + w.L * w.T * w.N)
    w2 = workloads.WORKLOADS[2]
    assert bench.algorithmic_counts(w2, 3)["k1_bytes"] == 33_619_968
    assert bench.algorithmic_counts(w2, 3)["k2_flops"] == 25_769_803_776


def test_store_bytes_counts_live_rows():
    w = workloads.WORKLOADS[2]
    cap = w.num_blocks * w.block_size
    rng = np.random.default_rng(5)
    slots = [rng.integers(-3, cap + 3, size=40).astype(np.int64) for _ in range(2)]
    for rope in (False, True):
        expect = 0
        for s in slots:
            for v in s:
                expect += 8                           # the slot itself
                if 0 <= v < cap:
                    expect += w.H * 64 * 2 * 2        # K and V read
                    expect += w.H * 128 * 2           # the cache row written
                    if rope:
                        expect += 8 + 64 * 2          # position and table row
        assert bench.store_bytes(w, slots, rope) == expect


def test_project_store_bytes_by_operand():
    w = workloads.WORKLOADS[2]
    cap = w.num_blocks * w.block_size
    rng = np.random.default_rng(9)
    slots = [rng.integers(-3, cap + 3, size=w.T).astype(np.int64) for _ in range(w.L)]
    for rope in (False, True):
        expect = w.L * w.T * w.D * 2 + w.L * w.D * w.N * 2     # normed rows and W, once
        for s in slots:
            for v in s:
                expect += 8
                if 0 <= v < cap:
                    expect += w.H * 128 * 2                     # the cache row written
                    if rope:
                        expect += 8 + 64 * 2
        assert bench.project_store_bytes(w, slots, rope) == expect


def test_front_bytes_by_operand():
    M, nh, nkv, D = 3, 4, 2, 256
    case = workloads.front_case(11, M, D=D, num_heads=nh, num_kv_heads=nkv)
    N = case["W"].shape[0]
    live = M
    expect = (case["W"].nbytes + case["hidden"].nbytes + M * N * 2 + case["positions"].nbytes
              + case["slots"].nbytes + M * case["cos_sin"].shape[1] * 2 + live * nkv * 128 * 2)
    assert bench.front_bytes(M, D, N, nkv, live) == expect


def test_clock_summary():
    lines = [
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
        "0, 1950, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
        "0, 1980, 2070, 1380.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
        "garbage line\n",
    ]
    c = bench.summarise_clocks(lines)
    assert c == {"sm_mhz": 1980.0, "sm_max_mhz": 2070.0, "power_w": 1380.0, "reasons": ["sw_power_cap"],
                 "samples": 3}
    hot = lines[:1] + ["0, 1500, 2070, 1200.0, 0x48, Active, Active, Not Active, Not Active\n"]
    assert bench.summarise_clocks(hot)["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
    assert bench.summarise_clocks(["\n"]) is None


def test_flush_buffers_exceed_l2():
    assert bench.L2_FLUSH_BYTES > L2_BYTES and bench.L2_CLEAN_BYTES > L2_BYTES
    f = bench.L2Flush("cpu")
    f(7)
    assert f.w.numel() == bench.L2_FLUSH_BYTES and int(f.w[0]) == 7
    assert f.r.numel() * f.r.element_size() == bench.L2_CLEAN_BYTES


def test_row_chunks_cover_rows_once():
    for T in (1, 5, 64, 512, 600, 4096, 16384, 32768):
        for n in (0, 1, 2, 3, 8):
            ch = bench.row_chunks(T, n)
            assert ch[0][0] == 0 and ch[-1][1] == T
            assert all(a < b for a, b in ch)
            assert all(ch[i][1] == ch[i + 1][0] for i in range(len(ch) - 1))
            assert max(b - a for a, b in ch) - min(b - a for a, b in ch) <= 1
            if n > 0:
                assert len(ch) == min(n, T)
    assert len(bench.row_chunks(512, 0)) == 1 and len(bench.row_chunks(4096, 0)) == 4
    assert len(bench.row_chunks(16384, 0)) == 8


def test_e2e_plan():
    """The end-to-end step: one in-place call where the chunked call splits x
    held in host memory itself; copied ranges on the store path otherwise;
    one in-place range on the other paths."""
    # workload 5: the chunked call's host plan has 7 chunks -> one call
    assert bench.e2e_plan("store", 32768, 7, 0, "auto") == ([(0, 32768)], "inplace")
    # the two calls (no host chunks) -> 8 copied ranges
    ch, mode = bench.e2e_plan("store", 32768, 1, 0, "auto")
    assert len(ch) == 8 and mode == "copy"
    # ranges asked for win over the chunked call's own plan
    ch, mode = bench.e2e_plan("store", 32768, 7, 4, "inplace")
    assert len(ch) == 4 and mode == "inplace"
    # below 2048 rows one range reads x in place
    assert bench.e2e_plan("store", 512, 1, 0, "auto") == ([(0, 512)], "inplace")
    # the variants and whole paths: one range (the variants' chunked call
    # splits x itself)
    assert bench.e2e_plan("variants", 32768, 7, 0, "auto") == ([(0, 32768)], "inplace")
    assert bench.e2e_plan("whole", 32768, 1, 0, "copy") == ([(0, 32768)], "inplace")


def test_traffic_figures_expire_with_their_sources(tmp_path, monkeypatch):
    """A stored ncu traffic figure is reported only while the sources of its
    call's kernels are those it was measured on: a change to the projection
    kernel's file voids the projection's figures, not the norms'."""
    import os
    import shutil
    src = os.path.join(bench.ROOT, "rope_chain_gb300", "csrc")
    dst = tmp_path / "rope_chain_gb300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the stored figures as if taken on the sources of this tree
    fresh = {k: (v[0], bench.source_digest(bench.CALL_SOURCES[k[2]]), v[2])
             for k, v in bench.NCU_TRAFFIC.items()}
    monkeypatch.setattr(bench, "NCU_TRAFFIC", fresh)
    keys = list(bench.NCU_TRAFFIC)
    assert keys and all(bench.ncu_traffic(k)[0] is not None for k in keys)
    with open(dst / "k2_gemm.cu", "a") as f:
        f.write("\n// changed\n")
    for k in keys:
        nbytes, note = bench.ncu_traffic(k)
        if "k2_gemm.cu" in bench.CALL_SOURCES[k[2]]:
            assert nbytes is None and "predates" in note
        else:
            assert nbytes == bench.NCU_TRAFFIC[k][0]
    assert bench.ncu_traffic((9, "store", "project_store"))[0] is None
