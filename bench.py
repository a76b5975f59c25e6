"""Benchmark of the context K/V chain (norms -> projection -> store).

One step = one pass of the whole chain over one batch of context rows of a
workload (default: workload 5, the largest: T=32768 rows, L=8 layers, H=8 KV
heads, RoPE), inputs resident in HBM.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I]
  python bench.py --impl reference ...   # the CPU oracle as the reference arm

Under torchrun (N > 1) every rank runs its own replica of the workload on
its own GPU (the rows of different batches are independent: weak scaling,
no collective on the data path); the timed region is bracketed by a barrier
and a device synchronisation, and the slowest rank's time counts.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "context rows/s through norm+proj+store; norm/store HBM GB/s vs GB300 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20          # > 129 MB L2: written between timed steps
L2_CLEAN_BYTES = 256 << 20          # > 129 MB L2: then read, so the written lines leave it


# DRAM bytes (read + write) per call, from ncu captures of this bench
# command (dram__bytes_read.sum + dram__bytes_write.sum, summed over the
# kernels the call launches), keyed by (workload, path, call): (bytes,
# digest of the sources the call's kernels are built from, how).  The digest
# (source_digest(CALL_SOURCES[call])) covers the call's kernel file, the
# shared headers and the host launch path; when one of them changes the
# figure no longer describes the kernels and the bench reports traffic as
# null.
_SHARED_SOURCES = ("rc_internal.cuh", "rc_api.cu")
CALL_SOURCES = {
    "project_store": ("k2_gemm.cu", "k3_store.cu", "rc_tcgen05.cuh") + _SHARED_SOURCES,
    "norms": ("k1_norms.cu",) + _SHARED_SOURCES,
    "store": ("k3_store.cu",) + _SHARED_SOURCES,
    "k4_qkv_front": ("k4_qkv_front.cu", "rc_tcgen05.cuh") + _SHARED_SOURCES,
}
NCU_TRAFFIC = {
    # rc_kv_project_store at workload 5 over all rows (the breakdown's call,
    # the one the roofline times): one k2_project_pair_persistent launch
    # (dynamic tile order), 4,861,931,520 B read + 527,136,512 B written
    # (profiles/k2_pair_persistent_workload5.md)
    (5, "store", "project_store"): (5_389_068_032, "8bb10d3211a5d91f",
                                    "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, "
                                    "one launch at full size (one pass)"),
    # rc_context_norms at workload 5: one k1_context_norms2 launch,
    # 537,302,016 B read + 4,233,134,336 B written
    (5, "unfused", "norms"): (4_770_436_352, "2655d675e990d059",
                              "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, "
                              "one launch at full size (one pass)"),
    # rc_kv_store at workload 5: one k3_kv_store_heads launch (8 layers),
    # 574,425,600 B read + 482,196,992 B written
    (5, "unfused", "store"): (1_056_622_592, "b4f44c2c856746c9",
                              "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, "
                              "one launch at full size (one pass)"),
    # rc_kv_project_store at workload 2: k2_project_pair (52,795,648 B read,
    # 19,434,752 B written) then k3_reduce_store (82,688 B read, 1,630,976 B
    # written), captured in sequence without ncu's cache flush between them
    # (the split-K partials are read back from L2, as in the step)
    (2, "store", "project_store"): (73_944_064, "8bb10d3211a5d91f",
                                    "ncu --cache-control none --metrics dram__bytes_read.sum,"
                                    "dram__bytes_write.sum, the call's two launches in sequence"),
}


def source_digest(names) -> str:
    """Short digest of the named sources under rope_chain_gb300/csrc, in
    name order."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "rope_chain_gb300", "csrc")
    for name in sorted(names):
        h.update(name.encode())
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(key):
    """(bytes, note) of NCU_TRAFFIC[key] when it was measured on the current
    sources, else (None, why)."""
    entry = NCU_TRAFFIC.get(key)
    if entry is None:
        return None, "no ncu capture of this call at this workload"
    nbytes, digest, how = entry
    if digest != source_digest(CALL_SOURCES[key[2]]):
        return None, "the ncu capture predates the current kernel sources"
    return nbytes, how


class L2Flush:
    """Run before each timed step: a write of a buffer larger than L2, then a
    read of another one larger than L2.  The step starts with a cold L2 that
    holds only clean lines: the written lines are written back to HBM during
    the read, not during the step that follows (with the write alone, the
    step would pay for up to 129 MB of the flush's own write-back)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_CLEAN_BYTES // 4, dtype=torch.int32, device=dev)
        self.s = torch.empty(1, dtype=torch.int32, device=dev)

    def __call__(self, i: int):
        import torch
        self.w.fill_(i & 0xFF)
        torch.sum(self.r, dim=0, keepdim=True, dtype=torch.int32, out=self.s)


def row_chunks(T: int, n: int):
    """n nearly equal row ranges covering rows 0..T-1; n = 0 picks 8 ranges
    from 16384 rows, 4 from 2048 rows and one range below that (at 512 rows
    the ranges' smaller projections cost more than the overlap saves)."""
    if n <= 0:
        n = 8 if T >= 16384 else (4 if T >= 2048 else 1)
    n = max(1, min(n, T))
    edges = [T * i // n for i in range(n + 1)]
    return [(edges[i], edges[i + 1]) for i in range(n)]


def e2e_plan(path: str, T: int, host_chunks: int, e2e_chunks: int, e2e_mode: str):
    """The end-to-end step's row ranges and transfer mode.  Where the
    chunked call splits x held in host memory itself (host_chunks > 1), the
    step is that one call reading x in place, unless ranges are asked for;
    otherwise the store path copies row ranges (from 2048 rows) and the
    other paths take one range.  One range always reads x in place."""
    if path == "store" and not (host_chunks > 1 and e2e_chunks == 0):
        chunks = row_chunks(T, e2e_chunks)
    else:
        chunks = [(0, T)]
    mode = ("copy" if e2e_mode == "auto" else e2e_mode) if len(chunks) > 1 else "inplace"
    return chunks, mode


class OverlappedChain:
    """rc_context_norms + rc_kv_project_store over row ranges of x held in
    pinned host memory, overlapping the host-to-device transfer of x with
    the chain.  Rows are independent, so every row's K and V reach the caches
    as the single pair of calls would store them; only the projection's plan
    follows the range's size, so its FP32 summation order (and with it the
    last bit of a K/V value) may differ.  Each range gets its own slice of one
    [L, T, D] norms buffer, and the ranges' projections share one workspace.

    mode "copy": the copy engines move range c + 1 of x into one of two
    device buffers (one cudaMemcpyAsync per range on a copy stream) while
    the current stream runs the norms and the projection + store of range c,
    so the transfer takes no SM time.  mode "inplace": the norms kernel of
    range c + 1 reads its rows of x in place over the host link while range
    c is projected and stored on a second stream."""

    def __init__(self, L: int, T: int, D: int, N: int, chunks, dev, mode: str = "copy"):
        import torch
        import rope_chain_gb300 as rc
        assert mode in ("copy", "inplace")
        self.rc, self.L, self.chunks, self.mode = rc, L, chunks, mode
        flat = torch.empty(L * T * D, dtype=torch.bfloat16, device=dev)
        self.normed = [flat[L * r0 * D:L * r1 * D].view(L, r1 - r0, D) for r0, r1 in chunks]
        ws = max(rc.workspace_size(L, r1 - r0, D, N) for r0, r1 in chunks)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev) if ws else None
        self.side = torch.cuda.Stream(device=dev)
        self.done = [torch.cuda.Event() for _ in chunks]
        if mode == "copy":
            rows = max(r1 - r0 for r0, r1 in chunks)
            self.xbuf = [torch.empty((rows, D), dtype=torch.bfloat16, device=dev) for _ in range(2)]
            self.copied = [torch.cuda.Event() for _ in chunks]

    def __call__(self, x, hidden_w, pre_w, W, H, positions, slots, cos_sin, caches, eps, err,
                 inputs_ready=None):
        """One pass on the current stream; inputs_ready (a stream) is waited
        for before the first projection (positions and slots copied there)."""
        import torch
        main = torch.cuda.current_stream()
        sl = lambda r0, r1: [None if s_ is None else s_[r0:r1] for s_ in slots]
        if self.mode == "copy":
            # copy stream: range c into buffer c % 2 once the norms of range
            # c - 2 (the buffer's last reader) are done.  Each copy is queued
            # just before its range's chain, so the event it waits for has
            # already been recorded in this pass (a wait on an event not yet
            # recorded would not wait).
            self.side.wait_stream(main)
            if inputs_ready is not None:
                main.wait_stream(inputs_ready)
            for c, ((r0, r1), nc) in enumerate(zip(self.chunks, self.normed)):
                with torch.cuda.stream(self.side):
                    if c >= 2:
                        self.side.wait_event(self.done[c - 2])
                    self.xbuf[c % 2][:r1 - r0].copy_(x[r0:r1], non_blocking=True)
                    self.copied[c].record(self.side)
                main.wait_event(self.copied[c])
                self.rc.context_norms(self.xbuf[c % 2][:r1 - r0], hidden_w, pre_w, self.L, eps, out=nc)
                self.done[c].record(main)
                self.rc.kv_project_store(nc, W, H, positions[r0:r1], sl(r0, r1), cos_sin, caches,
                                         eps, err=err, workspace=self.ws)
            main.wait_stream(self.side)
            return
        self.side.wait_stream(main)
        if inputs_ready is not None:
            self.side.wait_stream(inputs_ready)
        for (r0, r1), nc, ev in zip(self.chunks, self.normed, self.done):
            self.rc.context_norms(x[r0:r1], hidden_w, pre_w, self.L, eps, out=nc)
            ev.record(main)
            self.side.wait_event(ev)
            with torch.cuda.stream(self.side):
                self.rc.kv_project_store(nc, W, H, positions[r0:r1], sl(r0, r1), cos_sin, caches,
                                         eps, err=err, workspace=self.ws)
        main.wait_stream(self.side)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def algorithmic_counts(w, splits: int):
    """Per-step algorithmic bytes / flops of each kernel: the norms read x once
    and write L rows (plus the gains), the projection does 2 L T D N FLOP."""
    T, D, L, H, N = w.T, w.D, w.L, w.H, w.N
    k1 = 2 * T * D * (1 + L) + 2 * D * ((1 if w.hidden_weighted else 0) + (L if w.pre_weighted else 0))
    k2_flops = 2 * L * T * D * N
    k2_bytes = 2 * (L * T * D + L * D * N + L * T * N)
    return dict(k1_bytes=k1, k2_flops=k2_flops, k2_bytes=k2_bytes, splits=splits)


def store_bytes(w, slots, rope: bool) -> int:
    """K3: per (row, layer) 8 B of slot; a row whose slot is in range reads
    K and V (256 H B), writes 256 H B to the cache, and with RoPE reads its
    position (8 B) and 128 B of table."""
    total = 0
    cap = w.num_blocks * w.block_size
    for s in slots:
        live = int(((s >= 0) & (s < cap)).sum())
        total += 8 * len(s) + live * (512 * w.H + (8 + 128 if rope else 0))
    return total


def project_store_bytes(w, slots, rope: bool) -> int:
    """Algorithmic bytes of the fused projection + store call: the normed
    rows and W read once, and per (row, layer) the slot, plus for a row
    whose slot is in range its cache row written (256 H B) and with RoPE its
    position and table row; the projection itself never leaves the chip."""
    total = 2 * (w.L * w.T * w.D + w.L * w.D * w.N)
    cap = w.num_blocks * w.block_size
    for s in slots:
        live = int(((s >= 0) & (s < cap)).sum())
        total += 8 * len(s) + live * (256 * w.H + (8 + 128 if rope else 0))
    return total


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return summarise_clocks(lines)


def summarise_clocks(lines):
    """Median SM clock, the maximum clock and the throttle reasons seen in
    nvidia-smi's CSV lines (the fields of ClockSampler.FIELDS, no header,
    no units); None when no line parses."""
    rows = [[p.strip() for p in line.split(",")] for line in lines]
    rows = [r for r in rows if len(r) >= 9]
    if not rows:
        return None
    sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
    watts = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
    reasons = set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for r in rows:
        for n, v in zip(names, r[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
            "power_w": statistics.median(watts) if watts else None,
            "reasons": sorted(reasons), "samples": len(rows)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_chain_rows(case, w, R: int, threads: int = 0) -> float:
    """The oracle's whole chain on the first R rows of a workload; seconds."""
    import numpy as np
    import oracle
    x = np.ascontiguousarray(case["x"][:R])
    slots = [np.ascontiguousarray(s[:R]) for s in case["slots"]]
    caches = [np.zeros(case["cache_shape"], dtype=np.uint16) for _ in range(w.L)]
    t0 = time.perf_counter()
    normed = oracle.context_norms(x, case["hidden_w"], case["pre_w"], w.L, w.eps, threads=threads)
    kv64, _ = oracle.kv_project(normed, case["W"], with_abs=False, threads=threads)
    kv = oracle.bf16_rn_f64_array(kv64)
    oracle.kv_store_from_projection(kv, w.H, case["positions"][:R], slots, case["cos_sin"], caches,
                                    w.eps, R, threads=threads)
    return time.perf_counter() - t0


def host_cpu() -> str:
    """The host CPU's model name (lscpu), else the machine type."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return f"{line.split(':', 1)[1].strip()} ({platform.machine()})"
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


def make_case(args, w):
    """The workload's inputs; with --rows, the first rows of the full draw."""
    import workloads
    if getattr(args, "full_T", None):
        return workloads.make_inputs(workloads.WORKLOADS[args.workload], T=w.T)
    return workloads.make_inputs(w)


def cpu_sample_rows(w) -> int:
    return min(w.T, 256)


def base_record(args, w, world):
    return {"metric": METRIC, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, shapes of the workload)",
            "config": {"workload": f"workload {w.index}: {w.describe()} ({w.label})",
                       "T": w.T, "D": w.D, "L": w.L, "H": w.H, "N": w.N, "rope": w.rope,
                       "eps": w.eps, "num_blocks": w.num_blocks, "block_size": w.block_size,
                       "parallelism": f"replicas x{world} (rows independent, no collective)"}}


def run_reference(args, w):
    """The reference arm: the CPU oracle on the host cores (rank 0 only)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import workloads
    oracle.build()
    case = make_case(args, w)
    R = cpu_sample_rows(w)
    cores = oracle.max_threads()
    for _ in range(args.warmup):
        oracle_chain_rows(case, w, R)
    times = [oracle_chain_rows(case, w, R) for _ in range(args.steps)]
    total = sum(times)
    value = R * args.steps / total
    rec = base_record(args, w, world)
    rec.update({"impl": "reference", "value": value, "ms_per_step": 1e3 * total / args.steps,
                "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "cpu": host_cpu(), "kind": "oracle",
                                 "sample": f"first {R} rows of the workload per step, whole chain"},
                "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}})
    rec["dtype"] = "f32 (f64 projection)"
    print(json.dumps(rec))


def run_ours(args, w):
    import numpy as np
    import torch
    import rope_chain_gb300 as rc
    import workloads
    from rope_chain_gb300 import _build

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0 or not os.path.exists(rc.LIB_PATH):
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    rc.lib()

    case = make_case(args, w)
    bf = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    x, hw, pw, W, cs = bf(case["x"]), bf(case["hidden_w"]), bf(case["pre_w"]), bf(case["W"]), bf(case["cos_sin"])
    positions = torch.from_numpy(case["positions"]).to(dev)
    slots = [torch.from_numpy(s).to(dev) for s in case["slots"]]
    caches = [torch.zeros(case["cache_shape"], dtype=torch.bfloat16, device=dev) for _ in range(w.L)]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    normed = torch.empty((w.L, w.T, w.D), dtype=torch.bfloat16, device=dev)
    kv = torch.empty((w.L, w.T, w.N), dtype=torch.bfloat16, device=dev)
    ws_bytes = rc.workspace_size(w.L, w.T, w.D, w.N)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    cws = rc.context_kv_workspace(w.L, w.T, w.H, dev)   # the whole-chain call's workspace
    chunked = args.path in ("store", "variants") and args.chunks != 1
    if chunked:                                      # the chunked chain's normed rows and counters
        kws = rc.context_kv_chunked_workspace(w.L, w.T, w.H, dev, chunks=args.chunks)
    z = torch.empty((w.T, w.D), dtype=torch.bfloat16, device=dev)
    r2 = torch.empty((w.T,), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    use_ws = ws_bytes > 0
    # how the library runs this projection with that workspace
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    plan = rc.project_plan(w.L, w.T, w.D, w.N, sms, ws_bytes)
    pair = plan["kernel"] != "single CTAs"
    tail = plan["tail_splits"] > 0
    split = plan["splits"] > 1
    # norms (or row pass) + GEMM + (reduce-and-store when K is split; the
    # pair epilogue stores otherwise, plus the tail's split GEMM and
    # reduce-and-store; single CTAs without split: store kernel).  The
    # whole-chain call's forming projection takes every tile itself.
    launches_per_step = 2 + (1 if split else (0 if pair else (w.L + 7) // 8))
    if tail and args.path != "whole":
        launches_per_step += 2
    # the chunked chain: per row chunk the norms and one persistent
    # projection + store (a memset of the chunks' tile counters first)
    # (the variants' FP32 gains keep one chunk with x in device memory unless
    # more are asked for)
    n_chunks = (rc.context_kv_chunks(w.L, w.T, w.H, sms, args.chunks)
                if chunked and not (args.path == "variants" and args.chunks <= 0) else 1)
    if n_chunks > 1:
        launches_per_step = 2 * n_chunks

    whole = args.path == "whole"
    variants = args.path == "variants"
    if variants:
        # the norm options and per-layer slot lengths: FP32 gains, the hidden
        # gain scaling the input, a layer gain centre of 1, separate eps,
        # layer l storing T - l * T / (2 L) rows
        hw32 = None if hw is None else hw.float()
        pw32 = None if pw is None else pw.float()
        layer_rows = [w.T - l * (w.T // (2 * w.L)) for l in range(w.L)]

    def norms_variant(xs=None):
        rc.context_norms_ex(x if xs is None else xs, w.L, hidden_w=hw32, pre_w=pw32, hidden_eps=w.eps,
                            pre_eps=10.0 * w.eps, pre_center=1.0, hidden_input_scale=True,
                            out=normed)

    def chain(ev=None, xs=None, pos=None, sl=None, before_store=None):
        """One step through the public calls (ev[0] / ev[2] bracket it):
        "store" path: rc_context_norms, then rc_kv_project_store (projection
        with the store fused); "whole" path: rc_context_kv (the norms formed
        inside the projection as well).  xs, pos, sl replace the resident
        inputs and before_store runs just before the first call that reads
        pos and sl (the end-to-end steps)."""
        xs = x if xs is None else xs
        pos = positions if pos is None else pos
        sl = slots if sl is None else sl
        if ev:
            ev[0].record()
        ready = before_store or (lambda: None)
        if whole:
            ready()
            rc.context_kv(xs, hw, pw, W, w.H, pos, sl, cs, caches, w.eps, cws, err=err)
        elif variants and chunked:
            ready()
            rc.context_kv_chunked_ex(xs, W, w.H, pos, sl, cs, caches, w.eps, kws, hidden_w=hw32,
                                     pre_w=pw32, hidden_eps=w.eps, pre_eps=10.0 * w.eps,
                                     pre_center=1.0, hidden_input_scale=True, rows=layer_rows,
                                     err=err, chunks=args.chunks)
        elif variants:
            norms_variant(xs)
            ready()
            rc.kv_project_store(normed, W, w.H, pos, sl, cs, caches, w.eps, rows=layer_rows,
                                err=err, workspace=ws if use_ws else None)
        elif chunked:
            ready()
            rc.context_kv_chunked(xs, hw, pw, W, w.H, pos, sl, cs, caches, w.eps, kws, err=err,
                                  chunks=args.chunks)
        else:
            rc.context_norms(xs, hw, pw, w.L, w.eps, out=normed)
            ready()
            rc.kv_project_store(normed, W, w.H, pos, sl, cs, caches, w.eps, err=err,
                                workspace=ws if use_ws else None)
        if ev:
            ev[2].record()

    def chain_split(ev):
        """The work of chain() over all rows in one chunk, an event between
        its two calls (breakdown; the projection + store call is the one the
        roofline times)."""
        ev[0].record()
        if whole and pair:
            rc.context_rows(x, hw, w.eps, z=z, r2=r2)
            ev[1].record()
            rc.context_kv_from_rows(z, r2, pw, W, w.H, positions, slots, cs, caches, w.eps, err=err,
                                    workspace=ws if use_ws else None)
        elif variants:
            norms_variant()
            ev[1].record()
            rc.kv_project_store(normed, W, w.H, positions, slots, cs, caches, w.eps, rows=layer_rows,
                                err=err, workspace=ws if use_ws else None)
        else:
            rc.context_norms(x, hw, pw, w.L, w.eps, out=normed)
            ev[1].record()
            rc.kv_project_store(normed, W, w.H, positions, slots, cs, caches, w.eps, err=err,
                                workspace=ws if use_ws else None)
        ev[2].record()

    def chain_unfused(ev):
        """The three calls of the boundary, an event after each (breakdown)."""
        ev[0].record()
        rc.context_norms(x, hw, pw, w.L, w.eps, out=normed)
        ev[1].record()
        rc.kv_project(normed, W, out=kv, workspace=ws if use_ws else None)
        ev[2].record()
        rc.kv_store_from_projection(kv, w.H, positions, slots, cs, caches, w.eps, err=err)
        ev[3].record()

    for i in range(args.warmup):
        flush(i)
        chain()
        chain_split([torch.cuda.Event(enable_timing=True) for _ in range(3)])
        chain_unfused([torch.cuda.Event(enable_timing=True) for _ in range(4)])
    torch.cuda.synchronize()
    # The K timed steps run as one captured CUDA graph (what a serving loop
    # does with these graph-capturable calls), each step preceded by the L2
    # flush; without event nodes in graphs (older torch) they launch eagerly.
    timing = "cuda graph"
    try:
        make_event = lambda: torch.cuda.Event(enable_timing=True, external=True)
        make_event()
    except TypeError:
        make_event = lambda: torch.cuda.Event(enable_timing=True)
        timing = "eager"
    evs = [[make_event() for _ in range(3)] for _ in range(args.steps)]
    kevs = [[make_event() for _ in range(3)] for _ in range(args.steps)]
    uevs = [[make_event() for _ in range(4)] for _ in range(args.steps)]

    def steps(kind):
        for i in range(args.steps):
            flush(i)            # L2 flushed before every step (not timed)
            if kind == "timed":
                chain(evs[i])
            elif kind == "kernels":
                chain_split(kevs[i])
            else:
                chain_unfused(uevs[i])

    graphs = {}
    if timing == "cuda graph":
        for kind in ("timed", "kernels", "unfused"):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                steps(kind)
            g.replay()                       # warm the graph itself
            graphs[kind] = g
        torch.cuda.synchronize()
    run = lambda kind: graphs[kind].replay() if graphs else steps(kind)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    run("timed")                             # the timed K steps
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    # breakdowns (roofline figures), replayed after the timed region
    run("kernels")
    run("unfused")
    torch.cuda.synchronize()
    step_ms = [e[0].elapsed_time(e[2]) for e in evs]
    total_ms = max_over_ranks(sum(step_ms), world)
    k1_ms = [e[0].elapsed_time(e[1]) for e in kevs]
    ps_ms = [e[1].elapsed_time(e[2]) for e in kevs]
    u_ms = [[e[j].elapsed_time(e[j + 1]) for e in uevs] for j in range(3)]
    faults = rc.read_device_faults(clear=True)
    if faults:
        raise RuntimeError(f"projection kernel raised fault bits {faults:#x}")
    # ---- end to end: inputs from pinned host memory, the status word read
    # back.  The norms kernel reads x in place over the host link (NVLink-C2C;
    # no staging copy, so the transfer overlaps the norms); positions and
    # every layer's slot map travel in one pinned buffer, one copy per step,
    # on a side stream alongside the norms.
    x_h = torch.from_numpy(case["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    assert all(len(s_) == w.T for s_ in case["slots"])
    meta_h = torch.from_numpy(np.stack([case["positions"], *case["slots"]])).pin_memory()
    meta_d = torch.empty(tuple(meta_h.shape), dtype=torch.int64, device=dev)
    pos_e, slots_e = meta_d[0], [meta_d[1 + l] for l in range(w.L)]
    err_h = torch.zeros(1, dtype=torch.int32).pin_memory()
    h2d = x_h.numel() * 2 + meta_h.numel() * 8

    side = torch.cuda.Stream(device=dev)
    # On the default path the rows go through in ranges (OverlappedChain):
    # the transfer of x for range c + 1 overlaps the chain of range c, by the
    # copy engines into device buffers ("copy") or by the norms kernel
    # reading host memory in place ("inplace").  One range: the norms read x
    # in place (the read overlaps the norms' own work).
    # With the chunked call, x in host memory is chunked by the call itself
    # (a plan of its own for x read over the host link): one call whose
    # chunks' norms read their rows of x in place beside the previous
    # chunk's projection, unless the ranges are asked for.
    host_chunks = (rc.context_kv_chunks(w.L, w.T, w.H, sms, args.chunks, x_on_host=True)
                   if chunked else 1)
    chunks, e2e_mode = e2e_plan(args.path, w.T, host_chunks, args.e2e_chunks, args.e2e_mode)
    overlapped = OverlappedChain(w.L, w.T, w.D, w.N, chunks, dev, e2e_mode) if len(chunks) > 1 else None

    def e2e_step(ev0, ev1):
        # the metadata copy runs on a side stream while the norms read x;
        # the projection + store waits for it
        ev0.record()
        main = torch.cuda.current_stream()
        side.wait_stream(main)
        with torch.cuda.stream(side):
            meta_d.copy_(meta_h, non_blocking=True)
        if overlapped is not None:
            overlapped(x_h, hw, pw, W, w.H, pos_e, slots_e, cs, caches, w.eps, err,
                       inputs_ready=side)
        else:
            chain(xs=x_h, pos=pos_e, sl=slots_e, before_store=lambda: main.wait_stream(side))
        err_h.copy_(err, non_blocking=True)
        ev1.record()

    for i in range(args.warmup):
        flush(i)
        e2e_step(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    torch.cuda.synchronize()
    # The end-to-end steps (copies from pinned host memory, the calls, the
    # status word back) run as one captured graph too when event nodes are
    # available, as a serving loop would issue them; eagerly otherwise.
    e2e_evs = [(make_event(), make_event()) for _ in range(args.steps)]

    def e2e_steps():
        for i in range(args.steps):
            flush(i)
            e2e_step(*e2e_evs[i])

    e2e_graph = None
    if graphs:
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph):
            e2e_steps()
        e2e_graph.replay()                   # warm the graph itself
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    if e2e_graph is not None:
        e2e_graph.replay()
    else:
        e2e_steps()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_evs), world)

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    counts = algorithmic_counts(w, 2 if ws_bytes else 1)
    k3_bytes = store_bytes(w, case["slots"], w.rope)
    hbm, tc = peaks["hbm_gbs"], peaks["bf16_tflops"]
    us = lambda ms: 1e3 * statistics.mean(ms)

    def hbm_entry(nbytes, t_us):
        return {"us": t_us, "GB/s": nbytes / t_us / 1e3, "frac": nbytes / t_us / 1e3 / hbm,
                "bound": "hbm"}

    def tc_entry(t_us):
        return {"us": t_us, "TFLOP/s": counts["k2_flops"] / t_us / 1e6,
                "frac": counts["k2_flops"] / t_us / 1e6 / tc, "bound": "tensor"}

    rows_bytes = 2 * w.T * w.D * 2 + 2 * w.D + 4 * w.T   # read x, write z, gains, r2
    fused_norms = whole and pair
    if variants:                              # FP32 gains: 4 bytes per weight
        counts["k1_bytes"] += 2 * w.D * ((1 if w.hidden_weighted else 0) + (w.L if w.pre_weighted else 0))
    kern = {
        "row_pass" if fused_norms else "norms": hbm_entry(rows_bytes if fused_norms else counts["k1_bytes"],
                                                          us(k1_ms)),
        "project_store": dict(tc_entry(us(ps_ms)), workspace_bytes=ws_bytes,
                              plan=plan, tail_split=bool(tail and not fused_norms),
                              norms_fused=fused_norms),
        "unfused": {"norms": hbm_entry(counts["k1_bytes"], us(u_ms[0])),
                    "project": tc_entry(us(u_ms[1])),
                    "store": hbm_entry(k3_bytes, us(u_ms[2]))},
    }
    if n_chunks > 1:
        kern["note"] = ("norms and project_store: the step's two kernels over all rows, one "
                        "after the other between events (the chunked step overlaps them)")
    first = "row_pass" if fused_norms else "norms"
    dominant = "project_store" if kern["project_store"]["us"] >= kern[first]["us"] else first
    d = kern[dominant]
    # the stored figures are full-size captures: none for a --rows prefix
    traffic_of = ((lambda key: (None, f"a --rows case (the first {w.T} rows): no capture of "
                                      "this size")) if getattr(args, "full_T", None) else ncu_traffic)
    traffic, traffic_note = traffic_of((args.workload, args.path, dominant))
    for name, entry in (("norms", kern["unfused"]["norms"]), ("store", kern["unfused"]["store"])):
        entry["traffic"], entry["traffic_note"] = traffic_of((args.workload, "unfused", name))
    if d["bound"] == "tensor":
        roof = {"kernel": dominant, "bound": "tensor", "achieved": d["TFLOP/s"], "peak": tc,
                "unit": "TFLOP/s", "frac": d["frac"], "traffic": traffic,
                "traffic_note": traffic_note,
                "algorithmic_bytes": project_store_bytes(w, case["slots"], w.rope),
                "peak_source": f"bf16_tflops (burst) of {peak_src}",
                "frac_of_sustained": d["TFLOP/s"] / peaks.get("bf16_tflops_sustained", tc),
                # the same FLOPs over the whole timed step (norms, and in the
                # chunked step their overlap with the projection, included)
                "step_tflops": counts["k2_flops"] / (total_ms / args.steps) / 1e9,
                "step_frac": counts["k2_flops"] / (total_ms / args.steps) / 1e9 / tc}
    else:
        roof = {"kernel": dominant, "bound": "hbm", "achieved": d["GB/s"], "peak": hbm,
                "unit": "GB/s", "frac": d["frac"], "traffic": traffic,
                "traffic_note": traffic_note, "peak_source": f"hbm_gbs of {peak_src}"}
    import oracle
    oracle.build()
    R = cpu_sample_rows(w)
    cpu_s = oracle_chain_rows(case, w, R)
    R1 = min(w.T, 32)
    cpu1_s = oracle_chain_rows(case, w, R1, threads=1)
    rec = base_record(args, w, world)
    rec["config"]["l2"] = ("flushed before every timed step: a 512 MiB write, then a 256 MiB "
                           "read, so each step starts with a cold L2 of clean lines")
    rec["config"]["timing"] = timing
    rec["config"]["path"] = ("rc_context_kv (row pass; projection forming the normed rows in shared "
                             "memory, store fused)" if whole else
                             (f"rc_context_kv_chunked_ex ({n_chunks} row chunks; " if n_chunks > 1 else
                              "rc_context_kv_chunked_ex (one chunk; " if chunked else
                              "rc_context_norms_ex + rc_kv_project_store_rows (") +
                             "FP32 gains, hidden gain on the input, layer gain centre 1, separate "
                             "eps, per-layer slot lengths)" if variants else
                             f"rc_context_kv_chunked ({n_chunks} row chunks: the norms of chunk "
                             "c + 1 run beside the projection + store of chunk c)" if n_chunks > 1 else
                             "rc_context_kv_chunked (one chunk: rc_context_norms, then "
                             "rc_kv_project_store with the store fused)" if chunked else
                             "rc_context_norms + rc_kv_project_store (projection with the store fused)")
    rec["config"]["row_chunks"] = n_chunks
    rec.update({
        "value": world * w.T * args.steps / (total_ms / 1e3),
        "ms_per_step": total_ms / args.steps,
        "roofline": roof,
        "kernels": kern,
        "cpu_baseline": {"value": R / cpu_s, "unit": "rows/s", "cores": oracle.max_threads(), "cpu": host_cpu(),
                         "kind": "oracle", "sample": f"first {R} rows of the workload, whole chain, once",
                         "one_core": {"value": R1 / cpu1_s, "unit": "rows/s", "cores": 1,
                                      "sample": f"first {R1} rows, whole chain, once"}},
        "e2e": {"value": world * w.T * args.steps / (e2e_ms / 1e3), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4, "timing": timing,
                "inputs": ("x copied from pinned host memory by the copy engines, one "
                           "cudaMemcpyAsync per row range into two device buffers"
                           if e2e_mode == "copy" else
                           "x read in place from pinned host memory by the norms kernel "
                           "(NVLink-C2C)") +
                          "; positions and slot maps in one pinned buffer, one copy per step" +
                          ("" if whole or chunked else " alongside the norms"),
                "outputs": "the K/V result stays in the device caches (the operation's "
                           "output); only the 4-byte skip count is copied back per step",
                "row_ranges": len(chunks),
                "row_chunks": host_chunks if overlapped is None else 1,
                "overlap": (f"{host_chunks} row chunks in one call: the norms of chunk c + 1 read "
                            "their rows of x over the host link while chunk c is projected and "
                            "stored" if overlapped is None and host_chunks > 1 else
                            "none" if overlapped is None else
                            f"{len(chunks)} row ranges: the copy of range c + 1 runs while "
                            "range c goes through the chain" if e2e_mode == "copy" else
                            f"{len(chunks)} row ranges: the norms of range c + 1 read x "
                            "while range c is projected and stored on a second stream")},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    })
    print(json.dumps(rec))


FRONT_METRIC = "decode QKV front tokens/s (one draft layer, W streamed from HBM); W GB/s vs GB300 peak"


def front_bytes(M: int, D: int, N: int, nkv: int, live: int) -> int:
    """Algorithmic bytes of one decode front call: W once, the hidden rows,
    the output rows, positions and slots, a table row per token, and K and V
    of every live token into the cache."""
    return 2 * N * D + 2 * M * D + 2 * M * N + 16 * M + 128 * M + live * 256 * nkv


def oracle_front_seconds(case, M: int) -> float:
    import numpy as np
    import oracle
    cache = np.zeros(case["cache_shape"], dtype=np.uint16)
    t0 = time.perf_counter()
    ref64, _ = oracle.qkv_project(case["hidden"], case["W"])
    raw = oracle.bf16_rn_f64_array(ref64)
    oracle.qkv_front_post(raw, case["num_heads"], case["num_kv_heads"], case["positions"],
                          case["cos_sin"], case["slots"], cache, case["eps"])
    return time.perf_counter() - t0


def front_record(args, case, world, M):
    N, D = case["W"].shape
    return {"metric": FRONT_METRIC, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded)",
            "config": {"workload": f"decode QKV front: M={M} tokens, D={D}, {case['num_heads']} query "
                                   f"heads, {case['num_kv_heads']} KV heads, W [{N}, {D}], RoPE, "
                                   "paged insert",
                       "M": M, "D": D, "Nqkv": N, "num_heads": case["num_heads"],
                       "num_kv_heads": case["num_kv_heads"],
                       "parallelism": f"replicas x{world} (no collective)"}}


def run_front(args):
    """--path front: the decode QKV front (rc_qkv_front) on M tokens."""
    import numpy as np
    import workloads
    rank, world, local = dist_env()
    M = args.tokens
    case = workloads.front_case(3000 + M, M)
    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build()
        for _ in range(args.warmup):
            oracle_front_seconds(case, M)
        total = sum(oracle_front_seconds(case, M) for _ in range(args.steps))
        value = M * args.steps / total
        rec = front_record(args, case, world, M)
        rec.update({"impl": "reference", "value": value, "ms_per_step": 1e3 * total / args.steps,
                    "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.max_threads(), "cpu": host_cpu(),
                                     "kind": "oracle", "sample": f"all {M} tokens per step"},
                    "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}})
        rec["dtype"] = "f32 (f64 projection)"
        print(json.dumps(rec))
        return
    import torch
    import rope_chain_gb300 as rc
    from rope_chain_gb300 import _build
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0 or not os.path.exists(rc.LIB_PATH):
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    rc.lib()
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    hidden, W, cs = bf(case["hidden"]), bf(case["W"]), bf(case["cos_sin"])
    N, D = case["W"].shape
    positions = torch.from_numpy(case["positions"]).to(dev)
    slots = torch.from_numpy(case["slots"]).to(dev)
    cache = torch.zeros(case["cache_shape"], dtype=torch.bfloat16, device=dev)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    nh, nkv, eps = case["num_heads"], case["num_kv_heads"], case["eps"]
    # Consecutive steps use two draft layers' weights in turn, as a decode
    # step's layers do: each W (151 MB) exceeds L2 and the other was read
    # since, so every step reads its W from HBM, and no flush is needed.
    Ws = [W, bf(workloads.front_case(4000 + M, M)["W"])]
    call = lambda i: rc.qkv_front(hidden, Ws[i % 2], nh, nkv, positions, cs, slots, cache, eps,
                                  out=out, err=err)
    for i in range(max(args.warmup, 2)):
        call(i)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True, external=True),
            torch.cuda.Event(enable_timing=True, external=True)) for _ in range(args.steps)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(args.steps):
            evs[i][0].record()
            call(i)
            evs[i][1].record()
    g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    step_us = [a.elapsed_time(b) * 1e3 for a, b in evs]
    total_ms = max_over_ranks(sum(step_us) / 1e3, world)
    if rc.read_device_faults(clear=True):
        raise RuntimeError("QKV front raised fault bits")
    # end to end: hidden rows in from pinned memory, the output rows back
    h_h = torch.from_numpy(case["hidden"].view(np.int16)).view(torch.bfloat16).pin_memory()
    o_h = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    def e2e_step(i, ev=None):
        if ev:
            ev[0].record()
        hidden.copy_(h_h, non_blocking=True)
        call(i)
        o_h.copy_(out, non_blocking=True)
        if ev:
            ev[1].record()

    for i in range(max(args.warmup, 2)):
        e2e_step(i)
    torch.cuda.synchronize()
    # as one captured graph, like the timed device steps
    e2e_evs = [(torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True)) for _ in range(args.steps)]
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge):
        for i in range(args.steps):
            e2e_step(i, e2e_evs[i])
    ge.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ge.replay()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_evs), world)
    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    nbytes = front_bytes(M, D, N, nkv, int((case["slots"] >= 0).sum()))
    t_us = statistics.mean(step_us)
    import oracle
    oracle.build()
    cpu_s = oracle_front_seconds(case, M)
    rec = front_record(args, case, world, M)
    rec["config"]["l2"] = ("no flush: inputs larger than L2 (steps alternate two layers' weights, "
                           "2 x 151 MB against 129 MB of L2, so each step reads its W from HBM)")
    rec["config"]["timing"] = "cuda graph"
    rec.update({
        "value": world * M * args.steps / (total_ms / 1e3),
        "ms_per_step": total_ms / args.steps,
        "roofline": {"kernel": "k4_qkv_front", "bound": "hbm", "achieved": nbytes / t_us / 1e3,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": nbytes / t_us / 1e3 / peaks["hbm_gbs"],
                     "traffic": ncu_traffic(("front", M, "k4_qkv_front"))[0],
                     "peak_source": f"hbm_gbs of {peak_src}"},
        "kernels": {"qkv_front": {"us": t_us, "GB/s": nbytes / t_us / 1e3, "bytes": nbytes}},
        "cpu_baseline": {"value": M / cpu_s, "unit": "tokens/s", "cores": oracle.max_threads(), "cpu": host_cpu(),
                         "kind": "oracle", "sample": f"all {M} tokens, once"},
        "e2e": {"value": world * M * args.steps / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": M * D * 2, "d2h_bytes_per_step": M * N * 2,
                "timing": "cuda graph"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    })
    print(json.dumps(rec))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--e2e-chunks", type=int, default=0, metavar="N",
                    help="row ranges of the end-to-end steps on the default path "
                         "(0: 8 from 16384 rows, 4 from 2048, else 1)")
    ap.add_argument("--e2e-mode", default="auto", choices=["auto", "copy", "inplace"],
                    help="how x reaches the GPU in the end-to-end row ranges: copy engines "
                         "(copy; the default) or the norms reading host memory (inplace)")
    ap.add_argument("--rows", type=int, default=0, metavar="R",
                    help="run only the first R rows of the workload (a smaller case of its "
                         "shape, for profiler captures; 0: all rows)")
    ap.add_argument("--chunks", type=int, default=0, metavar="N",
                    help="row chunks of the store path's step (rc_context_kv_chunked: each "
                         "chunk's norms beside the previous chunk's projection); 0: the "
                         "library's choice; 1: the two calls rc_context_norms and "
                         "rc_kv_project_store")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default="store", choices=["store", "whole", "variants", "front"],
                    help="store: norms + fused projection/store; whole: rc_context_kv; variants: "
                         "the norm options and per-layer slot lengths; front: the decode QKV "
                         "front (rc_qkv_front)")
    ap.add_argument("--tokens", type=int, default=16, choices=range(1, 17), metavar="1..16",
                    help="tokens of the decode QKV front (--path front)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.path == "front":
        run_front(args)
        return
    import dataclasses
    import workloads
    w = workloads.WORKLOADS[args.workload]
    if 0 < args.rows < w.T:
        # the first R rows of the same draw (workloads.make_inputs(w, T=R))
        w = dataclasses.replace(w, T=args.rows, label=f"{w.label}; first {args.rows} rows")
        args.full_T = workloads.WORKLOADS[args.workload].T
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
