"""Parity helpers: run the CUDA chain and the oracle chain on the same seeded
inputs and compare them.

Rules (written once here, used by every GPU test and by smoke()):
  * norms (a1, a2): bit-exact over every element;
  * store (a5-a7): bit-exact over the whole cache, the oracle fed the GPU's
    own projection output, sentinel-filled caches so untouched entries count;
  * projection (a3): |gpu - ref64| <= 2 ulp_bf16(max(|ref64|, 2^-12 sum|a*w|)),
    ref64 the oracle's float64 sum.  The floor covers outputs near
    cancellation, where the FP32 accumulation error exceeds 2 ulp of the
    (small) result; a dropped 64-wide K block moves an output by far more.
"""
from __future__ import annotations

import json
import os
from typing import Optional

import numpy as np
import torch

import oracle
import rope_chain_gb300 as rc

SENTINEL = 0x5A5A


def dev_bf16(a: Optional[np.ndarray], dev) -> Optional[torch.Tensor]:
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (x > 0), subnormal spacing 2^-133 below."""
    _, e = np.frexp(np.abs(x))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def assert_projection_close(gpu_bits: np.ndarray, ref64: np.ndarray, abs64: np.ndarray,
                            what: str = "projection") -> float:
    g = (gpu_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    scale = np.maximum(np.abs(ref64), 2.0 ** -12 * abs64)
    tol = 2.0 * ulp_bf16(np.where(scale > 0, scale, 2.0 ** -133))
    err = np.abs(g - ref64)
    bad = err > tol
    if np.any(bad):
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside 2 ulp; first at {tuple(i)}: "
            f"gpu={g[tuple(i)]!r} ref={ref64[tuple(i)]!r} tol={tol[tuple(i)]!r}")
    return float(np.max(err / tol)) if err.size else 0.0


# Bins of an error measured in bf16 ulps at the comparison's scale: exact,
# within rounding (<= 1/2), one rounding step (<= 1), up to the rule's bound
# (<= 2), and beyond it (a failure).
ULP_BINS = ((0.0, "0"), (0.5, "(0,0.5]"), (1.0, "(0.5,1]"), (1.5, "(1,1.5]"), (2.0, "(1.5,2]"),
            (np.inf, ">2"))


def ulp_stats(err: np.ndarray, scale: np.ndarray) -> dict:
    """Max error and a histogram of |error| in units of ulp_bf16(scale)."""
    u = err / ulp_bf16(np.where(scale > 0, scale, 2.0 ** -133))
    u = u.reshape(-1)
    hist, lo = {}, -1.0
    for hi, name in ULP_BINS:
        hist[name] = int(np.count_nonzero((u > lo) & (u <= hi))) if hi > 0 else int(np.count_nonzero(u == 0))
        lo = hi
    return {"n": int(u.size), "max_ulp": float(u.max()) if u.size else 0.0,
            "over_1_ulp": int(np.count_nonzero(u > 1.0)), "hist": hist}


def projection_ulp_stats(gpu_bits: np.ndarray, ref64: np.ndarray, abs64: np.ndarray) -> dict:
    """The projection's error in ulps at the 2-ulp rule's scale
    max(|ref|, 2^-12 sum|a*w|), and separately in ulps of |ref| itself over
    the outputs away from cancellation (|ref| >= 2^-12 sum|a*w|)."""
    g = (gpu_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    err = np.abs(g - ref64)
    floor = 2.0 ** -12 * abs64
    st = ulp_stats(err, np.maximum(np.abs(ref64), floor))
    away = np.abs(ref64) >= floor
    st["relative_away_from_cancellation"] = ulp_stats(err[away], np.abs(ref64[away]))
    return st


def report(name: str, stats: dict) -> None:
    """Appends one JSON line {name, stats} to the file named by the
    RC_PARITY_REPORT environment variable (nothing when it is unset)."""
    path = os.environ.get("RC_PARITY_REPORT")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"name": name, **stats}) + "\n")


def make_caches(case, L: int, fill: int) -> list:
    return [np.full(case["cache_shape"], fill, dtype=np.uint16) for _ in range(L)]


def run_gpu_chain(case: dict, dev, *, w_layout: int = rc.RC_W_KN, use_workspace: bool = True,
                  cache_fill: int = SENTINEL, L: Optional[int] = None) -> dict:
    """The CUDA chain through the C ABI; returns host copies of normed, kv,
    the caches and the error count."""
    L = len(case["slots"]) if L is None else L
    H = case["cache_shape"][1]
    x = dev_bf16(case["x"], dev)
    hw = dev_bf16(case["hidden_w"], dev)
    pw = dev_bf16(case["pre_w"], dev)
    W = case["W"]
    if w_layout == rc.RC_W_NK:
        W = np.ascontiguousarray(W.transpose(0, 2, 1))
    Wd = dev_bf16(W, dev)
    T = case["x"].shape[0]
    N = 128 * H
    positions = torch.from_numpy(case["positions"]).to(dev)
    slots = [None if s is None else torch.from_numpy(s).to(dev) for s in case["slots"]]
    cs = dev_bf16(case["cos_sin"], dev)
    caches = [dev_bf16(c, dev) for c in make_caches(case, L, cache_fill)]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = None
    if use_workspace:
        nbytes = rc.workspace_size(L, T, 8192, N)
        if nbytes:
            ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    normed = rc.context_norms(x, hw, pw, L, case["eps"])
    kv = rc.kv_project(normed, Wd, w_layout=w_layout, workspace=ws)
    rc.kv_store_from_projection(kv, H, positions, slots, cs, caches, case["eps"], err=err)
    torch.cuda.synchronize(dev)
    return dict(normed=host_bits(normed), kv=host_bits(kv), caches=[host_bits(c) for c in caches],
                err=int(err.item()))


def run_oracle_chain(case: dict, kv_gpu: np.ndarray, *, rows: Optional[np.ndarray] = None,
                     cache_fill: int = SENTINEL, normed: Optional[np.ndarray] = None,
                     threads: int = 0) -> dict:
    """The oracle chain: norms of every row, the float64 projection of
    ``rows`` (all rows when None), and the store fed the GPU's ``kv_gpu``."""
    L = len(case["slots"])
    H = case["cache_shape"][1]
    if normed is None:
        normed = oracle.context_norms(case["x"], case["hidden_w"], case["pre_w"], L, case["eps"],
                                      threads=threads)
    kv64, kvabs = oracle.kv_project(normed, case["W"], rows=rows, threads=threads)
    caches = make_caches(case, L, cache_fill)
    err = oracle.kv_store_from_projection(kv_gpu, H, case["positions"], case["slots"],
                                          case["cos_sin"], caches, case["eps"],
                                          kv_gpu.shape[1], threads=threads)
    return dict(normed=normed, kv64=kv64, kvabs=kvabs, caches=caches, err=err)
