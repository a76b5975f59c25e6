"""CPU oracle of the draft's context K/V chain: a ctypes binding of
``rope_chain_oracle.c`` over numpy arrays.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` may import this package.  The product path
(``rope_chain_gb300``) never does; the two share no code.

bf16 tensors are numpy ``uint16`` bit patterns throughout.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rope_chain_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

# -ffp-contract=off: no a*b+c is fused behind the source's back; no
# -ffast-math: IEEE semantics (sqrt, divide, subnormals) are kept.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-fopenmp", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile the oracle (gcc) next to its source; returns the .so path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_c = ctypes


class _Norm(ctypes.Structure):
    """rco_norm: one norm's weight (bf16 or FP32 bits), scale side, gain
    center and eps."""
    _fields_ = [("weight", ctypes.c_void_p), ("fp32", ctypes.c_int32),
                ("input_scale", ctypes.c_int32), ("center", ctypes.c_float),
                ("eps", ctypes.c_float)]


def lib():
    global _lib
    if _lib is None:
        # RCO_ORACLE_LIB: tests of the pins load a copy of the oracle with
        # one mistake planted (tests/test_oracle_mutants.py) through it
        override = os.environ.get("RCO_ORACLE_LIB")
        L = ctypes.CDLL(override if override else build())
        sig = {
            "rco_f32": ([_c.c_uint16], _c.c_float),
            "rco_bf16_rn": ([_c.c_float], _c.c_uint16),
            "rco_bf16_rn_f64": ([_c.c_double], _c.c_uint16),
            "rco_bf16_rn_array": ([_f32p, _u16p, _c.c_int64], None),
            "rco_bf16_rn_f64_array": ([_f64p, _u16p, _c.c_int64], None),
            "rco_row_sumsq": ([_f32p], _c.c_float),
            "rco_head_sumsq": ([_f32p], _c.c_float),
            "rco_inv_rms": ([_c.c_float] * 3, _c.c_float),
            "rco_rope": ([_c.c_float] * 4 + [_f32p, _f32p], None),
            "rco_max_threads": ([], _c.c_int32),
            "rco_context_norms": ([_u16p, _c.c_int64, _c.c_int32, _u16p, _u16p,
                                   _c.c_int32, _c.c_float, _u16p, _c.c_int32],
                                  _c.c_int32),
            "rco_context_norms_ex": ([_u16p, _c.c_int64, _c.c_int32, _c.POINTER(_Norm),
                                      _c.POINTER(_Norm), _c.c_int32, _u16p, _c.c_int32],
                                     _c.c_int32),
            "rco_qkv_front_post": ([_u16p, _c.c_int32, _c.c_int32, _c.c_int32, _i64p, _u16p,
                                    _c.c_int64, _i64p, _u16p, _c.c_int32, _c.c_int32, _c.c_float,
                                    _u16p, _i32p], _c.c_int32),
            "rco_kv_project": ([_u16p, _u16p, _c.c_int32, _c.c_int32, _c.c_int64,
                                _c.c_int32, _c.c_int32, _i64p, _c.c_int64, _f64p,
                                _f64p, _c.c_int32], _c.c_int32),
            "rco_kv_store": ([_u16p, _u16p, _c.c_int64, _c.c_int64, _c.c_int64,
                              _c.c_int64, _i64p, _c.POINTER(_i64p), _u16p,
                              _c.c_int64, _c.POINTER(_u16p), _c.c_int32,
                              _c.c_int32, _c.c_int32, _c.c_int32, _c.c_float,
                              _c.c_int64, _i32p, _c.c_int32], _c.c_int32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _p(a: Optional[np.ndarray], t):
    if a is None:
        return ctypes.cast(None, t)
    assert a.flags["C_CONTIGUOUS"], "oracle operands must be contiguous"
    return a.ctypes.data_as(t)


def max_threads() -> int:
    return int(lib().rco_max_threads())


# ----------------------------------------------------------------- scalars

def f32(b: int) -> float:
    return float(lib().rco_f32(int(b)))


def bf16_rn(f: float) -> int:
    return int(lib().rco_bf16_rn(float(np.float32(f))))


def bf16_rn_f64(d: float) -> int:
    return int(lib().rco_bf16_rn_f64(float(d)))


def bf16_rn_array(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    lib().rco_bf16_rn_array(_p(a, _f32p), _p(out, _u16p), a.size)
    return out


def bf16_rn_f64_array(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    lib().rco_bf16_rn_f64_array(_p(a, _f64p), _p(out, _u16p), a.size)
    return out


def row_sumsq(v: np.ndarray) -> np.float32:
    v = np.ascontiguousarray(v, dtype=np.float32)
    assert v.shape == (8192,)
    return np.float32(lib().rco_row_sumsq(_p(v, _f32p)))


def head_sumsq(k: np.ndarray) -> np.float32:
    k = np.ascontiguousarray(k, dtype=np.float32)
    assert k.shape == (64,)
    return np.float32(lib().rco_head_sumsq(_p(k, _f32p)))


def inv_rms(sumsq: float, inv_width: float, eps: float) -> np.float32:
    return np.float32(lib().rco_inv_rms(sumsq, inv_width, eps))


def rope(x: float, y: float, c: float, s: float):
    xo, yo = ctypes.c_float(), ctypes.c_float()
    lib().rco_rope(x, y, c, s, ctypes.byref(xo), ctypes.byref(yo))
    return np.float32(xo.value), np.float32(yo.value)


# ------------------------------------------------------------------ chain

def context_norms(x: np.ndarray, hidden_w: Optional[np.ndarray],
                  pre_w: Optional[np.ndarray], L: int, eps: float,
                  threads: int = 0) -> np.ndarray:
    """bf16 [L, T, 8192] = stack_l(pre_norm_l(bf16(hidden_norm(x))))."""
    T, D = x.shape
    out = np.empty((L, T, D), dtype=np.uint16)
    rc = lib().rco_context_norms(_p(x, _u16p), T, D, _p(hidden_w, _u16p),
                                 _p(pre_w, _u16p), L, eps, _p(out, _u16p), threads)
    if rc != 0:
        raise ValueError("oracle: unsupported context_norms arguments")
    return out


def _norm(weight: Optional[np.ndarray], input_scale: bool, center: float, eps: float,
          shape) -> _Norm:
    if weight is None:
        return _Norm(None, 0, 0, 0.0, eps)
    assert weight.shape == shape and weight.flags["C_CONTIGUOUS"]
    if weight.dtype == np.float32:
        fp32 = 1
    elif weight.dtype == np.uint16:
        fp32 = 0
    else:
        raise TypeError("norm weights are bf16 bits (uint16) or float32")
    return _Norm(weight.ctypes.data, fp32, int(bool(input_scale)), center, eps)


def context_norms_ex(x: np.ndarray, L: int, *, hidden_w: Optional[np.ndarray] = None,
                     pre_w: Optional[np.ndarray] = None, hidden_eps: float,
                     pre_eps: float, hidden_center: float = 0.0, pre_center: float = 0.0,
                     hidden_input_scale: bool = False, pre_input_scale: bool = False,
                     threads: int = 0) -> np.ndarray:
    """``context_norms`` with every option of the norms kernel: weights as
    bf16 bits (uint16) or float32, each norm's eps and gain center, and
    whether each weight scales the norm's input (else its output)."""
    T, D = x.shape
    out = np.empty((L, T, D), dtype=np.uint16)
    h = _norm(hidden_w, hidden_input_scale, hidden_center, hidden_eps, (D,))
    p = _norm(pre_w, pre_input_scale, pre_center, pre_eps, (L, D))
    rc = lib().rco_context_norms_ex(_p(x, _u16p), T, D, ctypes.byref(h), ctypes.byref(p), L,
                                    _p(out, _u16p), threads)
    if rc != 0:
        raise ValueError("oracle: unsupported context_norms_ex arguments")
    return out


def kv_project(normed: np.ndarray, W: np.ndarray, rows: Optional[np.ndarray] = None,
               w_nd: bool = False, with_abs: bool = True, threads: int = 0):
    """float64 [L, R, N] projection of the selected rows (all rows when
    ``rows`` is None), and the float64 sum of |products| (or None)."""
    L, T, D = normed.shape
    N = W.shape[1] if w_nd else W.shape[2]
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        R = rows.shape[0]
    else:
        R = T
    out = np.empty((L, R, N), dtype=np.float64)
    ab = np.empty((L, R, N), dtype=np.float64) if with_abs else None
    rc = lib().rco_kv_project(_p(normed, _u16p), _p(W, _u16p), int(w_nd), L, T, D,
                              N, _p(rows, _i64p), R, _p(out, _f64p), _p(ab, _f64p),
                              threads)
    if rc != 0:
        raise ValueError("oracle: unsupported kv_project arguments")
    return out, ab


def kv_store(k: np.ndarray, v: np.ndarray, k_layer_stride: int, k_row_stride: int,
             v_layer_stride: int, v_row_stride: int, positions: Optional[np.ndarray],
             slots: Sequence[Optional[np.ndarray]], cos_sin: Optional[np.ndarray],
             caches: Sequence[np.ndarray], H: int, eps: float, rows: int,
             threads: int = 0) -> int:
    """Runs the store chain in place on ``caches`` (numpy uint16
    [num_blocks, H, block_size, 128] each).  ``k`` and ``v`` are flat uint16
    buffers addressed with the given element strides (they may view the same
    buffer).  Returns the count of rows skipped for an out-of-range slot or
    position."""
    L = len(caches)
    nb, h_, bs, w_ = caches[0].shape
    assert h_ == H and w_ == 128
    slot_arr = (_i64p * L)(*[_p(s, _i64p) if s is not None else ctypes.cast(None, _i64p)
                             for s in slots])
    cache_arr = (_u16p * L)(*[_p(c, _u16p) for c in caches])
    err = np.zeros(1, dtype=np.int32)
    max_pos = cos_sin.shape[0] if cos_sin is not None else 0
    rc = lib().rco_kv_store(_p(k, _u16p), _p(v, _u16p), k_layer_stride, k_row_stride,
                            v_layer_stride, v_row_stride, _p(positions, _i64p),
                            slot_arr, _p(cos_sin, _u16p), max_pos, cache_arr, nb, bs,
                            H, L, eps, rows, _p(err, _i32p), threads)
    if rc != 0:
        raise ValueError("oracle: unsupported kv_store arguments")
    return int(err[0])


def kv_store_from_projection(kv: np.ndarray, H: int, positions, slots, cos_sin,
                             caches, eps: float, rows: int, threads: int = 0) -> int:
    """The store chain fed a projection output ``kv`` bf16 [L, T, 2*H*64]:
    K is columns [0, 64H) and V columns [64H, 128H) of each row ([rt]
    ContextKV.store: ``all_kv.view(L, -1, 2, H, 64)``)."""
    L, T, N = kv.shape
    assert N == 128 * H
    flat = np.ascontiguousarray(kv).reshape(-1)
    if not np.isscalar(rows):
        # per-layer row counts ([rt] _slot_groups: each layer inserts the
        # first len(slots[l]) rows): one layer at a time
        err = 0
        for l in range(L):
            k_l = flat[l * T * N:]
            err += kv_store(k_l, k_l[64 * H:], T * N, N, T * N, N, positions, [slots[l]],
                            cos_sin, [caches[l]], H, eps, int(rows[l]), threads)
        return err
    v_view = flat[64 * H:]          # a view: V starts 64*H elements into a row
    return kv_store(flat, v_view, T * N, N, T * N, N, positions, slots, cos_sin,
                    caches, H, eps, rows, threads)


def qkv_front_post(raw: np.ndarray, num_heads: int, num_kv_heads: int,
                   positions: Optional[np.ndarray], cos_sin: Optional[np.ndarray],
                   slots: Optional[np.ndarray], cache: Optional[np.ndarray], eps: float):
    """The decode QKV front after its projection (reading R15): returns
    (out bf16 [M, Nqkv], skipped-row count); ``cache`` (bf16 [num_blocks,
    num_kv_heads, block_size, 128]) is updated in place."""
    M, N = raw.shape
    assert N == 64 * (2 * num_heads + 2 * num_kv_heads)
    out = np.empty_like(raw)
    err = np.zeros(1, dtype=np.int32)
    nb, bs = (cache.shape[0], cache.shape[2]) if cache is not None else (1, 1)
    max_pos = cos_sin.shape[0] if cos_sin is not None else 0
    rc = lib().rco_qkv_front_post(_p(np.ascontiguousarray(raw), _u16p), M, num_heads, num_kv_heads,
                                  _p(positions, _i64p), _p(cos_sin, _u16p), max_pos,
                                  _p(slots, _i64p), _p(cache, _u16p), nb, bs, eps,
                                  _p(out, _u16p), _p(err, _i32p))
    if rc != 0:
        raise ValueError("oracle: unsupported qkv_front_post arguments")
    return out, int(err[0])


def qkv_project(hidden: np.ndarray, W: np.ndarray, threads: int = 0):
    """float64 projection of the decode QKV front: hidden [M, D] x W^T with W
    the nn.Linear weight [Nqkv, D]; returns (sum, sum of |products|)."""
    M, D = hidden.shape
    out, ab = kv_project(hidden.reshape(1, M, D), W.reshape(1, *W.shape), w_nd=True,
                         threads=threads)
    return out[0], ab[0]
