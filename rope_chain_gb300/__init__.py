"""rope_chain_gb300: the speculative draft's context K/V chain on GB300.

A thin ctypes binding of librope_chain.so (include/rope_chain.h).  It only
marshals torch CUDA tensors into pointers, sizes and the current stream;
every step of the chain runs in the library's CUDA kernels.  There is no CPU
path: if the library is missing, every call raises.

    normed = context_norms(x, hidden_w, pre_w, L, eps)          # [L, T, 8192]
    kv     = kv_project(normed, W)                              # [L, T, 128*H]
    kv_store_from_projection(kv, H, positions, slots, cos_sin, caches, eps)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librope_chain.so")

RC_OK, RC_ERR_INVALID_ARG, RC_ERR_UNSUPPORTED, RC_ERR_CUDA = 0, 1, 2, 3
RC_W_KN, RC_W_NK = 0, 1
HEAD_DIM = 64
MAX_LAYERS_PER_LAUNCH = 8


class RopeChainError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"status {status}: {message}")
        self.status = status


_lib = None
_c = ctypes
_vp = ctypes.c_void_p

SIGNATURES = {
    "rc_last_error": ([], _c.c_char_p),
    "rc_version": ([], _c.c_int32),
    "rc_context_norms": ([_vp, _c.c_int64, _c.c_int32, _vp, _vp, _c.c_int32, _c.c_float, _vp, _vp],
                         _c.c_int),
    "rc_kv_project": ([_vp, _vp, _c.c_int32, _vp, _c.c_int32, _c.c_int64, _c.c_int32, _c.c_int32,
                       _vp, _c.c_size_t, _vp], _c.c_int),
    "rc_kv_project_workspace_size": ([_c.c_int32, _c.c_int64, _c.c_int32, _c.c_int32], _c.c_size_t),
    "rc_kv_project_workspace_size_sms": ([_c.c_int32, _c.c_int64, _c.c_int32, _c.c_int32, _c.c_int32],
                                         _c.c_size_t),
    "rc_kv_store": ([_vp, _vp, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64, _vp,
                     _c.POINTER(_vp), _vp, _c.c_int64, _c.POINTER(_vp), _c.c_int32, _c.c_int32,
                     _c.c_int32, _c.c_int32, _c.c_float, _c.c_int64, _vp, _vp], _c.c_int),
    "rc_read_device_faults": ([_c.POINTER(_c.c_uint32), _c.c_int32], _c.c_int),
    "rc_device_address": ([_vp, _c.POINTER(_vp)], _c.c_int),
    "rc_kv_project_no_alloc": ([_vp, _vp, _c.c_int32, _vp, _c.c_int32, _c.c_int64, _c.c_int32,
                                _c.c_int32, _vp], _c.c_int),
    "rc_context_kv": ([_vp, _c.c_int64, _c.c_int32, _vp, _vp, _c.c_int32, _c.c_float, _vp,
                       _c.c_int32, _c.c_int32, _vp, _c.POINTER(_vp), _vp, _c.c_int64,
                       _c.POINTER(_vp), _c.c_int32, _c.c_int32, _c.c_int64, _vp, _vp, _vp,
                       _c.c_size_t, _vp], _c.c_int),
    "rc_context_rows": ([_vp, _c.c_int64, _c.c_int32, _vp, _c.c_float, _vp, _vp, _vp], _c.c_int),
    "rc_context_kv_from_rows": ([_vp, _vp, _c.c_int64, _c.c_int32, _vp, _c.c_int32, _c.c_float, _vp,
                                 _c.c_int32, _c.c_int32, _vp, _c.POINTER(_vp), _vp, _c.c_int64,
                                 _c.POINTER(_vp), _c.c_int32, _c.c_int32, _c.c_int64, _vp, _vp,
                                 _vp, _c.c_size_t, _vp], _c.c_int),
    "rc_context_kv_workspace_size": ([_c.c_int32, _c.c_int64, _c.c_int32, _c.c_int32], _c.c_size_t),
    "rc_kv_project_store": ([_vp, _vp, _c.c_int32, _c.c_int32, _c.c_int64, _c.c_int32, _c.c_int32,
                             _vp, _c.POINTER(_vp), _vp, _c.c_int64, _c.POINTER(_vp), _c.c_int32,
                             _c.c_int32, _c.c_float, _c.c_int64, _vp, _vp, _vp, _c.c_size_t, _vp],
                            _c.c_int),
    "rc_kv_project_store_rows": ([_vp, _vp, _c.c_int32, _c.c_int32, _c.c_int64, _c.c_int32,
                                  _c.c_int32, _vp, _c.POINTER(_vp), _vp, _c.c_int64,
                                  _c.POINTER(_vp), _c.c_int32, _c.c_int32, _c.c_float,
                                  _c.POINTER(_c.c_int64), _vp, _vp, _vp, _c.c_size_t, _vp],
                                 _c.c_int),
    "rc_kv_store_rows": ([_vp, _vp, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64, _vp,
                          _c.POINTER(_vp), _vp, _c.c_int64, _c.POINTER(_vp), _c.c_int32, _c.c_int32,
                          _c.c_int32, _c.c_int32, _c.c_float, _c.POINTER(_c.c_int64), _vp, _vp],
                         _c.c_int),
}


class NormParams(ctypes.Structure):
    """rc_norm_params: one norm's weight (device pointer), its dtype
    (RC_NORM_*), scale side, gain center and eps."""
    _fields_ = [("weight", _vp), ("weight_dtype", _c.c_int32), ("input_scale", _c.c_int32),
                ("gain_center", _c.c_float), ("eps", _c.c_float)]


class ProjectPlan(ctypes.Structure):
    """rc_project_plan: how a projection runs (kernel 0 single CTAs, 1 CTA
    pairs, 2 persistent CTA pairs; K splits; tail splits; dynamic tiles;
    workspace bytes used)."""
    _fields_ = [("kernel", _c.c_int32), ("splits", _c.c_int32), ("tail_splits", _c.c_int32),
                ("dynamic_tiles", _c.c_int32), ("tail_row0", _c.c_int64),
                ("workspace_bytes", _c.c_size_t)]


SIGNATURES["rc_kv_project_plan"] = ([_c.c_int32, _c.c_int64, _c.c_int32, _c.c_int32, _c.c_int32,
                                     _c.c_size_t, _c.POINTER(ProjectPlan)], _c.c_int)

RC_NORM_NONE, RC_NORM_BF16, RC_NORM_F32 = 0, 1, 2
SIGNATURES["rc_qkv_front"] = ([_vp, _c.c_int32, _c.c_int32, _vp, _c.c_int32, _c.c_int32, _vp, _vp,
                               _c.c_int64, _vp, _vp, _c.c_int32, _c.c_int32, _c.c_float, _vp, _vp,
                               _vp, _vp], _c.c_int)
SIGNATURES["rc_context_norms_ex"] = ([_vp, _c.c_int64, _c.c_int32, _c.POINTER(NormParams),
                                      _c.POINTER(NormParams), _c.c_int32, _vp, _vp], _c.c_int)
SIGNATURES["rc_context_kv_chunked"] = ([_vp, _c.c_int64, _c.c_int32, _vp, _vp, _c.c_int32, _c.c_float,
                                        _vp, _c.c_int32, _c.c_int32, _vp, _c.POINTER(_vp), _vp,
                                        _c.c_int64, _c.POINTER(_vp), _c.c_int32, _c.c_int32,
                                        _c.c_int64, _vp, _c.c_int32, _vp, _c.c_size_t, _vp], _c.c_int)
SIGNATURES["rc_context_kv_chunked_ex"] = ([_vp, _c.c_int64, _c.c_int32, _c.POINTER(NormParams),
                                           _c.POINTER(NormParams), _c.c_int32, _vp, _c.c_int32,
                                           _c.c_int32, _vp, _c.POINTER(_vp), _vp, _c.c_int64,
                                           _c.POINTER(_vp), _c.c_int32, _c.c_int32, _c.c_float,
                                           _c.POINTER(_c.c_int64), _vp, _c.c_int32, _vp, _c.c_size_t,
                                           _vp], _c.c_int)
SIGNATURES["rc_context_kv_chunked_workspace_size"] = ([_c.c_int32, _c.c_int64, _c.c_int32, _c.c_int32,
                                                       _c.c_int32], _c.c_size_t)
SIGNATURES["rc_context_kv_chunks"] = ([_c.c_int32, _c.c_int64, _c.c_int32, _c.c_int32, _c.c_int32,
                                       _c.c_int32, _c.c_int32, _c.POINTER(_c.c_int64)], _c.c_int32)


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != RC_OK:
        raise RopeChainError(status, lib().rc_last_error().decode())


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _bf16(t: torch.Tensor, name: str) -> None:
    if t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA bfloat16 tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def device_address(t: torch.Tensor) -> int:
    """The address at which the current GPU reads t's data: t's own for a
    CUDA tensor; for a pinned (page-locked) CPU tensor its mapped device
    address (rc_device_address), so that a kernel reads it in place over the
    host link."""
    if t.is_cuda:
        return t.data_ptr()
    if t.device.type == "cpu" and t.is_pinned():
        # the mapping of the storage's start, plus t's offset into it (t may
        # be a slice of a pinned buffer)
        base = t.untyped_storage().data_ptr()
        d = _vp(0)
        _check(lib().rc_device_address(base, ctypes.byref(d)))
        return int(d.value) + (t.data_ptr() - base)
    raise TypeError("expected a CUDA tensor or a pinned CPU tensor")


def _in_bf16(t: torch.Tensor, name: str) -> int:
    """A bf16 input the kernels may read in place (CUDA or pinned host
    memory); returns its device address."""
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be a bfloat16 tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return device_address(t)


def _out_device(x: torch.Tensor) -> torch.device:
    return x.device if x.is_cuda else torch.device("cuda", torch.cuda.current_device())


# ------------------------------------------------------------------- calls

def context_norms(x: torch.Tensor, hidden_w: Optional[torch.Tensor],
                  pre_w: Optional[torch.Tensor], L: int, eps: float,
                  out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """bf16 [L, T, 8192] = stack_l(pre_norm_l(bf16(hidden_norm(x)))).  x may
    be a pinned CPU tensor (read in place over the host link)."""
    xa = _in_bf16(x, "x")
    T, D = x.shape
    if out is None:
        out = torch.empty((L, T, D), dtype=torch.bfloat16, device=_out_device(x))
    _bf16(out, "out")
    for w, n in ((hidden_w, "hidden_w"), (pre_w, "pre_w")):
        if w is not None:
            _bf16(w, n)
    _check(lib().rc_context_norms(xa, T, D, _ptr(hidden_w), _ptr(pre_w), L, eps,
                                  out.data_ptr(), _stream(stream)))
    return out


def _norm_params(w: Optional[torch.Tensor], input_scale: bool, center: float, eps: float,
                 name: str) -> NormParams:
    if w is None:
        return NormParams(None, RC_NORM_NONE, 0, 0.0, eps)
    if not w.is_cuda or not w.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if w.dtype == torch.bfloat16:
        dt = RC_NORM_BF16
    elif w.dtype == torch.float32:
        dt = RC_NORM_F32
    else:
        raise TypeError(f"{name} must be bfloat16 or float32")
    return NormParams(w.data_ptr(), dt, int(bool(input_scale)), center, eps)


def context_norms_ex(x: torch.Tensor, L: int, *, hidden_w: Optional[torch.Tensor] = None,
                     pre_w: Optional[torch.Tensor] = None, hidden_eps: float, pre_eps: float,
                     hidden_center: float = 0.0, pre_center: float = 0.0,
                     hidden_input_scale: bool = False, pre_input_scale: bool = False,
                     out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """context_norms with every norm option (rc_context_norms_ex): weights
    bf16 or float32 ([8192] hidden, [L, 8192] layers), each norm's eps and
    gain center, and whether each weight scales the norm's input.  x may be a
    pinned CPU tensor."""
    xa = _in_bf16(x, "x")
    T, D = x.shape
    if out is None:
        out = torch.empty((L, T, D), dtype=torch.bfloat16, device=_out_device(x))
    _bf16(out, "out")
    if hidden_w is not None and tuple(hidden_w.shape) != (D,):
        raise ValueError("hidden_w must be [8192]")
    if pre_w is not None and tuple(pre_w.shape) != (L, D):
        raise ValueError("pre_w must be [L, 8192]")
    h = _norm_params(hidden_w, hidden_input_scale, hidden_center, hidden_eps, "hidden_w")
    p = _norm_params(pre_w, pre_input_scale, pre_center, pre_eps, "pre_w")
    _check(lib().rc_context_norms_ex(xa, T, D, ctypes.byref(h), ctypes.byref(p), L,
                                     out.data_ptr(), _stream(stream)))
    return out


def _layer_rows(slots, rows):
    """(rows, per-layer row counts or None): an int applies to every layer; a
    sequence gives each layer its count; None takes each layer's slot-mapping
    length (0 for a None layer), collapsing to one count when they agree."""
    if rows is None:
        lens = [0 if sl is None else int(sl.shape[0]) for sl in slots]
        live = {n for n, sl in zip(lens, slots) if sl is not None}
        if len(live) <= 1:
            return (live.pop() if live else 0), None
        return 0, lens
    if isinstance(rows, int):
        return rows, None
    lens = [int(r) for r in rows]
    if len(lens) != len(slots):
        raise ValueError("rows needs one count per layer")
    return 0, lens


def _check_slot_lengths(slots, rows, per_layer):
    for i, sl in enumerate(slots):
        need = rows if per_layer is None else per_layer[i]
        if sl is not None and sl.shape[0] < need:
            raise ValueError(f"slots[{i}] has fewer than its {need} rows")


def workspace_size(L: int, T: int, D: int, N: int) -> int:
    """Bytes of split-K scratch rc_kv_project uses for these sizes (0: none)."""
    return int(lib().rc_kv_project_workspace_size(L, T, D, N))


def new_workspace(L: int, T: int, D: int, N: int, device) -> Optional[torch.Tensor]:
    """A split-K workspace for these sizes (None when not needed)."""
    n = workspace_size(L, T, D, N)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def _project_shapes(normed: torch.Tensor, W: torch.Tensor, w_layout: int):
    """(L, T, D, N) of a projection; W must be [L, D, N] (RC_W_KN) or
    [L, N, D] (RC_W_NK) for normed [L, T, D]."""
    _bf16(normed, "normed")
    _bf16(W, "W")
    if normed.dim() != 3 or W.dim() != 3:
        raise ValueError("normed and W must be 3-dimensional")
    L, T, D = normed.shape
    if w_layout == RC_W_KN:
        N = W.shape[2]
        want = (L, D, N)
    elif w_layout == RC_W_NK:
        N = W.shape[1]
        want = (L, N, D)
    else:
        raise ValueError(f"unknown weight layout {w_layout}")
    if tuple(W.shape) != want:
        raise ValueError(f"W has shape {tuple(W.shape)}; normed {tuple(normed.shape)} needs {want}")
    return L, T, D, N


def _project_out_shape(out: torch.Tensor, L: int, T: int, N: int) -> None:
    if tuple(out.shape) != (L, T, N):
        raise ValueError(f"out has shape {tuple(out.shape)}; the projection writes {(L, T, N)}")


def project_plan(L: int, T: int, D: int, N: int, num_sms: int, workspace_bytes: int) -> dict:
    """How a projection of these sizes runs on a GPU with num_sms SMs given
    workspace_bytes of workspace (host-only)."""
    p = ProjectPlan()
    _check(lib().rc_kv_project_plan(L, T, D, N, num_sms, workspace_bytes, ctypes.byref(p)))
    return {"kernel": ("single CTAs", "CTA pairs", "persistent CTA pairs")[p.kernel],
            "splits": p.splits, "tail_splits": p.tail_splits,
            "dynamic_tiles": bool(p.dynamic_tiles), "tail_row0": int(p.tail_row0),
            "workspace_bytes": int(p.workspace_bytes)}


def workspace_size_for(L: int, T: int, D: int, N: int, num_sms: int) -> int:
    """Split-K workspace bytes of a projection on a GPU with num_sms SMs
    (host-only: no device is needed)."""
    return int(lib().rc_kv_project_workspace_size_sms(L, T, D, N, num_sms))


def kv_project(normed: torch.Tensor, W: torch.Tensor, out: Optional[torch.Tensor] = None,
               w_layout: int = RC_W_KN, workspace: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """bf16 [L, T, N] = normed [L, T, D] x W, W [L, D, N] (RC_W_KN) or
    [L, N, D] (RC_W_NK).  ``workspace`` (any dtype, contiguous; see
    new_workspace() and workspace_size()) enables split-K for small T."""
    L, T, D, N = _project_shapes(normed, W, w_layout)
    if out is None:
        out = torch.empty((L, T, N), dtype=torch.bfloat16, device=normed.device)
    _bf16(out, "out")
    _project_out_shape(out, L, T, N)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        if not (workspace.is_cuda and workspace.is_contiguous()):
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(lib().rc_kv_project(normed.data_ptr(), W.data_ptr(), w_layout, out.data_ptr(), L, T, D,
                               N, ws_ptr, ws_bytes, _stream(stream)))
    return out


def kv_project_no_alloc(normed: torch.Tensor, W: torch.Tensor, out: torch.Tensor,
                        w_layout: int = RC_W_KN, stream=None) -> torch.Tensor:
    """kv_project for callers that cannot allocate device memory: the split-K
    scratch lives inside the library (24 MiB per GPU), ``out`` must be given,
    and calls that overlap on the GPU must not be issued (they share the
    scratch)."""
    L, T, D, N = _project_shapes(normed, W, w_layout)
    _bf16(out, "out")
    _project_out_shape(out, L, T, N)
    _check(lib().rc_kv_project_no_alloc(normed.data_ptr(), W.data_ptr(), w_layout,
                                        out.data_ptr(), L, T, D, N, _stream(stream)))
    return out


def kv_store(k: torch.Tensor, v: torch.Tensor, positions: Optional[torch.Tensor],
             slots: Sequence[Optional[torch.Tensor]], cos_sin: Optional[torch.Tensor],
             caches: Sequence[torch.Tensor], eps: float, rows: Optional[int] = None,
             err: Optional[torch.Tensor] = None, stream=None) -> None:
    """K-norm, GPT-J RoPE (with ``cos_sin``) and paged insert.  ``k`` and
    ``v`` are bf16 [L, T, H, 64] views (unit stride over the last two dims);
    ``caches[l]`` bf16 [num_blocks, H, block_size, 128] contiguous;
    ``slots[l]`` int64 [rows] or None; ``err`` an int32 [1] counter."""
    L, T, H, hd = k.shape
    if hd != HEAD_DIM or tuple(v.shape) != (L, T, H, hd):
        raise ValueError("k and v must be [L, T, H, 64] views of one shape")
    for t, n in ((k, "k"), (v, "v")):
        if t.dtype != torch.bfloat16 or t.stride(3) != 1 or t.stride(2) != HEAD_DIM:
            raise ValueError(f"{n} must be bf16 with strides (*, *, 64, 1)")
    if len(slots) != L or len(caches) != L:
        raise ValueError("slots and caches need one entry per layer")
    nb, h_, bs, w_ = caches[0].shape
    if h_ != H or w_ != 2 * HEAD_DIM:
        raise ValueError("caches must be [num_blocks, H, block_size, 128]")
    for c in caches:
        _bf16(c, "cache")
        if tuple(c.shape) != (nb, h_, bs, w_):
            raise ValueError("all caches must have one shape")
    for s in slots:
        if s is not None and (s.dtype != torch.int64 or not s.is_contiguous() or not s.is_cuda):
            raise ValueError("slots must be contiguous CUDA int64 tensors")
    rows, per_layer = _layer_rows(slots, rows)
    _check_slot_lengths(slots, rows, per_layer)
    if cos_sin is not None:
        _bf16(cos_sin, "cos_sin")
        if positions is None or positions.dtype != torch.int64 or not positions.is_contiguous():
            raise ValueError("RoPE needs contiguous int64 positions")
    slot_arr = (_vp * L)(*[_ptr(s) for s in slots])
    cache_arr = (_vp * L)(*[c.data_ptr() for c in caches])
    args = (k.data_ptr(), v.data_ptr(), k.stride(0), k.stride(1), v.stride(0), v.stride(1),
            _ptr(positions), slot_arr, _ptr(cos_sin), 0 if cos_sin is None else cos_sin.shape[0],
            cache_arr, nb, bs, H, L, eps)
    if per_layer is None:
        _check(lib().rc_kv_store(*args, rows, _ptr(err), _stream(stream)))
    else:
        _check(lib().rc_kv_store_rows(*args, (_c.c_int64 * L)(*per_layer), _ptr(err),
                                      _stream(stream)))


def kv_project_store(normed: torch.Tensor, W: torch.Tensor, H: int, positions, slots,
                     cos_sin, caches, eps: float, rows: Optional[int] = None, err=None,
                     kv_out: Optional[torch.Tensor] = None, w_layout: int = RC_W_KN,
                     workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Projection and store in one pass (rc_kv_project_store): the caches get
    the bits kv_project + kv_store_from_projection would write."""
    _bf16(normed, "normed")
    _bf16(W, "W")
    L, T, D = normed.shape
    if len(slots) != L or len(caches) != L:
        raise ValueError("slots and caches need one entry per layer")
    nb, h_, bs, w_ = caches[0].shape
    if h_ != H or w_ != 2 * HEAD_DIM:
        raise ValueError("caches must be [num_blocks, H, block_size, 128]")
    for c in caches:
        _bf16(c, "cache")
        if tuple(c.shape) != (nb, h_, bs, w_):
            raise ValueError("all caches must have one shape")
    for sl in slots:
        if sl is not None and (sl.dtype != torch.int64 or not sl.is_contiguous() or not sl.is_cuda):
            raise ValueError("slots must be contiguous CUDA int64 tensors")
    rows, per_layer = _layer_rows(slots, rows)
    _check_slot_lengths(slots, rows, per_layer)
    if cos_sin is not None:
        _bf16(cos_sin, "cos_sin")
        if positions is None or positions.dtype != torch.int64 or not positions.is_contiguous():
            raise ValueError("RoPE needs contiguous int64 positions")
    if kv_out is not None:
        _bf16(kv_out, "kv_out")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    slot_arr = (_vp * L)(*[_ptr(sl) for sl in slots])
    cache_arr = (_vp * L)(*[c.data_ptr() for c in caches])
    head = (normed.data_ptr(), W.data_ptr(), w_layout, L, T, D, H, _ptr(positions), slot_arr,
            _ptr(cos_sin), 0 if cos_sin is None else cos_sin.shape[0], cache_arr, nb, bs, eps)
    tail = (_ptr(err), _ptr(kv_out), ws_ptr, ws_bytes, _stream(stream))
    if per_layer is None:
        _check(lib().rc_kv_project_store(*head, rows, *tail))
    else:
        _check(lib().rc_kv_project_store_rows(*head, (_c.c_int64 * L)(*per_layer), *tail))


def context_kv_workspace(L: int, T: int, H: int, device, D: int = 8192) -> torch.Tensor:
    """A workspace for context_kv (rc_context_kv_workspace_size bytes)."""
    n = int(lib().rc_context_kv_workspace_size(L, T, D, H))
    if n == 0:
        raise RopeChainError(RC_ERR_UNSUPPORTED, "no workspace size for these sizes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def _store_operands(H, slots, caches, positions, cos_sin, rows):
    L = len(caches)
    nb, h_, bs, w_ = caches[0].shape
    if h_ != H or w_ != 2 * HEAD_DIM:
        raise ValueError("caches must be [num_blocks, H, block_size, 128]")
    for c in caches:
        _bf16(c, "cache")
        if tuple(c.shape) != (nb, h_, bs, w_):
            raise ValueError("all caches must have one shape")
    if len(slots) != L:
        raise ValueError("slots and caches need one entry per layer")
    for sl in slots:
        if sl is not None and (sl.dtype != torch.int64 or not sl.is_contiguous() or not sl.is_cuda):
            raise ValueError("slots must be contiguous CUDA int64 tensors")
    if rows is None:
        first = next((sl for sl in slots if sl is not None), None)
        rows = 0 if first is None else first.shape[0]
    for sl in slots:
        if sl is not None and sl.shape[0] < rows:
            raise ValueError("every slot mapping needs at least `rows` entries")
    if cos_sin is not None:
        _bf16(cos_sin, "cos_sin")
        if positions is None or positions.dtype != torch.int64 or not positions.is_contiguous():
            raise ValueError("RoPE needs contiguous int64 positions")
    slot_arr = (_vp * L)(*[_ptr(sl) for sl in slots])
    cache_arr = (_vp * L)(*[c.data_ptr() for c in caches])
    return slot_arr, cache_arr, nb, bs, rows


def context_kv(x: torch.Tensor, hidden_w, pre_w, W: torch.Tensor, H: int, positions, slots,
               cos_sin, caches, eps: float, workspace: torch.Tensor, rows: Optional[int] = None,
               err=None, kv_out: Optional[torch.Tensor] = None, w_layout: int = RC_W_KN,
               stream=None) -> None:
    """The whole chain in one call (rc_context_kv): norms fused into the
    projection, store fused after it.  ``workspace``: context_kv_workspace()."""
    xa = _in_bf16(x, "x")                          # CUDA or pinned host memory
    _bf16(W, "W")
    T, D = x.shape
    L = len(caches)
    for w_, n in ((hidden_w, "hidden_w"), (pre_w, "pre_w")):
        if w_ is not None:
            _bf16(w_, n)
    if kv_out is not None:
        _bf16(kv_out, "kv_out")
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    slot_arr, cache_arr, nb, bs, rows = _store_operands(H, slots, caches, positions, cos_sin, rows)
    _check(lib().rc_context_kv(xa, T, D, _ptr(hidden_w), _ptr(pre_w), L, eps,
                               W.data_ptr(), w_layout, H, _ptr(positions), slot_arr, _ptr(cos_sin),
                               0 if cos_sin is None else cos_sin.shape[0], cache_arr, nb, bs, rows,
                               _ptr(err), _ptr(kv_out), workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), _stream(stream)))


def context_kv_chunks(L: int, T: int, H: int, num_sms: int, chunks: int = 0, D: int = 8192,
                      x_on_host: bool = False) -> int:
    """Row chunks rc_context_kv_chunked uses for these sizes (host only)."""
    return int(lib().rc_context_kv_chunks(L, T, D, H, chunks, int(x_on_host), num_sms, None))


def context_kv_chunk_rows(L: int, T: int, H: int, num_sms: int, chunks: int = 0,
                          D: int = 8192, x_on_host: bool = False) -> list:
    """The first row of each chunk rc_context_kv_chunked uses, then T (host
    only; [] for unsupported sizes)."""
    row0 = (_c.c_int64 * 17)()
    n = int(lib().rc_context_kv_chunks(L, T, D, H, chunks, int(x_on_host), num_sms, row0))
    return [int(row0[i]) for i in range(n + 1)] if n else []


def context_kv_chunked_workspace(L: int, T: int, H: int, device, chunks: int = 0,
                                 D: int = 8192) -> torch.Tensor:
    """A workspace for context_kv_chunked (rc_context_kv_chunked_workspace_size bytes)."""
    n = int(lib().rc_context_kv_chunked_workspace_size(L, T, D, H, chunks))
    if n == 0:
        raise RopeChainError(RC_ERR_UNSUPPORTED, "no workspace size for these sizes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def context_kv_chunked(x: torch.Tensor, hidden_w, pre_w, W: torch.Tensor, H: int, positions, slots,
                       cos_sin, caches, eps: float, workspace: torch.Tensor,
                       rows: Optional[int] = None, err=None, chunks: int = 0,
                       w_layout: int = RC_W_KN, stream=None) -> None:
    """Norms, projection and store by row chunks (rc_context_kv_chunked): a
    chunk's norms run beside the previous chunk's projection.
    ``workspace``: context_kv_chunked_workspace() with the same ``chunks``."""
    xa = _in_bf16(x, "x")                          # CUDA or pinned host memory
    _bf16(W, "W")
    T, D = x.shape
    L = len(caches)
    for w_, n in ((hidden_w, "hidden_w"), (pre_w, "pre_w")):
        if w_ is not None:
            _bf16(w_, n)
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    slot_arr, cache_arr, nb, bs, rows = _store_operands(H, slots, caches, positions, cos_sin, rows)
    _check(lib().rc_context_kv_chunked(xa, T, D, _ptr(hidden_w), _ptr(pre_w), L, eps,
                                       W.data_ptr(), w_layout, H, _ptr(positions), slot_arr,
                                       _ptr(cos_sin), 0 if cos_sin is None else cos_sin.shape[0],
                                       cache_arr, nb, bs, rows, _ptr(err), chunks,
                                       workspace.data_ptr(),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream)))


def context_kv_chunked_ex(x: torch.Tensor, W: torch.Tensor, H: int, positions, slots, cos_sin,
                          caches, eps: float, workspace: torch.Tensor, *,
                          hidden_w: Optional[torch.Tensor] = None,
                          pre_w: Optional[torch.Tensor] = None, hidden_eps: float, pre_eps: float,
                          hidden_center: float = 0.0, pre_center: float = 0.0,
                          hidden_input_scale: bool = False, pre_input_scale: bool = False,
                          rows=None, err=None, chunks: int = 0, w_layout: int = RC_W_KN,
                          stream=None) -> None:
    """context_kv_chunked with every norm option of context_norms_ex and a
    row count per layer (rc_context_kv_chunked_ex).  ``eps``: the K-norm's;
    ``rows``: an int, one count per layer, or None for each layer's
    slot-mapping length."""
    xa = _in_bf16(x, "x")                          # CUDA or pinned host memory
    _bf16(W, "W")
    T, D = x.shape
    L = len(caches)
    if hidden_w is not None and tuple(hidden_w.shape) != (D,):
        raise ValueError("hidden_w must be [8192]")
    if pre_w is not None and tuple(pre_w.shape) != (L, D):
        raise ValueError("pre_w must be [L, 8192]")
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    h = _norm_params(hidden_w, hidden_input_scale, hidden_center, hidden_eps, "hidden_w")
    p = _norm_params(pre_w, pre_input_scale, pre_center, pre_eps, "pre_w")
    n_rows, per_layer = _layer_rows(slots, rows)
    _check_slot_lengths(slots, n_rows, per_layer)
    slot_arr, cache_arr, nb, bs, _ = _store_operands(H, slots, caches, positions, cos_sin, 0)
    counts = (_c.c_int64 * L)(*(per_layer if per_layer is not None else [n_rows] * L))
    _check(lib().rc_context_kv_chunked_ex(xa, T, D, ctypes.byref(h), ctypes.byref(p), L,
                                          W.data_ptr(), w_layout, H, _ptr(positions), slot_arr,
                                          _ptr(cos_sin), 0 if cos_sin is None else cos_sin.shape[0],
                                          cache_arr, nb, bs, eps, counts, _ptr(err), chunks,
                                          workspace.data_ptr(),
                                          workspace.numel() * workspace.element_size(),
                                          _stream(stream)))


def context_rows(x: torch.Tensor, hidden_w, eps: float, z: Optional[torch.Tensor] = None,
                 r2: Optional[torch.Tensor] = None, stream=None):
    """The row pass of context_kv: (z bf16 [T, 8192], r2 float32 [T]); x may
    be a pinned CPU tensor."""
    xa = _in_bf16(x, "x")
    T, D = x.shape
    if z is None:
        z = torch.empty((T, D), dtype=torch.bfloat16, device=_out_device(x))
    if r2 is None:
        r2 = torch.empty((T,), dtype=torch.float32, device=_out_device(x))
    if hidden_w is not None:
        _bf16(hidden_w, "hidden_w")
    _check(lib().rc_context_rows(xa, T, D, _ptr(hidden_w), eps, z.data_ptr(),
                                 r2.data_ptr(), _stream(stream)))
    return z, r2


def context_kv_from_rows(z: torch.Tensor, r2: torch.Tensor, pre_w, W: torch.Tensor, H: int,
                         positions, slots, cos_sin, caches, eps: float, rows=None, err=None,
                         kv_out=None, workspace=None, w_layout: int = RC_W_KN, stream=None) -> None:
    """The projection and store of context_kv from its row pass."""
    _bf16(z, "z")
    _bf16(W, "W")
    T, D = z.shape
    L = len(caches)
    if pre_w is not None:
        _bf16(pre_w, "pre_w")
    if kv_out is not None:
        _bf16(kv_out, "kv_out")
    slot_arr, cache_arr, nb, bs, rows = _store_operands(H, slots, caches, positions, cos_sin, rows)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    _check(lib().rc_context_kv_from_rows(z.data_ptr(), r2.data_ptr(), T, D, _ptr(pre_w), L, eps,
                                         W.data_ptr(), w_layout, H, _ptr(positions), slot_arr,
                                         _ptr(cos_sin), 0 if cos_sin is None else cos_sin.shape[0],
                                         cache_arr, nb, bs, rows, _ptr(err), _ptr(kv_out), ws_ptr,
                                         ws_bytes, _stream(stream)))


def split_kv(kv: torch.Tensor, H: int):
    """K and V views of a projection output kv [L, T, 2*H*64]: K is the first
    64H columns of each row, V the next 64H."""
    L, T, N = kv.shape
    v5 = kv.view(L, T, 2, H, HEAD_DIM)
    return v5[:, :, 0], v5[:, :, 1]


def kv_store_from_projection(kv: torch.Tensor, H: int, positions, slots, cos_sin, caches,
                             eps: float, rows: Optional[int] = None, err=None, stream=None):
    k, v = split_kv(kv, H)
    kv_store(k, v, positions, slots, cos_sin, caches, eps, rows=rows, err=err, stream=stream)


def context_kv_chain(x, hidden_w, pre_w, W, positions, slots, cos_sin, caches, eps, H,
                     normed=None, kv=None, workspace=None, err=None, stream=None):
    """The whole chain: norms, projection, store.  Intermediates may be
    passed in to avoid allocation.  Returns (normed, kv)."""
    L = len(caches)
    normed = context_norms(x, hidden_w, pre_w, L, eps, out=normed, stream=stream)
    kv = kv_project(normed, W, out=kv, workspace=workspace, stream=stream)
    kv_store_from_projection(kv, H, positions, slots, cos_sin, caches, eps, err=err, stream=stream)
    return normed, kv


def qkv_front(hidden: torch.Tensor, W: torch.Tensor, num_heads: int, num_kv_heads: int,
              positions: Optional[torch.Tensor], cos_sin: Optional[torch.Tensor],
              slots: Optional[torch.Tensor], cache: Optional[torch.Tensor], eps: float,
              out: Optional[torch.Tensor] = None, raw_out: Optional[torch.Tensor] = None,
              err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The decode QKV front of one layer (rc_qkv_front): hidden bf16 [M, D]
    (M <= 16), W bf16 [Nqkv, D]; returns out bf16 [M, Nqkv] = [Q | K | V |
    gate] with Q and K normed and rotated, and inserts K and V into ``cache``
    (bf16 [num_blocks, num_kv_heads, block_size, 128]) at ``slots``."""
    _bf16(hidden, "hidden")
    _bf16(W, "W")
    M, D = hidden.shape
    N = HEAD_DIM * (2 * num_heads + 2 * num_kv_heads)
    if tuple(W.shape) != (N, D):
        raise ValueError(f"W must be [{N}, {D}] for these head counts")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=hidden.device)
    _bf16(out, "out")
    if raw_out is not None:
        _bf16(raw_out, "raw_out")
    nb = bs = 0
    if slots is not None:
        if slots.dtype != torch.int64 or not slots.is_contiguous() or slots.shape[0] < M:
            raise ValueError("slots must be contiguous int64 [M]")
        _bf16(cache, "cache")
        nb, h_, bs, w_ = cache.shape
        if h_ != num_kv_heads or w_ != 2 * HEAD_DIM:
            raise ValueError("cache must be [num_blocks, num_kv_heads, block_size, 128]")
    if cos_sin is not None:
        _bf16(cos_sin, "cos_sin")
        if positions is None or positions.dtype != torch.int64 or not positions.is_contiguous():
            raise ValueError("RoPE needs contiguous int64 positions")
    _check(lib().rc_qkv_front(hidden.data_ptr(), M, D, W.data_ptr(), num_heads, num_kv_heads,
                              _ptr(positions), _ptr(cos_sin),
                              0 if cos_sin is None else cos_sin.shape[0], _ptr(slots),
                              _ptr(cache) if slots is not None else None, nb, bs, eps,
                              out.data_ptr(), _ptr(raw_out), _ptr(err), _stream(stream)))
    return out


def read_device_faults(clear: bool = True) -> int:
    """Sticky fault bits of the projection kernel's bounded waits (0: none)."""
    f = ctypes.c_uint32(0)
    _check(lib().rc_read_device_faults(ctypes.byref(f), 1 if clear else 0))
    return int(f.value)
