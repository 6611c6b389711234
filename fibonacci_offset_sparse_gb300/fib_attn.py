"""Thin Python binding of libfibattn.so (argument marshalling only).

Function names mirror the C ABI in include/fib_attn.h.  Tensors are torch tensors on the
plan's CUDA device, contiguous [B, H, N, 64]; the binding passes their data pointers and
the current torch stream.  Every computation runs in the library's CUDA kernels: there is
no CPU fallback, and a missing or unloadable library raises immediately.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfibattn.so")

FIB_OK, FIB_ERR_INVALID_ARG, FIB_ERR_UNSUPPORTED, FIB_ERR_CUDA, FIB_ERR_NOMEM, \
    FIB_ERR_TIMEOUT, FIB_ERR_DEVICE_ASSERT, FIB_ERR_RANGE = range(8)
FIB_DEBUG_SKIP_COPY, FIB_DEBUG_CORRUPT_TABLE = 1, 2
FIB_BASE_FIBONACCI, FIB_BASE_POW2, FIB_BASE_CUSTOM = 0, 1, 2
FIB_SCHED_FIXED, FIB_SCHED_LINEAR, FIB_SCHED_COPRIME = 0, 1, 2
FIB_MODE_MASK, FIB_MODE_INTERP = 0, 1
FIB_DTYPE_F32, FIB_DTYPE_BF16 = 0, 1
FIB_HEAD_DIM, FIB_MAX_RUNGS, FIB_MAX_WINDOW, FIB_MAX_LAYERS = 64, 32, 64, 256

EXPORTS = [
    "fib_attn_error_string", "fib_attn_base", "fib_attn_schedule", "fib_attn_mask_distances",
    "fib_attn_interp_rungs", "fib_attn_plan_create", "fib_attn_plan_destroy",
    "fib_attn_plan_distances", "fib_attn_fwd_workspace_size", "fib_attn_fwd",
    "fib_attn_fwd_prepare_kv", "fib_attn_fwd_attend", "fib_attn_bwd_workspace_size", "fib_attn_bwd",
    "fib_attn_debug_indices", "fib_attn_last_device_status", "fib_attn_plan_set_debug",
    "fib_attn_bwd_noalloc", "fib_attn_decode", "fib_attn_dense_fwd_workspace_size", "fib_attn_dense_fwd",
    "fib_attn_debug_fill_shared", "fib_attn_bwd_prepared",
]

_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_vp = ctypes.c_void_p
_i = ctypes.c_int

_SIGS = {
    "fib_attn_error_string": (ctypes.c_char_p, [_i]),
    "fib_attn_base": (_i, [_i, _i, _i32p, _i, ctypes.POINTER(_i)]),
    "fib_attn_schedule": (_i, [_i, _i, _i, _f64p]),
    "fib_attn_mask_distances": (_i, [_i32p, _i, ctypes.c_double, _i, _i, _i32p, _i, ctypes.POINTER(_i)]),
    "fib_attn_interp_rungs": (_i, [_i32p, _i, ctypes.c_double, _i, _i, _i32p, _i32p, _f32p, _i,
                                   ctypes.POINTER(_i)]),
    "fib_attn_plan_create": (_i, [ctypes.POINTER(_vp), _i, _i32p, _i, _f64p, _i, _i, _i, _i, _i,
                                  ctypes.c_double]),
    "fib_attn_plan_destroy": (_i, [_vp]),
    "fib_attn_plan_distances": (_i, [_vp, _i, _i, _i32p, _i, ctypes.POINTER(_i)]),
    "fib_attn_fwd_workspace_size": (ctypes.c_size_t, [_vp, _i, _i, _i, _i]),
    "fib_attn_fwd_prepare_kv": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "fib_attn_fwd_attend": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp, ctypes.c_size_t, _vp, _vp, _vp, _vp]),
    "fib_attn_fwd": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t,
                          _vp]),
    "fib_attn_bwd_workspace_size": (ctypes.c_size_t, [_vp, _i, _i, _i]),
    "fib_attn_bwd": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                          _vp, _vp, ctypes.c_size_t, _vp]),
    "fib_attn_debug_indices": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp]),
    "fib_attn_last_device_status": (_i, [_vp]),
    "fib_attn_debug_fill_shared": (_i, [ctypes.c_uint32, _vp]),
    "fib_attn_plan_set_debug": (_i, [_vp, _i, ctypes.c_longlong]),
    "fib_attn_decode": (_i, [_vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "fib_attn_dense_fwd_workspace_size": (ctypes.c_size_t, [_vp, _i, _i, _i, _i]),
    "fib_attn_dense_fwd": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "fib_attn_bwd_noalloc": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                  _vp, _vp, _vp, _vp]),
    "fib_attn_bwd_prepared": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp, ctypes.c_size_t, _vp, _vp, _vp, _vp,
                                   _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
}

_lib = None


class FibAttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {error_string(code)} (status {code})")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load libfibattn.so (built in-tree by build.py); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() first")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def error_string(code: int) -> str:
    return lib().fib_attn_error_string(int(code)).decode()


def _check(fn: str, code: int):
    if code != FIB_OK:
        raise FibAttnError(fn, code)


def _arr(ctype, values):
    a = (ctype * max(1, len(values)))(*values)
    return a


# ----------------------------------------------------------------------- host-only planner
def fib_attn_base(base_kind: int, N: int = 2) -> list[int]:
    n = _i(0)
    _check("fib_attn_base", lib().fib_attn_base(base_kind, N, None, 0, ctypes.byref(n)))
    out = (ctypes.c_int32 * max(1, n.value))()
    _check("fib_attn_base", lib().fib_attn_base(base_kind, N, out, n.value, ctypes.byref(n)))
    return list(out[: n.value])


def fib_attn_schedule(kind: int, n_layers: int, stride: int = 7) -> list[float]:
    out = (ctypes.c_double * n_layers)()
    _check("fib_attn_schedule", lib().fib_attn_schedule(kind, n_layers, stride, out))
    return list(out)


def fib_attn_mask_distances(base, alpha: float, W: int, N: int) -> list[int]:
    b = _arr(ctypes.c_int32, list(base))
    cap = FIB_MAX_RUNGS * 4
    out = (ctypes.c_int32 * cap)()
    n = _i(0)
    _check("fib_attn_mask_distances", lib().fib_attn_mask_distances(
        b, len(base), float(alpha), W, N, out, cap, ctypes.byref(n)))
    return list(out[: min(n.value, cap)])


def fib_attn_interp_rungs(base, alpha: float, W: int, N: int):
    b = _arr(ctypes.c_int32, list(base))
    cap = FIB_MAX_RUNGS * 4
    f, lo, w = (ctypes.c_int32 * cap)(), (ctypes.c_int32 * cap)(), (ctypes.c_float * cap)()
    n = _i(0)
    _check("fib_attn_interp_rungs", lib().fib_attn_interp_rungs(
        b, len(base), float(alpha), W, N, f, lo, w, cap, ctypes.byref(n)))
    return [(f[r], lo[r], w[r]) for r in range(min(n.value, cap))]


# ----------------------------------------------------------------------------- plan
class Plan:
    """Owns a fib_attn_plan_t (destroyed with the object)."""

    def __init__(self, handle, n_layers, W, N_max, mode, device):
        self.handle, self.n_layers, self.W, self.N_max, self.mode = handle, n_layers, W, N_max, mode
        self.device = device

    def close(self):
        if self.handle:
            lib().fib_attn_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fib_attn_plan_create(base_kind: int, alpha, W: int, N_max: int, mode: int,
                         custom_base=None, D: int = 64, rope_base: float = 10000.0) -> Plan:
    alpha = [float(a) for a in alpha]
    cb = list(custom_base) if custom_base is not None else []
    h = _vp()
    _check("fib_attn_plan_create", lib().fib_attn_plan_create(
        ctypes.byref(h), base_kind, _arr(ctypes.c_int32, cb) if cb else None, len(cb),
        _arr(ctypes.c_double, alpha), len(alpha), W, N_max, D, mode, float(rope_base)))
    return Plan(h, len(alpha), W, N_max, mode, torch.cuda.current_device())


def fib_attn_plan_distances(plan: Plan, layer: int, N: int) -> list[int]:
    out = (ctypes.c_int32 * FIB_MAX_RUNGS)()
    n = _i(0)
    _check("fib_attn_plan_distances", lib().fib_attn_plan_distances(
        plan.handle, layer, N, out, FIB_MAX_RUNGS, ctypes.byref(n)))
    return list(out[: n.value])


# ---------------------------------------------------------------------------- device ops
_DT = {torch.float32: FIB_DTYPE_F32, torch.bfloat16: FIB_DTYPE_BF16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _shape(q):
    if q.dim() != 4 or q.shape[-1] != FIB_HEAD_DIM:
        raise ValueError("expected [B, H, N, 64]")
    for t in (q,):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
    return q.shape[0], q.shape[1], q.shape[2]


def _same(q, *ts):
    for t in ts:
        if t is not None and (t.shape != q.shape or t.dtype != q.dtype or not t.is_cuda
                              or not t.is_contiguous()):
            raise ValueError("q/k/v/o/dO/dq/dk/dv must share shape, dtype and be contiguous CUDA")


def fib_attn_fwd_workspace_size(plan: Plan, B: int, H: int, N: int, dtype) -> int:
    return int(lib().fib_attn_fwd_workspace_size(plan.handle, B, H, N, _DT.get(dtype, dtype)))


def fib_attn_fwd(plan: Plan, layer: int, q, k, v, o=None, lse=None, alpha_dev=None,
                 want_lse: bool = True, workspace=None, stream=None):
    """Returns (o, lse).  o/lse and the workspace are allocated (by torch) when not given."""
    B, H, N = _shape(q)
    _same(q, k, v, o)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    need = fib_attn_fwd_workspace_size(plan, B, H, N, q.dtype)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("fib_attn_fwd", lib().fib_attn_fwd(
        plan.handle, layer, B, H, N, _DT[q.dtype], _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
        _ptr(alpha_dev), _ptr(workspace), ws_bytes, _stream(stream)))
    return o, lse


def fib_attn_fwd_prepare_kv(plan: Plan, k, v, workspace=None, stream=None):
    """K rotated at its own positions and V, as float16, into a workspace (allocated by torch
    when not given), for fib_attn_fwd_attend; returns the workspace."""
    B, H, N = _shape(k)
    _same(k, v)
    need = fib_attn_fwd_workspace_size(plan, B, H, N, k.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=k.device)
    _check("fib_attn_fwd_prepare_kv", lib().fib_attn_fwd_prepare_kv(
        plan.handle, B, H, N, _DT[k.dtype], _ptr(k), _ptr(v), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return workspace


def fib_attn_fwd_attend(plan: Plan, layer: int, q, workspace, o=None, lse=None, alpha_dev=None,
                        want_lse: bool = True, stream=None):
    """Attention of q against a workspace filled by fib_attn_fwd_prepare_kv; returns (o, lse)."""
    B, H, N = _shape(q)
    _same(q, o)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check("fib_attn_fwd_attend", lib().fib_attn_fwd_attend(
        plan.handle, layer, B, H, N, _DT[q.dtype], _ptr(q), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(o), _ptr(lse), _ptr(alpha_dev),
        _stream(stream)))
    return o, lse


def fib_attn_dense_fwd(plan: Plan, q, k, v, o=None, lse=None, want_lse: bool = True, workspace=None,
                       stream=None):
    """Dense causal attention with the plan's RoPE (bf16); returns (o, lse)."""
    B, H, N = _shape(q)
    _same(q, k, v, o)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    need = int(lib().fib_attn_dense_fwd_workspace_size(plan.handle, B, H, N, _DT[q.dtype]))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _check("fib_attn_dense_fwd", lib().fib_attn_dense_fwd(
        plan.handle, B, H, N, _DT[q.dtype], _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return o, lse


def fib_attn_decode(plan: Plan, layer: int, pos: int, q, k_cache, v_cache, o=None, lse=None,
                    alpha_dev=None, want_lse: bool = True, stream=None):
    """One token at position pos: q [B, H, 64], caches [B, H, N, 64]; returns (o, lse)."""
    if q.dim() != 3 or q.shape[-1] != FIB_HEAD_DIM or not q.is_cuda or not q.is_contiguous():
        raise ValueError("q must be a contiguous CUDA [B, H, 64] tensor")
    B, H, N = _shape(k_cache)
    _same(k_cache, v_cache)
    if q.shape[:2] != k_cache.shape[:2] or q.dtype != k_cache.dtype:
        raise ValueError("q and the caches must share B, H and dtype")
    o = torch.empty_like(q) if o is None else o
    if lse is None and want_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    _check("fib_attn_decode", lib().fib_attn_decode(
        plan.handle, layer, B, H, N, pos, _DT[q.dtype], _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(o), _ptr(lse), _ptr(alpha_dev), _stream(stream)))
    return o, lse


def fib_attn_bwd_workspace_size(plan: Plan, B: int, H: int, N: int) -> int:
    return int(lib().fib_attn_bwd_workspace_size(plan.handle, B, H, N))


def fib_attn_bwd(plan: Plan, layer: int, q, k, v, o, lse, dO, dq=None, dk=None, dv=None,
                 dalpha=None, alpha_dev=None, workspace=None, stream=None):
    """Returns (dq, dk, dv, dalpha[1])."""
    B, H, N = _shape(q)
    _same(q, k, v, o, dO, dq, dk, dv)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    if dalpha is None:
        dalpha = torch.empty(1, dtype=torch.float32, device=q.device)
    need = fib_attn_bwd_workspace_size(plan, B, H, N)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check("fib_attn_bwd", lib().fib_attn_bwd(
        plan.handle, layer, B, H, N, _DT[q.dtype], _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
        _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dalpha), _ptr(alpha_dev), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return dq, dk, dv, dalpha


def fib_attn_bwd_prepared(plan: Plan, layer: int, q, kv_prepared, o, lse, dO, dq=None, dk=None, dv=None,
                          dalpha=None, alpha_dev=None, workspace=None, stream=None):
    """Backward from the forward's prepared K'/V' rows (the uint8 workspace that
    fib_attn_fwd or fib_attn_fwd_prepare_kv filled for this layer's k and v): returns
    (dq, dk, dv, dalpha[1]), those of fib_attn_bwd up to the float16 rounding of K'."""
    B, H, N = _shape(q)
    _same(q, o, dO, dq, dk, dv)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    if dalpha is None:
        dalpha = torch.empty(1, dtype=torch.float32, device=q.device)
    need = fib_attn_bwd_workspace_size(plan, B, H, N)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check("fib_attn_bwd_prepared", lib().fib_attn_bwd_prepared(
        plan.handle, layer, B, H, N, _DT[q.dtype], _ptr(q), _ptr(kv_prepared),
        kv_prepared.numel() * kv_prepared.element_size(), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
        _ptr(dv), _ptr(dalpha), _ptr(alpha_dev), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return dq, dk, dv, dalpha


def fib_attn_bwd_noalloc(plan: Plan, layer: int, q, k, v, o, lse, dO, dq, dk, dv, dalpha,
                         alpha_dev=None, stream=None):
    """Backward into caller-provided dq, dk, dv, dalpha[1] with the library's fixed scratch
    array: no workspace argument and nothing allocated (for callers that may not allocate)."""
    B, H, N = _shape(q)
    _same(q, k, v, o, dO, dq, dk, dv)
    _check("fib_attn_bwd_noalloc", lib().fib_attn_bwd_noalloc(
        plan.handle, layer, B, H, N, _DT[q.dtype], _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
        _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dalpha), _ptr(alpha_dev), _stream(stream)))
    return dq, dk, dv, dalpha


def fib_attn_debug_indices(plan: Plan, layer: int, N: int, i_begin: int, i_end: int,
                           alpha_dev=None, stream=None):
    """Returns (rows int32 [(i_end-i_begin), W + 32] with -1 padding, w float32 [32])."""
    out = torch.empty((i_end - i_begin, plan.W + FIB_MAX_RUNGS), dtype=torch.int32, device="cuda")
    w = torch.empty(FIB_MAX_RUNGS, dtype=torch.float32, device="cuda")
    _check("fib_attn_debug_indices", lib().fib_attn_debug_indices(
        plan.handle, layer, N, i_begin, i_end, _ptr(out), _ptr(w), _ptr(alpha_dev), _stream(stream)))
    return out, w


def fib_attn_plan_set_debug(plan: Plan, skip_first_rung_copy: bool, wait_ns: int,
                            corrupt_table: bool = False):
    flags = (FIB_DEBUG_SKIP_COPY if skip_first_rung_copy else 0) | \
        (FIB_DEBUG_CORRUPT_TABLE if corrupt_table else 0)
    _check("fib_attn_plan_set_debug", lib().fib_attn_plan_set_debug(plan.handle, flags, int(wait_ns)))


def fib_attn_debug_fill_shared(pattern: int, stream=None):
    """Test hook: fill every SM's shared memory with a 32-bit pattern (stale contents for the
    kernels launched next)."""
    _check("fib_attn_debug_fill_shared", lib().fib_attn_debug_fill_shared(int(pattern) & 0xffffffff, _stream(stream)))


def fib_attn_last_device_status(plan: Plan) -> int:
    return int(lib().fib_attn_last_device_status(plan.handle))
