"""Thin ctypes binding over libdilution_attn.so (argument marshalling only).

Every function here has the name of the C entry point it forwards to (see
``include/dilution_attn.h``).  Tensors are torch tensors used only as device
memory; every step of the computation runs in the library's CUDA kernels.
The library is loaded on first use; if it cannot be loaded the call raises.
There is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import build as _build

DA_OK, DA_ERR_INVALID, DA_ERR_UNSUPPORTED, DA_ERR_CUDA, DA_ERR_TIMEOUT, DA_ERR_WORKSPACE = range(6)
DA_F32, DA_BF16 = 0, 1
DA_FLAG_EARLIER_DEMAND_ONLY = 1
DA_FLAG_KEEP_FOR_BACKWARD = 2
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dilution_attn.h")

_lib = None
_lock = threading.Lock()

_c_void_p = ctypes.c_void_p
_c_int = ctypes.c_int
_c_float = ctypes.c_float
_c_size_t = ctypes.c_size_t

_SIGNATURES = {
    "dilution_attn_status_string": (ctypes.c_char_p, [_c_int]),
    "dilution_attn_version": (_c_int, []),
    "dilution_attn_fwd_workspace_size": (_c_size_t, [_c_int] * 5),
    "dilution_attn_fwd": (_c_int, [_c_void_p] * 7 + [_c_int] * 4 + [_c_float, _c_float, _c_int, _c_void_p,
                                                                        _c_size_t, _c_void_p]),
    "dilution_attn_fwd_with_events": (_c_int, [_c_void_p] * 7 + [_c_int] * 4 + [_c_float, _c_float, _c_int,
                                                                                    _c_void_p, _c_size_t, _c_void_p,
                                                                                    _c_void_p]),
    "dilution_attn_fwd_ex": (_c_int, [_c_void_p] * 7 + [_c_int] * 4 + [_c_float, _c_void_p, _c_float, _c_int, _c_int,
                                                                       _c_void_p, _c_size_t, _c_void_p, _c_void_p]),
    "dilution_attn_bwd_workspace_size": (_c_size_t, [_c_int] * 5),
    "dilution_attn_bwd": (_c_int, [_c_void_p] * 8 + [_c_int] * 4 + [_c_float, _c_float, _c_int, _c_void_p, _c_size_t,
                                                                        _c_void_p]),
    "dilution_attn_bwd_ex": (_c_int, [_c_void_p] * 8 + [_c_int] * 4 + [_c_float, _c_void_p, _c_float, _c_int, _c_int,
                                                                       _c_void_p, _c_size_t, _c_void_p]),
    "dilution_attn_decode_workspace_size": (_c_size_t, [_c_int] * 4),
    "dilution_attn_decode_step": (_c_int, [_c_void_p] * 6 + [_c_int, _c_int, _c_void_p] + [_c_int] * 3 +
                                  [_c_float, _c_float, _c_int, _c_void_p, _c_size_t, _c_void_p]),
    "dilution_attn_decode_step_ex": (_c_int, [_c_void_p] * 6 + [_c_int, _c_int, _c_void_p] + [_c_int] * 3 +
                                     [_c_float, _c_void_p, _c_float, _c_int, _c_int, _c_void_p, _c_size_t,
                                      _c_void_p]),
    "dilution_attn_decode_step_noalloc": (_c_int, [_c_void_p] * 6 + [_c_int, _c_int, _c_void_p] + [_c_int] * 3 +
                                          [_c_float, _c_float, _c_int, _c_void_p]),
    "dilution_attn_decode_noalloc_scratch_bytes": (_c_size_t, []),
    "dilution_attn_decode_noalloc_get_error": (_c_int, [_c_void_p]),
    "dilution_attn_debug_decode_stall": (_c_int, [_c_void_p] * 6 + [_c_int, _c_int, _c_void_p] + [_c_int] * 3 +
                                         [_c_float, _c_float, _c_int, _c_void_p, _c_size_t, _c_void_p, _c_int, _c_int,
                                          ctypes.c_longlong]),
    "dilution_attn_get_error": (_c_int, [_c_void_p, _c_void_p]),
    "dilution_attn_debug_last_timeout": (_c_int, [_c_void_p, _c_void_p]),
    "dilution_attn_debug_tile_schedule": (_c_int, [_c_int, _c_int, _c_int, _c_void_p, _c_size_t]),
    "dilution_attn_debug_tile_mask": (_c_int, [_c_int, _c_int, _c_int, _c_void_p]),
}


class DilutionAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)}")
        self.status = status


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load (building first if needed) and return the ctypes library handle."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and not os.path.exists(path):
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libdilution_attn.so not found at {path}; run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def header_functions() -> list[str]:
    """Names of every function the public header declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dilution_attn_\w+)\s*\(", text)))


def status_string(status: int) -> str:
    return load().dilution_attn_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != DA_OK:
        raise DilutionAttnError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return DA_F32
    if t.dtype == torch.bfloat16:
        return DA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")


def _need(t, name, shape=None, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        # the library launches on the current device and takes its per-device
        # set-up (and the no-alloc scratch address) from it
        raise ValueError(f"{name} is on {t.device} but the current device is cuda:{torch.cuda.current_device()}; "
                         f"call inside torch.cuda.device({t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")


# --------------------------------------------------------------------------- forward
def dilution_attn_fwd_workspace_size(B: int, H: int, T: int, d: int, dtype: int) -> int:
    return int(load().dilution_attn_fwd_workspace_size(B, H, T, d, dtype))


def dilution_attn_fwd(q, k, v, out=None, lse2_out=None, rowsum_out=None, demand_out=None, *,
                      tau: float = 1.0, eps: float = 1e-6, workspace=None, stream=None, check: bool = True):
    """Forward over [B, H, T, d] q/k/v (float32 or bfloat16, contiguous, CUDA).

    Returns ``out`` (allocated if not given).  Optional fp32 [B, H, T] side
    outputs are filled when passed.  ``workspace`` (uint8 CUDA tensor) is
    allocated when omitted.
    """
    return dilution_attn_fwd_with_events(q, k, v, out, lse2_out, rowsum_out, demand_out, tau=tau, eps=eps,
                                         workspace=workspace, stream=stream, check=check, events=None)


def _event_handle(e):
    if e is None:
        return None
    if e.cuda_event == 0:   # torch creates the CUDA event lazily, on first record
        e.record()
    return e.cuda_event


def _fwd_prepare(q, k, v, out, lse2_out, rowsum_out, demand_out, workspace, flags=0):
    _need(q, "q")
    B, H, T, d = q.shape
    _need(k, "k", q.shape, q.dtype)
    _need(v, "v", q.shape, q.dtype)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.shape, q.dtype)
    for name, t in (("lse2_out", lse2_out), ("rowsum_out", rowsum_out), ("demand_out", demand_out)):
        if t is not None:
            _need(t, name, (B, H, T), torch.float32)
    dt = _dtype_code(q)
    need = (dilution_attn_bwd_workspace_size(B, H, T, d, dt) if flags & DA_FLAG_KEEP_FOR_BACKWARD
            else dilution_attn_fwd_workspace_size(B, H, T, d, dt))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    return out, workspace, dt


def _events_array(events):
    if events is None:
        return None
    return (ctypes.c_void_p * 4)(*[_event_handle(e) for e in events])


def _tau_bh_ptr(tau_bh, B, H):
    """Marshal an optional per-(batch, head) multiplier tensor: fp32 CUDA, B*H elements."""
    if tau_bh is None:
        return None
    _need(tau_bh, "tau_bh", None, torch.float32)
    if tau_bh.numel() != B * H:
        raise ValueError(f"tau_bh has {tau_bh.numel()} elements, expected B*H = {B * H}")
    return _ptr(tau_bh)


def dilution_attn_fwd_with_events(q, k, v, out=None, lse2_out=None, rowsum_out=None, demand_out=None, *,
                                  tau: float = 1.0, eps: float = 1e-6, workspace=None, stream=None,
                                  check: bool = True, events=None):
    """dilution_attn_fwd that also records up to four torch.cuda.Event
    (timing-enabled) on the stream: before row statistics, before the sweep,
    before finalize, after finalize."""
    lib = load()
    out, workspace, dt = _fwd_prepare(q, k, v, out, lse2_out, rowsum_out, demand_out, workspace)
    B, H, T, d = q.shape
    st = lib.dilution_attn_fwd_with_events(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse2_out), _ptr(rowsum_out),
                                           _ptr(demand_out), B, H, T, d, float(tau), float(eps), dt,
                                           _ptr(workspace), workspace.numel(), _stream_handle(stream),
                                           _events_array(events))
    if check:
        _check(st, "dilution_attn_fwd")
    return out


def dilution_attn_fwd_ex(q, k, v, out=None, lse2_out=None, rowsum_out=None, demand_out=None, *,
                         tau: float = 1.0, tau_bh=None, eps: float = 1e-6, flags: int = 0, workspace=None,
                         stream=None, check: bool = True, events=None):
    """Forward with a per-(batch, head) multiplier tensor ``tau_bh`` (fp32 CUDA,
    B*H elements, index b*H + h; replaces ``tau``) and ``flags``
    (``DA_FLAG_EARLIER_DEMAND_ONLY``, ``DA_FLAG_KEEP_FOR_BACKWARD``: pass the
    same ``workspace`` to ``dilution_attn_bwd_ex`` with the same flags; it is
    allocated backward-sized when omitted)."""
    lib = load()
    out, workspace, dt = _fwd_prepare(q, k, v, out, lse2_out, rowsum_out, demand_out, workspace, int(flags))
    B, H, T, d = q.shape
    st = lib.dilution_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse2_out), _ptr(rowsum_out),
                                  _ptr(demand_out), B, H, T, d, float(tau), _tau_bh_ptr(tau_bh, B, H), float(eps),
                                  int(flags), dt, _ptr(workspace), workspace.numel(), _stream_handle(stream),
                                  _events_array(events))
    if check:
        _check(st, "dilution_attn_fwd_ex")
    return out


# -------------------------------------------------------------------------- backward
def dilution_attn_bwd_workspace_size(B: int, H: int, T: int, d: int, dtype: int) -> int:
    return int(load().dilution_attn_bwd_workspace_size(B, H, T, d, dtype))


def _bwd_prepare(q, k, v, dout, lse2, dq, dk, dv, workspace):
    _need(q, "q")
    B, H, T, d = q.shape
    for name, t in (("k", k), ("v", v), ("dout", dout)):
        _need(t, name, q.shape, q.dtype)
    _need(lse2, "lse2", (B, H, T), torch.float32)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _need(t, name, q.shape, q.dtype)
    dt = _dtype_code(q)
    if workspace is None:
        workspace = torch.empty(max(dilution_attn_bwd_workspace_size(B, H, T, d, dt), 256), dtype=torch.uint8,
                                device=q.device)
    return dq, dk, dv, workspace, dt


def dilution_attn_bwd(q, k, v, dout, lse2, dq=None, dk=None, dv=None, *, tau: float = 1.0, eps: float = 1e-6,
                      workspace=None, stream=None, check: bool = True):
    """Gradients (dq, dk, dv) of sum(dout * out); lse2 is the forward's lse2_out."""
    lib = load()
    dq, dk, dv, workspace, dt = _bwd_prepare(q, k, v, dout, lse2, dq, dk, dv, workspace)
    B, H, T, d = q.shape
    st = lib.dilution_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse2), _ptr(dq), _ptr(dk), _ptr(dv), B,
                               H, T, d, float(tau), float(eps), dt, _ptr(workspace), workspace.numel(),
                               _stream_handle(stream))
    if check:
        _check(st, "dilution_attn_bwd")
    return dq, dk, dv


def dilution_attn_bwd_ex(q, k, v, dout, lse2, dq=None, dk=None, dv=None, *, tau: float = 1.0, tau_bh=None,
                         eps: float = 1e-6, flags: int = 0, workspace=None, stream=None, check: bool = True):
    """dilution_attn_bwd with the ``tau_bh`` and ``flags`` of the matching forward."""
    lib = load()
    dq, dk, dv, workspace, dt = _bwd_prepare(q, k, v, dout, lse2, dq, dk, dv, workspace)
    B, H, T, d = q.shape
    st = lib.dilution_attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse2), _ptr(dq), _ptr(dk), _ptr(dv),
                                  B, H, T, d, float(tau), _tau_bh_ptr(tau_bh, B, H), float(eps), int(flags), dt,
                                  _ptr(workspace), workspace.numel(), _stream_handle(stream))
    if check:
        _check(st, "dilution_attn_bwd_ex")
    return dq, dk, dv


# ---------------------------------------------------------------------------- decode
def dilution_attn_decode_workspace_size(B: int, H: int, T_cap: int, d: int) -> int:
    return int(load().dilution_attn_decode_workspace_size(B, H, T_cap, d))


def _decode_prepare(q_new, k_new, v_new, k_cache, v_cache, demand, out):
    _need(q_new, "q_new")
    B, H, d = q_new.shape
    _need(k_new, "k_new", q_new.shape, q_new.dtype)
    _need(v_new, "v_new", q_new.shape, q_new.dtype)
    _need(k_cache, "k_cache", None, q_new.dtype)
    T_cap = k_cache.shape[2]
    _need(k_cache, "k_cache", (B, H, T_cap, d))
    _need(v_cache, "v_cache", (B, H, T_cap, d), q_new.dtype)
    _need(demand, "demand", (B, H, T_cap), torch.float32)
    if out is None:
        out = torch.empty_like(q_new)
    _need(out, "out", q_new.shape, q_new.dtype)
    return out, T_cap


def dilution_attn_decode_step(q_new, k_new, v_new, k_cache, v_cache, demand, n_ctx: int, out=None, *,
                              tau: float = 1.0, eps: float = 1e-6, workspace=None, stream=None,
                              check: bool = True):
    """One cached decode step; caches [B, H, T_cap, d], demand [B, H, T_cap] fp32.

    Appends k_new/v_new at position n_ctx, updates ``demand`` in place and
    returns ``out`` [B, H, d].
    """
    lib = load()
    out, T_cap = _decode_prepare(q_new, k_new, v_new, k_cache, v_cache, demand, out)
    B, H, d = q_new.shape
    if workspace is None:
        workspace = torch.empty(max(dilution_attn_decode_workspace_size(B, H, T_cap, d), 256), dtype=torch.uint8,
                                device=q_new.device)
    st = lib.dilution_attn_decode_step(_ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(demand), int(n_ctx), T_cap, _ptr(out), B, H, d, float(tau), float(eps),
                                       _dtype_code(q_new), _ptr(workspace), workspace.numel(),
                                       _stream_handle(stream))
    if check:
        _check(st, "dilution_attn_decode_step")
    return out


def dilution_attn_decode_step_ex(q_new, k_new, v_new, k_cache, v_cache, demand, n_ctx: int, out=None, *,
                                 tau: float = 1.0, tau_bh=None, eps: float = 1e-6, flags: int = 0, workspace=None,
                                 stream=None, check: bool = True):
    """dilution_attn_decode_step with ``tau_bh`` and ``flags`` (see dilution_attn_fwd_ex)."""
    lib = load()
    out, T_cap = _decode_prepare(q_new, k_new, v_new, k_cache, v_cache, demand, out)
    B, H, d = q_new.shape
    if workspace is None:
        workspace = torch.empty(max(dilution_attn_decode_workspace_size(B, H, T_cap, d), 256), dtype=torch.uint8,
                                device=q_new.device)
    st = lib.dilution_attn_decode_step_ex(_ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(demand), int(n_ctx), T_cap, _ptr(out), B, H, d, float(tau),
                                          _tau_bh_ptr(tau_bh, B, H), float(eps), int(flags), _dtype_code(q_new),
                                          _ptr(workspace), workspace.numel(), _stream_handle(stream))
    if check:
        _check(st, "dilution_attn_decode_step_ex")
    return out


def dilution_attn_decode_step_noalloc(q_new, k_new, v_new, k_cache, v_cache, demand, n_ctx: int, out=None, *,
                                      tau: float = 1.0, eps: float = 1e-6, stream=None, check: bool = True):
    """dilution_attn_decode_step with the library's fixed scratch array instead of a workspace."""
    lib = load()
    out, T_cap = _decode_prepare(q_new, k_new, v_new, k_cache, v_cache, demand, out)
    B, H, d = q_new.shape
    st = lib.dilution_attn_decode_step_noalloc(_ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                               _ptr(demand), int(n_ctx), T_cap, _ptr(out), B, H, d, float(tau),
                                               float(eps), _dtype_code(q_new), _stream_handle(stream))
    if check:
        _check(st, "dilution_attn_decode_step_noalloc")
    return out


def dilution_attn_decode_noalloc_scratch_bytes() -> int:
    return int(load().dilution_attn_decode_noalloc_scratch_bytes())


def dilution_attn_decode_noalloc_get_error(stream=None) -> int:
    """Status of the no-alloc decode step's fixed array on the current
    device (synchronises the stream, then reads and clears the word)."""
    return int(load().dilution_attn_decode_noalloc_get_error(_stream_handle(stream)))


def dilution_attn_debug_decode_stall(q_new, k_new, v_new, k_cache, v_cache, demand, n_ctx: int, out=None, *,
                                     tau: float = 1.0, eps: float = 1e-6, workspace=None, stream=None,
                                     stall_chunk: int = 0, stall_bh: int = 0, wait_limit_ns: int = 2_000_000):
    """Test hook of the bounded waits: a decode step in which one block's ring
    slot is never handed back (see the header).  Returns (status, out); the
    kernel-side outcome is read with dilution_attn_debug_last_timeout /
    dilution_attn_get_error on ``workspace``."""
    lib = load()
    out, T_cap = _decode_prepare(q_new, k_new, v_new, k_cache, v_cache, demand, out)
    B, H, d = q_new.shape
    if workspace is None:
        workspace = torch.empty(max(dilution_attn_decode_workspace_size(B, H, T_cap, d), 256), dtype=torch.uint8,
                                device=q_new.device)
    st = lib.dilution_attn_debug_decode_stall(_ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                              _ptr(demand), int(n_ctx), T_cap, _ptr(out), B, H, d, float(tau),
                                              float(eps), _dtype_code(q_new), _ptr(workspace), workspace.numel(),
                                              _stream_handle(stream), int(stall_chunk), int(stall_bh),
                                              int(wait_limit_ns))
    return int(st), out


# ----------------------------------------------------------------------------- misc
def dilution_attn_get_error(workspace, stream=None) -> int:
    return int(load().dilution_attn_get_error(_ptr(workspace), _stream_handle(stream)))


def dilution_attn_status_string(status: int) -> str:
    return status_string(status)


def dilution_attn_version() -> int:
    return int(load().dilution_attn_version())


def dilution_attn_debug_last_timeout(workspace):
    """(status, mbarrier shared-memory offset, block, thread) of the workspace's status block."""
    import numpy as np
    buf = np.zeros(4, dtype=np.int32)
    _check(load().dilution_attn_debug_last_timeout(_ptr(workspace), buf.ctypes.data_as(ctypes.c_void_p)),
           "dilution_attn_debug_last_timeout")
    return tuple(int(x) for x in buf)


def dilution_attn_debug_tile_schedule(BH: int, T: int, kernel: int):
    """[n_ctas, 4] int32 array: (head, first query tile, query tiles, first key)."""
    import numpy as np
    lib = load()
    n = lib.dilution_attn_debug_tile_schedule(BH, T, kernel, None, 0)
    n = -n if n < 0 else n
    buf = np.zeros((max(n, 1), 4), dtype=np.int32)
    got = lib.dilution_attn_debug_tile_schedule(BH, T, kernel, buf.ctypes.data_as(ctypes.c_void_p), buf.size)
    if got < 0:
        raise RuntimeError("tile schedule export failed")
    return buf[:got]


def dilution_attn_debug_tile_mask(T: int, qt: int, kt: int):
    import numpy as np
    buf = np.zeros((128, 128), dtype=np.uint8)
    _check(load().dilution_attn_debug_tile_mask(T, qt, kt, buf.ctypes.data_as(ctypes.c_void_p)),
           "dilution_attn_debug_tile_mask")
    return buf
