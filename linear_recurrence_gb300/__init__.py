"""Selective-scan forward and pscan on GB300 (sm_103a): the Python binding.

The computation lives in ``libsscan.so`` (hand-written CUDA kernels behind
the C ABI of ``include/sscan.h``).  This module only checks tensor shapes,
dtypes and devices, allocates outputs with torch, and passes raw pointers and
the current CUDA stream through ctypes.  There is no fallback: if the library
is missing or fails to load, every call raises.

    y, h_last = sscan_fwd(u, delta, A, B, C, D=None, h0=None)
    h = pscan(a, b, h0=None)

Shapes: u, delta [batch, dim, L] (float32 or bfloat16); A [dim, N] float32;
B, C [batch, N, L] (same dtype as u); D [dim] float32; h0 [batch, dim, N]
float32.  Returns y [batch, dim, L] in the I/O dtype and the final state
[batch, dim, N] float32.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from ._build import LIB as LIB_PATH

SSCAN_OK, SSCAN_ERR_INVALID, SSCAN_ERR_CUDA, SSCAN_ERR_TIMEOUT = 0, 1, 2, 3
SSCAN_F32, SSCAN_BF16 = 0, 1
SSCAN_DELTA_SOFTPLUS, SSCAN_ZOH = 1, 2

_vp, _fp, _i64, _int = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
_lock = threading.Lock()
_lib = None

# name -> (restype, argtypes): every symbol include/sscan.h declares
SIGNATURES = {
    "sscan_fwd": (_int, [_vp, _vp, _fp, _vp, _vp, _fp, _fp, _vp, _fp,
                         _i64, _i64, _i64, _i64, _int, _vp]),
    "sscan_fwd_ex": (_int, [_vp, _vp, _fp, _vp, _vp, _fp, _fp, _vp, _fp,
                            _i64, _i64, _i64, _i64, _int, _int, _int, _vp]),
    "sscan_fwd_fused": (_int, [_vp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _fp, _vp, _fp,
                               _i64, _i64, _i64, _i64, _int, _int, _int, _int, _vp]),
    "sscan_fwd_noalloc": (_int, [_vp, _vp, _fp, _vp, _vp, _fp, _fp, _vp, _fp,
                                 _i64, _i64, _i64, _i64, _int, _int, _vp]),
    "sscan_bwd": (_int, [_vp, _vp, _fp, _vp, _vp, _fp, _fp, _vp, _fp, _vp, _vp, _fp, _fp, _fp, _fp,
                         _fp, _i64, _i64, _i64, _i64, _int, _vp]),
    "sscan_step": (_int, [_vp, _vp, _fp, _vp, _vp, _fp, _fp, _vp, _i64, _i64, _i64, _int, _vp]),
    "pscan": (_int, [_fp, _fp, _fp, _fp, _i64, _i64, _vp]),
    "sscan_status_string": (ctypes.c_char_p, [_int]),
    "sscan_get_last_error": (_int, []),
    "sscan_max_dstate": (_int, []),
    "sscan_debug_expire_next_wait": (None, [ctypes.c_uint]),
    "sscan_debug_expire_next_correction_wait": (None, [ctypes.c_uint]),
    "sscan_probe_ex2": (_int, [_fp, _int, _int, _vp]),
    "sscan_probe_ex2_count": (ctypes.c_longlong, [_int, _int]),
    "sscan_probe_element": (_int, [_fp, _int, _int, _int, _vp]),
    "sscan_probe_element_count": (ctypes.c_longlong, [_int, _int, _int]),
    "sscan_last_launch_count": (_int, []),
    "sscan_last_plan": (ctypes.c_char_p, []),
}


class SscanError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def load_library(path: str | None = None):
    """Load libsscan.so (building it first if this tree has sources but no
    library).  ``path``, else the SSCAN_LIBRARY environment variable, selects
    another build of the library.  Raises if it cannot be loaded."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or os.environ.get("SSCAN_LIBRARY") or LIB_PATH
        if p == LIB_PATH and not os.path.exists(p):
            from ._build import build
            build()
        if not os.path.exists(p):
            raise RuntimeError(f"libsscan.so not found at {p}; run __graft_entry__.build()")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def lib():
    return load_library()


def status_string(status: int) -> str:
    return lib().sscan_status_string(int(status)).decode()


def get_last_error() -> int:
    return int(lib().sscan_get_last_error())


def max_dstate() -> int:
    return int(lib().sscan_max_dstate())


def probe_ex2(blocks: int, iters: int, *, sink=None, stream=None) -> int:
    """Launch the exponent-unit throughput probe (see include/sscan.h) on the
    current device; returns the number of exponentials it computes.  Time it
    with CUDA events on ``stream``."""
    if sink is None:
        sink = torch.empty(blocks * 256, dtype=torch.float32, device="cuda")
    rc = lib().sscan_probe_ex2(_ptr(sink), int(blocks), int(iters), _stream_handle(stream))
    if rc != SSCAN_OK:
        raise SscanError(rc, "sscan_probe_ex2")
    return int(lib().sscan_probe_ex2_count(int(blocks), int(iters)))


def probe_element(blocks: int, iters: int, *, shared_rate: bool = False, sink=None, stream=None) -> int:
    """Launch the element-arithmetic throughput probe (see include/sscan.h) on
    the current device; returns the number of elements it computes.  Time it
    with CUDA events on ``stream``."""
    if sink is None:
        sink = torch.empty(blocks * 256, dtype=torch.float32, device="cuda")
    rc = lib().sscan_probe_element(_ptr(sink), int(blocks), int(iters), int(bool(shared_rate)),
                                   _stream_handle(stream))
    if rc != SSCAN_OK:
        raise SscanError(rc, "sscan_probe_element")
    return int(lib().sscan_probe_element_count(int(blocks), int(iters), int(bool(shared_rate))))


def debug_expire_next_wait(wait_limit_us: int) -> None:
    """Test aid: make the bounded waits of this thread's next forward call
    run out after ``wait_limit_us`` (see include/sscan.h)."""
    lib().sscan_debug_expire_next_wait(int(wait_limit_us))


def debug_expire_next_correction_wait(wait_limit_us: int) -> None:
    """Test aid: make the bounded waits of the carry correction of this
    thread's next forward call run out after ``wait_limit_us`` (see
    include/sscan.h)."""
    lib().sscan_debug_expire_next_correction_wait(int(wait_limit_us))


def last_launch_count() -> int:
    return int(lib().sscan_last_launch_count())


def last_plan() -> str:
    return lib().sscan_last_plan().decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, shape, dtype, device):
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def sscan_fwd(u, delta, A, B, C, D=None, h0=None, *, z=None, delta_bias=None,
              delta_softplus: bool = False, zoh: bool = False, out=None, final_state=None,
              return_final_state: bool = True, segments: int = 0, lanes: int = 0,
              stream=None):
    """Selective-scan forward on the GPU.  See the module docstring.

    Options (all inside the same kernels): ``delta_bias`` [dim] float32 is
    added to delta, ``delta_softplus`` then applies softplus to it, ``zoh``
    uses the zero-order-hold B-bar, and ``z`` [batch, dim, L] (I/O dtype)
    gates the output: out = (y + D*u) * silu(z).

    ``segments`` / ``lanes`` pin the launch plan (0 = automatic); the result is
    the same computation under any plan.  Returns ``(y, final_state)``
    (``final_state`` is None when ``return_final_state`` is False and none was
    passed).
    """
    if u.dim() != 3:
        raise ValueError("u must be [batch, dim, L]")
    batch, dim, L = u.shape
    if A.dim() != 2 or A.shape[0] != dim:
        raise ValueError("A must be [dim, N]")
    N = A.shape[1]
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("sscan_fwd runs on CUDA tensors only")
    io = u.dtype
    if io not in (torch.float32, torch.bfloat16):
        raise ValueError("u must be float32 or bfloat16")
    _check(u, "u", (batch, dim, L), io, dev)
    _check(delta, "delta", (batch, dim, L), io, dev)
    _check(A, "A", (dim, N), torch.float32, dev)
    _check(B, "B", (batch, N, L), io, dev)
    _check(C, "C", (batch, N, L), io, dev)
    if D is not None:
        _check(D, "D", (dim,), torch.float32, dev)
    if h0 is not None:
        _check(h0, "h0", (batch, dim, N), torch.float32, dev)
    if z is not None:
        _check(z, "z", (batch, dim, L), io, dev)
    if delta_bias is not None:
        _check(delta_bias, "delta_bias", (dim,), torch.float32, dev)
    if out is None:
        out = torch.empty((batch, dim, L), dtype=io, device=dev)
    else:
        _check(out, "out", (batch, dim, L), io, dev)
    if final_state is None and return_final_state:
        final_state = torch.empty((batch, dim, N), dtype=torch.float32, device=dev)
    elif final_state is not None:
        _check(final_state, "final_state", (batch, dim, N), torch.float32, dev)
    dtype = SSCAN_F32 if io == torch.float32 else SSCAN_BF16
    flags = (SSCAN_DELTA_SOFTPLUS if delta_softplus else 0) | (SSCAN_ZOH if zoh else 0)
    if z is None and delta_bias is None and flags == 0:
        rc = lib().sscan_fwd_ex(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                _ptr(h0), _ptr(out), _ptr(final_state), batch, dim, L, N,
                                dtype, int(segments), int(lanes), _stream_handle(stream))
    else:
        rc = lib().sscan_fwd_fused(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                   _ptr(z), _ptr(delta_bias), _ptr(h0), _ptr(out),
                                   _ptr(final_state), batch, dim, L, N, dtype, flags,
                                   int(segments), int(lanes), _stream_handle(stream))
    if rc != SSCAN_OK:
        raise SscanError(rc, "sscan_fwd")
    return out, final_state


def sscan_bwd(u, delta, A, B, C, D, h0, dy, dfinal_state=None, *, stream=None):
    """Gradients of :func:`sscan_fwd` (no options) for upstream gradients ``dy``
    [batch, dim, L] (I/O dtype) and ``dfinal_state`` [batch, dim, N] float32
    (None = 0).  Returns a dict with du, ddelta (I/O dtype), dA, dB, dC, dD (None
    when D is None) and dh0 (float32)."""
    if u.dim() != 3:
        raise ValueError("u must be [batch, dim, L]")
    batch, dim, L = u.shape
    if A.dim() != 2 or A.shape[0] != dim:
        raise ValueError("A must be [dim, N]")
    N = A.shape[1]
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("sscan_bwd runs on CUDA tensors only")
    io = u.dtype
    if io not in (torch.float32, torch.bfloat16):
        raise ValueError("u must be float32 or bfloat16")
    for t, name, shape, dt in ((u, "u", (batch, dim, L), io), (delta, "delta", (batch, dim, L), io),
                               (A, "A", (dim, N), torch.float32), (B, "B", (batch, N, L), io),
                               (C, "C", (batch, N, L), io), (dy, "dy", (batch, dim, L), io)):
        _check(t, name, shape, dt, dev)
    if D is not None:
        _check(D, "D", (dim,), torch.float32, dev)
    if h0 is not None:
        _check(h0, "h0", (batch, dim, N), torch.float32, dev)
    if dfinal_state is not None:
        _check(dfinal_state, "dfinal_state", (batch, dim, N), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    g = {"du": torch.empty((batch, dim, L), dtype=io, device=dev),
         "ddelta": torch.empty((batch, dim, L), dtype=io, device=dev),
         "dA": torch.empty((dim, N), **f32), "dB": torch.empty((batch, N, L), **f32),
         "dC": torch.empty((batch, N, L), **f32),
         "dD": None if D is None else torch.empty((dim,), **f32),
         "dh0": torch.empty((batch, dim, N), **f32)}
    dtype = SSCAN_F32 if io == torch.float32 else SSCAN_BF16
    rc = lib().sscan_bwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(h0), _ptr(dy),
                         _ptr(dfinal_state), _ptr(g["du"]), _ptr(g["ddelta"]), _ptr(g["dA"]),
                         _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]), _ptr(g["dh0"]),
                         batch, dim, L, N, dtype, _stream_handle(stream))
    if rc != SSCAN_OK:
        raise SscanError(rc, "sscan_bwd")
    return g


def sscan_step(u, delta, A, B, C, D=None, *, state, out=None, stream=None):
    """One decode step: advances ``state`` [batch, dim, N] (float32, in place)
    by one token and returns y [batch, dim].  u, delta: [batch, dim]; B, C:
    [batch, N] (float32 or bfloat16, like u); A [dim, N] and D [dim] float32."""
    if u.dim() != 2:
        raise ValueError("u must be [batch, dim]")
    batch, dim = u.shape
    if A.dim() != 2 or A.shape[0] != dim:
        raise ValueError("A must be [dim, N]")
    N = A.shape[1]
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("sscan_step runs on CUDA tensors only")
    io = u.dtype
    if io not in (torch.float32, torch.bfloat16):
        raise ValueError("u must be float32 or bfloat16")
    _check(u, "u", (batch, dim), io, dev)
    _check(delta, "delta", (batch, dim), io, dev)
    _check(A, "A", (dim, N), torch.float32, dev)
    _check(B, "B", (batch, N), io, dev)
    _check(C, "C", (batch, N), io, dev)
    if D is not None:
        _check(D, "D", (dim,), torch.float32, dev)
    _check(state, "state", (batch, dim, N), torch.float32, dev)
    if out is None:
        out = torch.empty((batch, dim), dtype=io, device=dev)
    else:
        _check(out, "out", (batch, dim), io, dev)
    dtype = SSCAN_F32 if io == torch.float32 else SSCAN_BF16
    rc = lib().sscan_step(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(state),
                          _ptr(out), batch, dim, N, dtype, _stream_handle(stream))
    if rc != SSCAN_OK:
        raise SscanError(rc, "sscan_step")
    return out


def pscan(a, b, h0=None, *, out=None, stream=None):
    """h[r,t] = a[r,t]*h[r,t-1] + b[r,t] with h[r,-1] = h0[r] (0 if None), on
    float32 CUDA tensors a, b [rows, len].  Returns h [rows, len]."""
    if a.dim() != 2:
        raise ValueError("a must be [rows, len]")
    rows, n = a.shape
    dev = a.device
    if dev.type != "cuda":
        raise ValueError("pscan runs on CUDA tensors only")
    _check(a, "a", (rows, n), torch.float32, dev)
    _check(b, "b", (rows, n), torch.float32, dev)
    if h0 is not None:
        _check(h0, "h0", (rows,), torch.float32, dev)
    if out is None:
        out = torch.empty((rows, n), dtype=torch.float32, device=dev)
    else:
        _check(out, "out", (rows, n), torch.float32, dev)
    rc = lib().pscan(_ptr(a), _ptr(b), _ptr(out), _ptr(h0), rows, n, _stream_handle(stream))
    if rc != SSCAN_OK:
        raise SscanError(rc, "pscan")
    return out


__all__ = ["sscan_fwd", "sscan_bwd", "sscan_step", "pscan", "status_string", "get_last_error", "max_dstate",
           "last_launch_count", "last_plan", "load_library", "SscanError",
           "SIGNATURES", "LIB_PATH"]
