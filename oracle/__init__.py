"""Double-precision CPU oracle for the selective scan and the pscan primitive.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package.  The product path (``linear_recurrence_gb300``) never imports it, and
this package never imports the product; the two share only the seeded input
generators in ``workloads.py``, which hold none of the method's arithmetic.

The arithmetic lives in ``sscan_oracle.c`` (plain C, double precision,
``-ffp-contract=off``); this module only builds it with gcc, loads it with
ctypes and converts arrays to float64.  Each function cites the passage it
follows:

* :func:`sscan_fwd` -- the sequential selective scan of the "Mamba 状态空间模型：从理论到生产级推理的 CUDA 内核优化实战"
  page, section 2.3 (pseudocode) and section 7.1 (PyTorch reference), and of
  the mamba.py listing on the "图解Blelloch并行扫描" page, section 3.2.
* :func:`sscan_fwd_full` -- the same scan with its options: softplus of
  delta + bias inside the op (section 7.1 and section 2.2 of that page), the
  zero-order-hold B-bar of its section 1.2, and an output gate
  (y + D*u) * silu(z) (the gate activation fused into the scan kernel on the
  "为什么Mamba的“并行扫描”不是真并行" page, section 2).
* :func:`sscan_bwd` -- the gradients of :func:`sscan_fwd` by the chain rule in
  reverse time (the backward pass of "并行扫描与硬件感知优化", section 3.3).
* :func:`pscan_seq` -- h_t = a_t*h_{t-1} + b_t row by row (the ``pscan``
  primitive of that listing; with a = 1 the prefix sum of its section 1.1).
* :func:`pscan_blelloch` -- the same recurrence by Blelloch up-sweep /
  down-sweep over (a, b) pairs ("图解Blelloch并行扫描", section 2), with the
  combine (a1,b1) o (a2,b2) = (a2*a1, a2*b1+b2) of the "并行扫描与硬件感知优化 (mhpq.cn/news/1077344)" page,
  section 2.2.

Every function is pinned by ``tests/test_oracle_pins.py`` to values the pages
print, closed forms, special cases and brute force; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sscan_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile ``sscan_oracle.c`` into ``_liboracle.so`` with gcc (host code
    only; identical results on x86-64 and aarch64)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_sscan_fwd_mutant.argtypes = [
            _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
            _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int]
        lib.oracle_sscan_fwd_mutant.restype = ctypes.c_int
        lib.oracle_sscan_fwd_full_mutant.argtypes = [
            _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
            _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_sscan_fwd_full_mutant.restype = ctypes.c_int
        lib.oracle_sscan_bwd_mutant.argtypes = [_dp] * 16 + [_i64, _i64, _i64, _i64, ctypes.c_int]
        lib.oracle_sscan_bwd_mutant.restype = ctypes.c_int
        lib.oracle_bwd_mutation_count.argtypes = []
        lib.oracle_bwd_mutation_count.restype = ctypes.c_int
        lib.oracle_mutation_count.argtypes = []
        lib.oracle_mutation_count.restype = ctypes.c_int
        lib.oracle_pscan_seq.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64]
        lib.oracle_pscan_seq.restype = ctypes.c_int
        lib.oracle_pscan_blelloch.argtypes = [
            _dp, _dp, ctypes.c_double, _dp, _i64, _dp, _dp,
            ctypes.POINTER(ctypes.c_int64)]
        lib.oracle_pscan_blelloch.restype = ctypes.c_int
        _lib = lib
        return lib


def _f64(x):
    """Contiguous float64 copy of an array-like (numpy or a CPU torch tensor;
    bfloat16 tensors are widened exactly through float32)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor, imported lazily by the caller
        t = x.detach().cpu()
        if str(t.dtype) == "torch.bfloat16":
            t = t.float()
        x = t.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def mutation_count() -> int:
    return int(_load().oracle_mutation_count())


def sscan_fwd(u, delta, A, B, C, D=None, h0=None, *, nthreads: int = 1,
              mutation: int = 0):
    """Sequential selective scan in float64.

    Shapes: u, delta [batch, dim, L]; A [dim, N]; B, C [batch, N, L];
    D [dim] or None; h0 [batch, dim, N] or None.
    Returns (y [batch, dim, L], final_state [batch, dim, N]) as float64.
    ``mutation`` != 0 plants a deliberate mistake; only the oracle's own pin
    tests use it.
    """
    u, delta, A, B, C = map(_f64, (u, delta, A, B, C))
    D, h0 = _f64(D), _f64(h0)
    if u.ndim != 3 or delta.shape != u.shape:
        raise ValueError("u and delta must both be [batch, dim, L]")
    batch, dim, L = u.shape
    if A.ndim != 2 or A.shape[0] != dim:
        raise ValueError("A must be [dim, N]")
    N = A.shape[1]
    if B.shape != (batch, N, L) or C.shape != (batch, N, L):
        raise ValueError("B and C must be [batch, N, L]")
    if D is not None and D.shape != (dim,):
        raise ValueError("D must be [dim]")
    if h0 is not None and h0.shape != (batch, dim, N):
        raise ValueError("h0 must be [batch, dim, N]")
    y = np.zeros((batch, dim, L), dtype=np.float64)
    hT = np.zeros((batch, dim, N), dtype=np.float64)
    rc = _load().oracle_sscan_fwd_mutant(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(h0),
        _ptr(y), _ptr(hT), batch, dim, L, N, int(nthreads), int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_sscan_fwd rejected its arguments ({rc})")
    return y, hT


FLAG_SOFTPLUS = 1
FLAG_ZOH = 2


def sscan_fwd_full(u, delta, A, B, C, D=None, z=None, delta_bias=None, h0=None, *,
                   delta_softplus: bool = False, zoh: bool = False, nthreads: int = 1,
                   mutation: int = 0):
    """The scan with its options, in float64 (the C function's header states
    the definitions and the passages they follow):

    * ``delta_bias`` [dim]: delta <- delta + delta_bias[d];
    * ``delta_softplus``: then delta <- softplus(delta);
    * ``zoh``: the zero-order-hold B-bar expm1(delta*A)/A * B instead of delta*B;
    * ``z`` [batch, dim, L]: out = (y + D*u) * silu(z).

    Returns (y, final_state) like :func:`sscan_fwd`.
    """
    u, delta, A, B, C = map(_f64, (u, delta, A, B, C))
    D, h0, z, delta_bias = _f64(D), _f64(h0), _f64(z), _f64(delta_bias)
    if u.ndim != 3 or delta.shape != u.shape:
        raise ValueError("u and delta must both be [batch, dim, L]")
    batch, dim, L = u.shape
    if A.ndim != 2 or A.shape[0] != dim:
        raise ValueError("A must be [dim, N]")
    N = A.shape[1]
    if B.shape != (batch, N, L) or C.shape != (batch, N, L):
        raise ValueError("B and C must be [batch, N, L]")
    if D is not None and D.shape != (dim,):
        raise ValueError("D must be [dim]")
    if z is not None and z.shape != u.shape:
        raise ValueError("z must be [batch, dim, L]")
    if delta_bias is not None and delta_bias.shape != (dim,):
        raise ValueError("delta_bias must be [dim]")
    if h0 is not None and h0.shape != (batch, dim, N):
        raise ValueError("h0 must be [batch, dim, N]")
    flags = (FLAG_SOFTPLUS if delta_softplus else 0) | (FLAG_ZOH if zoh else 0)
    y = np.zeros((batch, dim, L), dtype=np.float64)
    hT = np.zeros((batch, dim, N), dtype=np.float64)
    rc = _load().oracle_sscan_fwd_full_mutant(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
        _ptr(h0), _ptr(y), _ptr(hT), batch, dim, L, N, flags, int(nthreads), int(mutation))
    if rc != 0:
        raise ValueError(f"oracle_sscan_fwd_full rejected its arguments ({rc})")
    return y, hT


def bwd_mutation_count() -> int:
    return int(_load().oracle_bwd_mutation_count())


def sscan_bwd(u, delta, A, B, C, D, h0, dy, dhT=None, *, mutation: int = 0):
    """Gradients of the selective scan in float64 (the chain rule on the forward
    recurrence in reverse time; the C function's header states the formulas).

    dy [batch, dim, L] is dL/dy, dhT [batch, dim, N] dL/d(final_state) (None =
    0).  Returns a dict with du, ddelta [batch, dim, L]; dA [dim, N]; dB, dC
    [batch, N, L]; dD [dim] (None when D is None); dh0 [batch, dim, N].
    """
    u, delta, A, B, C, dy = map(_f64, (u, delta, A, B, C, dy))
    D, h0, dhT = _f64(D), _f64(h0), _f64(dhT)
    batch, dim, L = u.shape
    N = A.shape[1]
    if dy.shape != u.shape:
        raise ValueError("dy must be [batch, dim, L]")
    if dhT is not None and dhT.shape != (batch, dim, N):
        raise ValueError("dhT must be [batch, dim, N]")
    out = {"du": np.zeros((batch, dim, L)), "ddelta": np.zeros((batch, dim, L)),
           "dA": np.zeros((dim, N)), "dB": np.zeros((batch, N, L)), "dC": np.zeros((batch, N, L)),
           "dD": None if D is None else np.zeros(dim), "dh0": np.zeros((batch, dim, N))}
    rc = _load().oracle_sscan_bwd_mutant(
        _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(h0), _ptr(dy), _ptr(dhT),
        _ptr(out["du"]), _ptr(out["ddelta"]), _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]),
        _ptr(out["dD"]), _ptr(out["dh0"]), batch, dim, L, N, int(mutation))
    if rc != 0:
        raise ValueError("oracle_sscan_bwd rejected its arguments")
    return out


def sscan_fwd_channels(u, delta, A, B, C, D, h0, channels, *, nthreads: int = 1):
    """The oracle on a sample of channels of a larger problem.

    ``channels`` is a list of (b, d) pairs; each row is computed in full over
    all L steps (channels are independent, so the sample is exact).  Returns
    (y [k, L], final_state [k, N]) in the order given.
    """
    ys, hs = [], []
    for b, d in channels:
        ub = _f64(u[b:b + 1, d:d + 1])
        db = _f64(delta[b:b + 1, d:d + 1])
        Ab = _f64(A[d:d + 1])
        Bb = _f64(B[b:b + 1])
        Cb = _f64(C[b:b + 1])
        Db = None if D is None else _f64(D[d:d + 1])
        hb = None if h0 is None else _f64(h0[b:b + 1, d:d + 1])
        y, hT = sscan_fwd(ub, db, Ab, Bb, Cb, Db, hb, nthreads=nthreads)
        ys.append(y[0, 0])
        hs.append(hT[0, 0])
    return np.stack(ys), np.stack(hs)


def pscan_seq(a, b, h0=None):
    """h[r,t] = a[r,t]*h[r,t-1] + b[r,t] with h[r,-1] = h0[r] (0 if None).
    a, b: [rows, len]; returns float64 [rows, len]."""
    a, b = _f64(a), _f64(b)
    if a.ndim != 2 or b.shape != a.shape:
        raise ValueError("a and b must both be [rows, len]")
    rows, n = a.shape
    h0 = _f64(h0)
    if h0 is not None and h0.shape != (rows,):
        raise ValueError("h0 must be [rows]")
    h = np.zeros((rows, n), dtype=np.float64)
    rc = _load().oracle_pscan_seq(_ptr(a), _ptr(b), _ptr(h0), _ptr(h), rows, n)
    if rc != 0:
        raise ValueError("oracle_pscan_seq rejected its arguments")
    return h


def pscan_blelloch(a, b, h0: float = 0.0, *, trace: bool = False):
    """One row by Blelloch's up-sweep / down-sweep over (a, b) pairs.

    Returns h (float64 [len]); with ``trace=True`` also the up-sweep levels as
    (trace_a, trace_b), each [levels, padded_len].
    """
    a, b = _f64(a).ravel(), _f64(b).ravel()
    if a.shape != b.shape:
        raise ValueError("a and b must have the same length")
    n = a.shape[0]
    P = 1
    while P < n:
        P <<= 1
    levels = max(P.bit_length() - 1, 0)
    h = np.zeros(n, dtype=np.float64)
    ta = np.zeros((max(levels, 1), P), dtype=np.float64) if trace else None
    tb = np.zeros((max(levels, 1), P), dtype=np.float64) if trace else None
    lv = ctypes.c_int64(0)
    rc = _load().oracle_pscan_blelloch(_ptr(a), _ptr(b), float(h0), _ptr(h), n,
                                       _ptr(ta), _ptr(tb), ctypes.byref(lv))
    if rc != 0:
        raise ValueError("oracle_pscan_blelloch rejected its arguments")
    if trace:
        return h, (ta[:lv.value], tb[:lv.value])
    return h
