"""sscan_fwd_noalloc: the entry point for callers that cannot allocate device
memory while they run (fixed-budget plugin hooks, real-time loops, runtimes
that hand out memory up front).  It keeps the time-split carry in a fixed
device array instead of the stream-ordered pool and runs on the cp.async-fed
kernels, so its results must agree with sscan_fwd_ex's (up to float32 rounding
order) and with the double-precision oracle within the stated tolerances --
checked here through the C ABI, on two calls in a row (the second call reuses
the array the first one left behind).  This file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
SCRATCH_BYTES = 4 << 20  # SSCAN_NOALLOC_SCRATCH_BYTES in include/sscan.h


@pytest.fixture(scope="module")
def lr():
    import linear_recurrence_gb300 as m
    m.load_library()
    return m


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call(fn, g, out, fs, w, dtype_code, *extra):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(_p(g["u"]), _p(g["delta"]), _p(g["A"]), _p(g["B"]), _p(g["C"]), _p(g["D"]),
              _p(g["h0"]), _p(out), _p(fs), w.batch, w.dim, w.L, w.N, dtype_code, *extra, stream)


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b if isinstance(b, np.ndarray) else b.double().cpu().numpy()
    return float(np.max(np.abs(a - b) / (1.0 + np.abs(b))))


def _segments_fitting(w):
    """Largest time split whose carry (batch*dim*S*(dstate+2) floats) fits the array."""
    return SCRATCH_BYTES // (w.batch * w.dim * (w.N + 2) * 4)


@pytest.mark.parametrize("name,kw,segments", [
    ("long64k", dict(dim=40, L=5000), 6),          # fp32: local pass, fold, carry correction
    ("long64k", dict(dim=40, L=5000), 0),          # automatic plan within the array
    ("bf16_2k", dict(batch=2, dim=80, L=600), 3),  # bf16: local pass, fold, carry correction
    ("dim512", dict(dim=6000, L=512), -1),         # a pinned split that exactly fills the array
])
def test_noalloc_matches_sscan_fwd_and_the_oracle_on_two_calls(lr, name, kw, segments):
    w = workloads.WORKLOADS[name].scaled(**kw)
    if segments == -1:
        segments = _segments_fitting(w)
        w = w.scaled(L=64 * segments)  # segments of two whole chunks
        assert segments >= 2
    x = workloads.make_inputs(w)
    g = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    code = lr.SSCAN_F32 if w.dtype == "f32" else lr.SSCAN_BF16
    io = workloads.io_dtype(w.dtype)
    shape_y, shape_h = (w.batch, w.dim, w.L), (w.batch, w.dim, w.N)
    raw = lr.lib()
    yr, hr = oracle.sscan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["h0"], nthreads=8)

    ref_y = torch.empty(shape_y, dtype=io, device="cuda")
    ref_h = torch.empty(shape_h, dtype=torch.float32, device="cuda")
    # the existing entry point, with the same pinned split when one is given
    assert _call(raw.sscan_fwd_ex, g, ref_y, ref_h, w, code, segments, 0) == lr.SSCAN_OK
    for _ in range(2):
        y = torch.full(shape_y, float("nan"), dtype=io, device="cuda")
        h = torch.full(shape_h, float("nan"), dtype=torch.float32, device="cuda")
        assert _call(raw.sscan_fwd_noalloc, g, y, h, w, code, segments) == lr.SSCAN_OK
        plan = lr.last_plan()
        torch.cuda.synchronize()
        assert lr.get_last_error() == lr.SSCAN_OK
        if segments:
            assert plan.startswith("noalloc ") and f" S={segments} " in plan, plan
        assert _rel(y, ref_y) <= TOL[w.dtype] and _rel(h, ref_h) <= TOL[w.dtype], plan
        assert _rel(y, yr) <= TOL[w.dtype] and _rel(h, hr) <= TOL[w.dtype], plan


def test_noalloc_rejects_a_split_larger_than_its_array(lr):
    # one segment more than the array holds is rejected before any launch
    w = workloads.WORKLOADS["dim512"].scaled(dim=6000, L=512)
    too_many = _segments_fitting(w) + 1
    w = w.scaled(L=64 * too_many)
    assert w.batch * w.dim * too_many * (w.N + 2) * 4 > SCRATCH_BYTES
    x = workloads.make_inputs(w)
    g = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    y = torch.empty((w.batch, w.dim, w.L), device="cuda")
    h = torch.empty((w.batch, w.dim, w.N), device="cuda")
    rc = _call(lr.lib().sscan_fwd_noalloc, g, y, h, w, lr.SSCAN_F32, too_many)
    assert rc == lr.SSCAN_ERR_INVALID and lr.last_launch_count() == 0
    # the automatic plan stays within the array and still computes the scan
    ref_y, ref_h = lr.sscan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["h0"])
    assert _call(lr.lib().sscan_fwd_noalloc, g, y, h, w, lr.SSCAN_F32, 0) == lr.SSCAN_OK
    torch.cuda.synchronize()
    assert _rel(y, ref_y) <= 1e-4 and _rel(h, ref_h) <= 1e-4
