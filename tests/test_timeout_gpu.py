"""The SSCAN_ERR_TIMEOUT path of the error contract, exercised without a fault.

Every wait of the TMA-fed kernels on a copy is bounded.  Here one stage's
barrier is made to expect bytes that no copy delivers (the library's test aid,
sscan_debug_expire_next_wait, with a 2 ms bound), so the waits on it run out as
a stalled copy's would.  The kernel must record SSCAN_ERR_TIMEOUT, which
sscan_get_last_error() reports once and then clears, and the next ordinary
call on the same stream must still be correct against the oracle.  A second
aid, sscan_debug_expire_next_correction_wait, does the same to the carry
correction of a time split.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lr():
    import linear_recurrence_gb300 as m
    m.load_library()
    return m


def _rel_err(got, ref):
    got = got.double().cpu().numpy()
    return float(np.max(np.abs(got - ref) / (1.0 + np.abs(ref))))


@pytest.mark.parametrize("dtype,lanes", [("f32", 0), ("bf16", 0), ("f32", 4)])
def test_expired_wait_reports_timeout_and_the_next_call_is_exact(lr, dtype, lanes):
    w = workloads.WORKLOADS["long64k"].scaled(batch=1, dim=96, L=1024, N=16)
    w = workloads.Workload(**{**w.__dict__, "dtype": dtype})
    x = workloads.make_inputs(w)
    g = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    assert lr.get_last_error() == lr.SSCAN_OK

    lr.debug_expire_next_wait(2000)
    lr.sscan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["h0"], segments=1, lanes=lanes)
    plan = lr.last_plan()
    assert " tma " in plan, plan
    assert lr.get_last_error() == lr.SSCAN_ERR_TIMEOUT, plan
    assert lr.get_last_error() == lr.SSCAN_OK  # reported once, then cleared

    y, hT = lr.sscan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["h0"],
                         segments=1, lanes=lanes)
    torch.cuda.synchronize()
    assert lr.get_last_error() == lr.SSCAN_OK
    yr, hr = oracle.sscan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["h0"], nthreads=8)
    tol = 1e-4 if dtype == "f32" else 2e-2
    assert _rel_err(y, yr) <= tol and _rel_err(hT, hr) <= tol


@pytest.mark.parametrize("dtype,lanes,segments", [("f32", 2, 4), ("bf16", 2, 4), ("f32", 4, 2)])
def test_expired_correction_wait_reports_timeout_and_the_next_call_is_exact(lr, dtype, lanes, segments):
    """The same for the carry correction of a time split: the shuffle kernel's
    (fp32: every warp stages its own C rows and leaves on its own; bf16: a CTA
    ring) and the (4,4,2) kernel's for long segments."""
    w = workloads.WORKLOADS["long64k"].scaled(batch=1, dim=96, L=4096, N=16)
    w = workloads.Workload(**{**w.__dict__, "dtype": dtype})
    x = workloads.make_inputs(w)
    g = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    assert lr.get_last_error() == lr.SSCAN_OK

    lr.debug_expire_next_correction_wait(2000)
    lr.sscan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["h0"], segments=segments, lanes=lanes)
    plan = lr.last_plan()
    assert f"S={segments} " in plan and " corr=tma" in plan, plan
    assert lr.get_last_error() == lr.SSCAN_ERR_TIMEOUT, plan
    assert lr.get_last_error() == lr.SSCAN_OK

    y, hT = lr.sscan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["h0"],
                         segments=segments, lanes=lanes)
    torch.cuda.synchronize()
    assert lr.get_last_error() == lr.SSCAN_OK
    yr, hr = oracle.sscan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["h0"], nthreads=8)
    tol = 1e-4 if dtype == "f32" else 2e-2
    assert _rel_err(y, yr) <= tol and _rel_err(hT, hr) <= tol


def test_the_setting_is_consumed_by_one_call(lr):
    w = workloads.WORKLOADS["long64k"].scaled(batch=1, dim=64, L=512, N=16)
    x = workloads.make_inputs(w)
    g = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    lr.debug_expire_next_wait(2000)
    lr.debug_expire_next_wait(0)  # disarmed again
    lr.debug_expire_next_correction_wait(2000)
    lr.debug_expire_next_correction_wait(0)
    y, _ = lr.sscan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["h0"])
    assert lr.get_last_error() == lr.SSCAN_OK
    yr, _ = oracle.sscan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["h0"], nthreads=8)
    assert _rel_err(y, yr) <= 1e-4
