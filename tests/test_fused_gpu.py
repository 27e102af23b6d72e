"""GPU parity of the scan's options against the oracle: delta_bias and softplus
applied inside the op, the zero-order-hold B-bar, and the SiLU output gate,
alone and together, under single and time-split plans, on vector-aligned and
unaligned rows."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "bf16": 2e-2}
OPTIONS = {
    "bias_softplus": dict(bias=True, softplus=True, zoh=False, gate=False),
    "gate": dict(bias=False, softplus=False, zoh=False, gate=True),
    "zoh": dict(bias=False, softplus=False, zoh=True, gate=False),
    "all": dict(bias=True, softplus=True, zoh=True, gate=True),
}


@pytest.fixture(scope="module")
def lr():
    import linear_recurrence_gb300 as m
    m.load_library()
    return m


def _problem(dtype, L, N=16, A_kind="s4d_jitter", seed=5, batch=2, dim=70):
    base = workloads.WORKLOADS["bf16_2k"]
    w = workloads.Workload(**{**base.__dict__, "dtype": dtype, "batch": batch, "dim": dim, "L": L,
                              "N": N, "A_kind": A_kind, "h0_std": 0.3, "seed": seed})
    return w, workloads.make_inputs(w), workloads.make_option_inputs(w)


def _run_and_compare(lr, w, x, o, opt, segments=0, lanes=0):
    delta = o["delta_raw"] if opt["softplus"] else x["delta"]
    bias = o["delta_bias"] if opt["bias"] else None
    z = o["z"] if opt["gate"] else None
    dev = {k: (None if v is None else v.cuda()) for k, v in
           dict(u=x["u"], delta=delta, A=x["A"], B=x["B"], C=x["C"], D=x["D"], h0=x["h0"],
                z=z, bias=bias).items()}
    y, hT = lr.sscan_fwd(dev["u"], dev["delta"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"],
                         z=dev["z"], delta_bias=dev["bias"], delta_softplus=opt["softplus"],
                         zoh=opt["zoh"], segments=segments, lanes=lanes)
    torch.cuda.synchronize()
    assert lr.get_last_error() == 0
    plan = lr.last_plan()
    yr, hr = oracle.sscan_fwd_full(x["u"], delta, x["A"], x["B"], x["C"], x["D"], z, bias, x["h0"],
                                   delta_softplus=opt["softplus"], zoh=opt["zoh"], nthreads=8)
    tol = TOL[w.dtype]
    ey = float(np.max(np.abs(y.double().cpu().numpy() - yr) / (1 + np.abs(yr))))
    eh = float(np.max(np.abs(hT.double().cpu().numpy() - hr) / (1 + np.abs(hr))))
    assert ey <= tol, (ey, plan)
    assert eh <= tol, (eh, plan)
    return plan


@pytest.mark.parametrize("opt", list(OPTIONS), ids=list(OPTIONS))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("L", [320, 333])  # vector rows / element rows
def test_options_single_and_split(lr, opt, dtype, L):
    w, x, o = _problem(dtype, L)
    plan = _run_and_compare(lr, w, x, o, OPTIONS[opt])
    assert "single" in plan
    # aligned rows take the TMA-fed kernel, the others the cp.async kernel
    assert (" tma " in plan) == (L % 8 == 0), plan
    plan = _run_and_compare(lr, w, x, o, OPTIONS[opt], segments=3)
    assert "S=3" in plan
    if OPTIONS[opt]["zoh"]:
        assert " zoh" in plan
    if OPTIONS[opt]["gate"]:
        assert " gate" in plan


@pytest.mark.parametrize("opt", ["all", "gate", "bias_softplus"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_options_long_segments(lr, opt, dtype):
    # segments of 2048 steps: local pass and carry correction on the TMA kernel
    w, x, o = _problem(dtype, 4096, batch=1, dim=40, seed=11)
    plan = _run_and_compare(lr, w, x, o, OPTIONS[opt], segments=2)
    assert " tma " in plan and "S=2 " in plan, plan


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zoh_shared_rate_and_zero_rates(lr, dtype):
    # a decay rate shared by all states (one exponent per channel and step)
    w, x, o = _problem(dtype, 256, N=64, A_kind="scalar", seed=6, batch=1, dim=40)
    _run_and_compare(lr, w, x, o, OPTIONS["all"])
    # rates that are exactly zero (B-bar = delta*B there) or tiny (series branch)
    w, x, o = _problem(dtype, 256, N=16, seed=7, batch=1, dim=40)
    A = x["A"].clone()
    A[::3, ::2] = 0.0
    A[1::3, 1::2] = -1e-6
    x = {**x, "A": A}
    _run_and_compare(lr, w, x, o, OPTIONS["zoh"])
    _run_and_compare(lr, w, x, o, OPTIONS["all"], segments=2)


@pytest.mark.parametrize("lanes,N", [(4, 13), (8, 25), (16, 61), (4, 40)])
def test_options_on_other_shapes(lr, lanes, N):
    w, x, o = _problem("f32", 200, N=N, seed=8, dim=37)
    _run_and_compare(lr, w, x, o, OPTIONS["all"], lanes=lanes)


def test_softplus_large_and_negative_raw_delta(lr):
    w, x, o = _problem("f32", 128, seed=9, dim=16)
    raw = o["delta_raw"].clone()
    raw[:, :, ::7] = 30.0     # softplus is the identity there (fast decay)
    raw[:, :, 3::7] = -30.0   # and ~1e-13 there (the state holds)
    o = {**o, "delta_raw": raw}
    _run_and_compare(lr, w, x, o, OPTIONS["bias_softplus"])


def test_fused_full_size_every_element(lr):
    """The bf16 2048-channel workload with bias, softplus and the gate, at full
    size in the bench's plan; every output and final state against the oracle."""
    w = workloads.WORKLOADS["bf16_2k"]
    x = workloads.make_inputs(w)
    o = workloads.make_option_inputs(w)
    g = {k: v.cuda() for k, v in x.items() if v is not None}
    y, hT = lr.sscan_fwd(g["u"], o["delta_raw"].cuda(), g["A"], g["B"], g["C"], g["D"],
                         z=o["z"].cuda(), delta_bias=o["delta_bias"].cuda(), delta_softplus=True)
    torch.cuda.synchronize()
    assert lr.get_last_error() == 0
    yr, hr = oracle.sscan_fwd_full(x["u"], o["delta_raw"], x["A"], x["B"], x["C"], x["D"], o["z"],
                                   o["delta_bias"], None, delta_softplus=True,
                                   nthreads=os.cpu_count() or 1)
    y = y.double().cpu().numpy()
    hT = hT.double().cpu().numpy()
    ey = max(float(np.max(np.abs(y[b] - yr[b]) / (1 + np.abs(yr[b])))) for b in range(w.batch))
    eh = float(np.max(np.abs(hT - hr) / (1 + np.abs(hr))))
    assert ey <= TOL["bf16"] and eh <= TOL["bf16"], (ey, eh)
