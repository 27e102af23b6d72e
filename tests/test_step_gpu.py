"""GPU parity of the single-step decode update against the oracle.

The oracle's sequential scan with one step, h0 = the cached state, defines the
step; its final state is the new cache.  Several steps in a row must also
match one multi-step oracle call (the cache carries the recurrence)."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module")
def lr():
    import linear_recurrence_gb300 as m
    m.load_library()
    return m


def _rel(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - b) / (1 + np.abs(b))))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("batch,dim,N", [(1, 1, 1), (3, 7, 3), (4, 33, 16), (2, 130, 64), (5, 17, 5)])
def test_step_matches_oracle(lr, dtype, batch, dim, N):
    base = workloads.WORKLOADS["dim512"]
    w = workloads.Workload(**{**base.__dict__, "dtype": dtype, "batch": batch, "dim": dim,
                              "L": 6, "N": N, "h0_std": 0.5})
    x = workloads.make_inputs(w)
    st = x["h0"].clone().cuda()
    g = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    io = workloads.io_dtype(dtype)
    for t in range(w.L):
        y = lr.sscan_step(g["u"][:, :, t].contiguous(), g["delta"][:, :, t].contiguous(), g["A"],
                          g["B"][:, :, t].contiguous(), g["C"][:, :, t].contiguous(), g["D"], state=st)
        assert y.dtype == io
        yr, hr = oracle.sscan_fwd(x["u"][:, :, : t + 1], x["delta"][:, :, : t + 1], x["A"],
                                  x["B"][:, :, : t + 1], x["C"][:, :, : t + 1], x["D"], x["h0"])
        torch.cuda.synchronize()
        assert _rel(y.double().cpu().numpy(), yr[:, :, t]) <= TOL[dtype]
        assert _rel(st.double().cpu().numpy(), hr) <= TOL[dtype]


def test_step_without_skip_and_rejects_bad_args(lr):
    w = workloads.WORKLOADS["dim512"].scaled(batch=2, dim=9, L=1, N=8)
    x = workloads.make_inputs(w)
    st = torch.zeros((2, 9, 8), device="cuda")
    y = lr.sscan_step(x["u"][:, :, 0].contiguous().cuda(), x["delta"][:, :, 0].contiguous().cuda(),
                      x["A"].cuda(), x["B"][:, :, 0].contiguous().cuda(),
                      x["C"][:, :, 0].contiguous().cuda(), None, state=st)
    assert lr.last_launch_count() == 1
    yr, hr = oracle.sscan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], None, None)
    torch.cuda.synchronize()
    assert _rel(y.cpu().numpy(), yr[:, :, 0]) <= 1e-4 and _rel(st.cpu().numpy(), hr) <= 1e-4
    with pytest.raises(ValueError):
        lr.sscan_step(x["u"][:, :, 0].contiguous().cuda(), x["delta"][:, :, 0].contiguous().cuda(),
                      x["A"].cuda(), x["B"][:, :, 0].contiguous().cuda(),
                      x["C"][:, :, 0].contiguous().cuda(), None, state=torch.zeros((2, 9, 7), device="cuda"))


def test_step_decode_workload_sampled(lr):
    w = workloads.DECODE_WORKLOAD
    x = workloads.make_decode_inputs(w)
    g = {k: v.cuda() for k, v in x.items()}
    st = g["state"].clone()
    y = lr.sscan_step(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], state=st)
    torch.cuda.synchronize()
    rows = [(0, 0), (w.batch - 1, w.dim - 1), (7, 1234), (100, 4000)]
    for b, d in rows:
        yr, hr = oracle.sscan_fwd(x["u"][b:b + 1, d:d + 1, None], x["delta"][b:b + 1, d:d + 1, None],
                                  x["A"][d:d + 1], x["B"][b:b + 1, :, None], x["C"][b:b + 1, :, None],
                                  x["D"][d:d + 1], x["state"][b:b + 1, d:d + 1])
        assert _rel(y[b, d].float().cpu().numpy(), yr[0, 0, 0]) <= 2e-2
        assert _rel(st[b, d].cpu().numpy(), hr[0, 0]) <= 1e-3
