"""GPU parity of the backward pass (sscan_bwd) against the gradient oracle,
which is pinned to finite differences of the forward oracle.

Per-element gradients (du, ddelta, dh0) use the forward's elementwise forms;
the reductions over channels, batches or time (dA, dB, dC, dD) are compared
against the largest magnitude of their reference:
|err| <= tol * (1 + max|ref|), tol = 1e-4 (fp32) or 1e-3 (bf16 inputs, the
float32 sums of rounded values), since their terms cancel."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
ELEM_TOL = {"f32": 1e-4, "bf16": 2e-2}
SUM_TOL = {"f32": 1e-4, "bf16": 1e-3}


@pytest.fixture(scope="module")
def lr():
    import linear_recurrence_gb300 as m
    m.load_library()
    return m


def _inputs(dtype, batch, dim, L, N, seed, h0=True, D=True, A_kind="s4d_jitter"):
    base = workloads.WORKLOADS["bf16_2k"]
    w = workloads.Workload(**{**base.__dict__, "dtype": dtype, "batch": batch, "dim": dim, "L": L, "N": N,
                              "A_kind": A_kind, "h0_std": 0.3 if h0 else 0.0, "seed": seed})
    x = workloads.make_inputs(w)
    g = torch.Generator().manual_seed(seed + 7)
    dy = torch.randn((batch, dim, L), generator=g).to(workloads.io_dtype(dtype))
    dhT = torch.randn((batch, dim, N), generator=g)
    if not D:
        x = {**x, "D": None}
    return w, x, dy, dhT


def _check(lr, dtype, x, dy, dhT):
    dev = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    got = lr.sscan_bwd(dev["u"], dev["delta"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"],
                       dy.cuda(), None if dhT is None else dhT.cuda())
    torch.cuda.synchronize()
    assert lr.get_last_error() == 0
    ref = oracle.sscan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["h0"], dy, dhT)
    for name in ("du", "ddelta", "dh0"):
        r = ref[name]
        gv = got[name].double().cpu().numpy()
        err = float(np.max(np.abs(gv - r) / (1 + np.abs(r)))) if r.size else 0.0
        assert err <= ELEM_TOL[dtype], (name, err, lr.last_plan())
    for name in ("dA", "dB", "dC", "dD"):
        r = ref[name]
        if r is None:
            assert got[name] is None
            continue
        gv = got[name].double().cpu().numpy()
        err = float(np.max(np.abs(gv - r))) / (1 + float(np.max(np.abs(r)))) if r.size else 0.0
        assert err <= SUM_TOL[dtype], (name, err, lr.last_plan())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [3, 4, 8, 13, 16, 25, 64])
def test_bwd_matches_oracle(lr, dtype, N):
    _, x, dy, dhT = _inputs(dtype, 2, 37, 96, N, seed=50 + N)
    _check(lr, dtype, x, dy, dhT)


@pytest.mark.parametrize("L", [1, 15, 16, 17, 50, 333])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bwd_lengths_and_unaligned_rows(lr, L, dtype):
    _, x, dy, dhT = _inputs(dtype, 1, 20, L, 16, seed=60 + L)
    _check(lr, dtype, x, dy, dhT)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dim,L,N", [(20, 1024, 16), (37, 2000, 13), (8, 4096, 64)])
def test_bwd_time_split(lr, dtype, dim, L, N):
    # few channels and a long sequence: the plan splits time into segments
    _, x, dy, dhT = _inputs(dtype, 1, dim, L, N, seed=80 + N)
    _check(lr, dtype, x, dy, dhT)
    assert " S=1 " not in lr.last_plan() + " ", lr.last_plan()


def test_bwd_without_skip_h0_and_final_gradient(lr):
    _, x, dy, _ = _inputs("f32", 2, 18, 64, 16, seed=70, h0=False, D=False)
    _check(lr, "f32", x, dy, None)


def test_bwd_shared_rate(lr):
    _, x, dy, dhT = _inputs("bf16", 2, 24, 128, 64, seed=71, A_kind="scalar")
    _check(lr, "bf16", x, dy, dhT)


def test_bwd_zero_sizes(lr):
    u = torch.zeros((1, 3, 0), device="cuda")
    A = torch.zeros((3, 4), device="cuda")
    B = torch.zeros((1, 4, 0), device="cuda")
    dhT = torch.randn((1, 3, 4), device="cuda")
    g = lr.sscan_bwd(u, u, A, B, B, None, None, u, dhT)
    torch.cuda.synchronize()
    assert torch.equal(g["dh0"], dhT) and torch.count_nonzero(g["dA"]) == 0


def test_bwd_full_size_sampled(lr):
    """The bf16 2048-channel workload at full size: du, ddelta, dh0 on sampled
    channels, dA and dD of sampled channels (all batches), dB and dC of batch 0
    (all channels), against the oracle."""
    w = workloads.WORKLOADS["bf16_2k"]
    x = workloads.make_inputs(w)
    g = torch.Generator().manual_seed(123)
    dy = torch.randn((w.batch, w.dim, w.L), generator=g).to(torch.bfloat16)
    dhT = torch.randn((w.batch, w.dim, w.N), generator=g)
    dev = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    got = lr.sscan_bwd(dev["u"], dev["delta"], dev["A"], dev["B"], dev["C"], dev["D"], None, dy.cuda(),
                       dhT.cuda())
    torch.cuda.synchronize()
    for d in (0, 1500, 2047):
        sl = slice(d, d + 1)
        ref = oracle.sscan_bwd(x["u"][:, sl], x["delta"][:, sl], x["A"][sl], x["B"], x["C"], x["D"][sl],
                               None, dy[:, sl], dhT[:, sl])
        for name in ("du", "ddelta", "dh0"):
            gv = got[name][:, sl].double().cpu().numpy()
            assert np.max(np.abs(gv - ref[name]) / (1 + np.abs(ref[name]))) <= ELEM_TOL["bf16"], (d, name)
        for name in ("dA", "dD"):
            gv = got[name][sl].double().cpu().numpy()
            assert np.max(np.abs(gv - ref[name])) / (1 + np.max(np.abs(ref[name]))) <= SUM_TOL["bf16"], (d, name)
    ref = oracle.sscan_bwd(x["u"][:1], x["delta"][:1], x["A"], x["B"][:1], x["C"][:1], x["D"], None,
                           dy[:1], dhT[:1])
    for name in ("dB", "dC"):
        gv = got[name][:1].double().cpu().numpy()
        assert np.max(np.abs(gv - ref[name])) / (1 + np.max(np.abs(ref[name]))) <= SUM_TOL["bf16"], name
