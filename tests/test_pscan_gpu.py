"""GPU parity for the pscan primitive h_t = a_t h_{t-1} + b_t against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from conftest import read_golden

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lr():
    import linear_recurrence_gb300 as m
    m.load_library()
    return m


def _rel_err(got, ref):
    return float(np.max(np.abs(np.asarray(got, np.float64) - ref) / (1.0 + np.abs(ref))))


def test_prefix_sum_golden_exact(lr):
    g = read_golden("prefix_sum.txt")
    x = torch.tensor([g["input"][0]], dtype=torch.float32, device="cuda")
    h = lr.pscan(torch.ones_like(x), x)
    assert h.cpu().numpy().tolist() == [g["output"][0]]


def test_blelloch_example_exact(lr):
    g = read_golden("blelloch_upsweep.txt")
    x = torch.tensor([g["input"][0]], dtype=torch.float32, device="cuda")
    h = lr.pscan(torch.ones_like(x), x)
    assert h.cpu().numpy().tolist() == [[1, 3, 6, 10, 15, 21, 28, 36]]


@pytest.mark.parametrize("rows,n", [(1, 1), (3, 7), (37, 1000), (5, 4096), (2, 100003),
                                    (64, 513), (1000, 64)])
@pytest.mark.parametrize("with_h0", [True, False])
def test_pscan_parity(lr, rows, n, with_h0):
    gen = torch.Generator().manual_seed(rows * 7919 + n)
    a = torch.rand((rows, n), generator=gen) * 1.2 - 0.1   # mostly in (0,1), some outside
    b = torch.randn((rows, n), generator=gen)
    h0 = torch.randn((rows,), generator=gen) if with_h0 else None
    h = lr.pscan(a.cuda(), b.cuda(), None if h0 is None else h0.cuda())
    torch.cuda.synchronize()
    ref = oracle.pscan_seq(a, b, h0)
    assert _rel_err(h.cpu().numpy(), ref) <= 1e-4


def test_pscan_workload_sampled_rows(lr):
    w = workloads.PSCAN_WORKLOADS["pscan_8k"]
    x = workloads.make_pscan_inputs(w)
    h = lr.pscan(x["a"].cuda(), x["b"].cuda(), x["h0"].cuda())
    torch.cuda.synchronize()
    rows = [0, 1, 17, 4095, w.rows - 1]
    ref = oracle.pscan_seq(x["a"][rows], x["b"][rows], x["h0"][rows])
    assert _rel_err(h[rows].cpu().numpy(), ref) <= 1e-4


def test_pscan_rejects_bad_arguments(lr):
    raw = lr.lib()
    assert raw.pscan(None, None, None, None, 1, 1, None) == lr.SSCAN_ERR_INVALID
    assert lr.last_launch_count() == 0
