"""The exponent-unit probe that gives the roofline its MUFU peak: it launches,
reports how many exponentials it computes, and times to a plausible rate (the
GB300's exponent units: 152 SMs at up to 2.07 GHz, 32 lanes per clock each
nominally)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_ex2_probe_rate_is_plausible():
    import linear_recurrence_gb300 as lr
    lr.load_library()
    blocks, iters = 152 * 8, 500
    sink = torch.empty(blocks * 256, device="cuda")
    stream = torch.cuda.current_stream()
    lr.probe_ex2(blocks, iters, sink=sink, stream=stream)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    n = lr.probe_ex2(blocks, iters, sink=sink, stream=stream)
    e.record(stream)
    e.synchronize()
    assert n == blocks * 256 * 16 * iters
    rate = n / (s.elapsed_time(e) * 1e-3)
    assert 1e12 < rate < 152 * 2.2e9 * 32 * 1.05, rate
    with pytest.raises(lr.SscanError):
        lr.probe_ex2(0, iters, sink=sink, stream=stream)
