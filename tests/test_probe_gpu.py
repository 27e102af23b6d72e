"""The probes that give the roofline its arithmetic peaks: the exponent unit's
(MUFU ex2) and the scan element's (one 2^x and four FP32 per element, or three
FP32 when the states share a rate).  Each launches, reports how many
operations it computes, and times to a plausible rate (152 SMs at up to
2.07 GHz; 32 exponent lanes and 128 FP32 lanes per clock each nominally)."""
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


def _rate(launch, stream):
    import torch
    launch()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    n = launch()
    e.record(stream)
    e.synchronize()
    return n, n / (s.elapsed_time(e) * 1e-3)


def test_element_probe_rates_are_plausible():
    import linear_recurrence_gb300 as lr
    lr.load_library()
    blocks, iters = 152 * 4, 500
    sink = torch.empty(blocks * 256, device="cuda")
    stream = torch.cuda.current_stream()
    n, gen = _rate(lambda: lr.probe_element(blocks, iters, sink=sink, stream=stream), stream)
    assert n == blocks * 256 * 16 * iters
    ns, shared = _rate(lambda: lr.probe_element(blocks, iters, shared_rate=True, sink=sink, stream=stream), stream)
    assert ns == blocks * 256 * 32 * iters
    _, ex2 = _rate(lambda: lr.probe_ex2(blocks, iters, sink=sink, stream=stream), stream)
    clk = 152 * 2.2e9
    # an element with its own 2^x is slower than the exponent unit alone and
    # than the FP32 pipe alone (four operations on 128 lanes); one with a
    # shared rate is bound by its three FP32 operations
    assert 1e12 < gen < min(ex2 * 1.02, clk * 32), (gen, ex2)
    assert gen < shared < clk * 128 / 3, (gen, shared)
    with pytest.raises(lr.SscanError):
        lr.probe_element(blocks, 0, sink=sink, stream=stream)
