"""Host-side multi-rank logic of bench.py on CPU (gloo, world_size 2).

The selective scan partitions into independent (batch, channel) problems, so
N GPUs run N independent replicas with no data-path collective; the only
cross-rank steps are the timing barrier and the max-over-ranks of the step
time (the job is as slow as its slowest rank).  These run as two gloo ranks on
CPU, with no GPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(ws), "LOCAL_RANK": str(rank)})
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, got_local = bench._dist()
        bench.barrier(ws)
        slowest = bench.max_over_ranks(1.0 + 0.5 * rank, ws)
        # weak scaling: every rank processes its own full workload
        w = bench.workloads.WORKLOADS["dim512"]
        value = ws * w.channels * w.L / slowest
        q.put((rank, got_ws, got_rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step_time():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(ws))
    for rank, got_ws, got_rank, slowest, value in res:
        assert got_ws == ws and got_rank == rank
        assert slowest == pytest.approx(1.5)
        assert value == pytest.approx(2 * 512 * 8192 / 1.5)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1",
                                      "--warmup", "0"])
    assert bench.main() == 0
    assert capsys.readouterr().out == ""


def test_roofline_arithmetic():
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    pk = {"hbm_gbs": 6788.3, "sm_max_mhz": 2070.0, "source": "measured"}
    w = bench.workloads.WORKLOADS["dim512"]
    a = bench.algorithmic(w)
    assert a["bytes"] == 3 * 512 * 8192 * 4 + 2 * 16 * 8192 * 4 + 512 * 16 * 4 + 512 * 4 + 512 * 16 * 4
    # one state per channel: the bytes bind
    w1 = w.scaled(N=1)
    a1 = bench.algorithmic(w1)
    r = bench.roofline(w1, 1e-5, pk)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(a1["bytes"] / 1e-5 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6788.3)
    assert r["frac_of_hbm"] == pytest.approx(r["frac"])
    # the arithmetic bound: every exponent and FP32 operation one issue-slot
    # lane, 128 lanes per clock per SM at the maximum clock
    issue = 128 * 152 * 2070e6
    rb = bench.roofline(bench.workloads.WORKLOADS["bf16_2k"], 1e-4, pk)
    ab = bench.algorithmic(bench.workloads.WORKLOADS["bf16_2k"])
    assert ab["exps"] == ab["elements"] and ab["fp32"] == 4 * ab["elements"]
    assert rb["bound"] == "alu" and rb["peak"] == pytest.approx(issue / 1e12)
    assert rb["t_issue_us"] == pytest.approx(5 * ab["elements"] / issue * 1e6)
    assert rb["frac"] == pytest.approx(5 * ab["elements"] / 1e-4 / issue)
    assert rb["frac_of_roofline"] == pytest.approx(rb["t_issue_us"] * 1e-6 / 1e-4)
    # dim512: the issue bound (8.3 us) is above the HBM bound (7.6 us)
    r = bench.roofline(w, 1e-5, pk)
    assert r["bound"] == "alu" and r["t_issue_us"] > r["t_hbm_us"]
    assert r["frac_of_hbm"] == pytest.approx(a["bytes"] / (6788.3e9 * 1e-5))
    # one rate per channel: one exponent per (b, d, t), three FP32 per element
    ww = bench.workloads.WORKLOADS["wide64"]
    aw = bench.algorithmic(ww)
    assert aw["exps"] == aw["tokens_channels"] and aw["fp32"] == 3 * aw["elements"]
    rw = bench.roofline(ww, 1e-3, pk)
    assert rw["t_issue_us"] == pytest.approx((aw["exps"] + aw["fp32"]) / issue * 1e6)
    # the element probe's measured rates are reported beside the bound
    pk.update({"elem_per_s": 5.8e12, "elem_shared_per_s": 9.7e12})
    rw = bench.roofline(ww, 1e-3, pk)
    assert rw["t_alu_measured_us"] == pytest.approx(aw["elements"] / 9.7e12 * 1e6)
    assert rw["frac_of_measured_alu"] == pytest.approx(aw["elements"] / 9.7e12 / 1e-3)
