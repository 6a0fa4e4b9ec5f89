"""Host-side logic of bench.py without a GPU: the multi-rank timing
reduction over two gloo ranks on the CPU, the whole-job throughput, the
reference arm's rank handling, the clock-sample parser and the lookup of
committed ncu traffic figures."""
import datetime as dt
import os
import socket
import sys
from pathlib import Path

import pytest
import torch
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parent.parent
sys.path.insert(0, str(ROOT))
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist = bench.init_dist(ws, use_cuda=False)
    my_ms = [3.0, 5.0][rank]
    worst = bench.max_over_ranks(my_ms, dist, torch.device("cpu"))
    bench.barrier(dist)
    results[rank] = (worst, bench.job_throughput(1000.0, ws, worst))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ws = 2
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(ws, _free_port(), results), nprocs=ws, join=True)
        res = dict(results)
    for rank in range(ws):
        worst, rate = res[rank]
        assert worst == 5.0
        assert rate == pytest.approx(1000.0 * 2 / 5e-3)


def test_single_process_needs_no_process_group():
    assert bench.init_dist(1, use_cuda=False) is None
    assert bench.max_over_ranks(2.5, None, torch.device("cpu")) == 2.5
    assert bench.job_throughput(404_750_336, 1, 1.0) == pytest.approx(404_750_336e3)


def test_reference_arm_only_on_rank_zero():
    class A:
        steps, warmup = 1, 3
    assert bench.run_reference("qgz_single_hop", A, ws=2, rank=1) is None


def test_clock_parser_keeps_the_timed_window():
    t0 = dt.datetime(2026, 1, 1, 12, 0, 0).timestamp()
    def row(sec, mhz, cap="Not Active", therm="Not Active"):
        ts = dt.datetime.fromtimestamp(t0 + sec).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{ts}, {mhz}, 2070, 900.0, 0x0, Not Active, Not Active, {therm}, {cap}"
    rows = [row(-1.0, 600), row(0.1, 1900), row(0.2, 1950, cap="Active"), row(0.3, 2000),
            row(5.0, 700, therm="Active")]
    out = bench.ClockSampler.parse(rows, t0, t0 + 0.4)
    assert out["samples"] == 3
    assert out["sm_mhz"] == 1950
    assert out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]


def test_traffic_lookup_requires_the_captured_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = bench.kernel_source_hash("ef_quant_int4")
    (prof / "traffic.txt").write_text(
        "# kernel workload dram_bytes units source\n"
        f"ef_quant_int4 qgz_single_hop 1000 100 {h}\n"
        "dequant_reduce qgz_single_hop 1000 100 0000000000000000\n")
    for rel in bench.KERNEL_SOURCES["ef_quant_int4"] + bench.KERNEL_SOURCES["dequant_reduce"]:
        (tmp_path / rel).parent.mkdir(parents=True, exist_ok=True)
        (tmp_path / rel).write_bytes((ROOT / rel).read_bytes())
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    assert bench.ncu_traffic("ef_quant_int4", "qgz_single_hop", 400) == 4000
    assert bench.ncu_traffic("dequant_reduce", "qgz_single_hop", 400) is None
    assert bench.ncu_traffic("ef_quant_int4", "qgz_tiny", 400) is None


def test_cpulist_parser():
    assert bench.parse_cpulist("0-3,8,10-11\n") == [0, 1, 2, 3, 8, 10, 11]
    assert bench.parse_cpulist("72-143") == list(range(72, 144))
    assert bench.parse_cpulist("") == []


@pytest.mark.parametrize("name", ["qgz_tiny", "qgz_hierarchical"])
def test_threaded_oracle_step_matches_the_plain_step(name):
    """The all-cores CPU baseline runs the oracle's per-slice quantization,
    per-unit first hop and ranged destination reduces on threads; it must
    compute the same bits (and leave the same error buffer) as the oracle's
    whole-step calls."""
    from concurrent.futures import ThreadPoolExecutor
    import numpy as np
    import oracle
    from weight_communication_gb300 import workloads as wl
    orc = oracle.get()
    w = bench.qgz_sample(wl.QGZ_WORKLOADS[name], 1 << 12)
    g = wl.as_u16(wl.qgz_gradients(w, 0)).ravel().copy()
    ef_a = np.zeros(w.R * w.N, np.float32)
    ef_b = np.zeros(w.R * w.N, np.float32)
    with ThreadPoolExecutor(4) as pool:
        for pieces in (1, 3):
            a = bench.oracle_qgz_step(orc, w, g, ef_a)
            b = bench.oracle_qgz_step_threaded(orc, w, g, ef_b, pool, pieces)
            assert a.dtype == b.dtype and np.array_equal(a.view(np.uint8), b.view(np.uint8))
            assert np.array_equal(ef_a.view(np.uint32), ef_b.view(np.uint32))


def test_percentiles_and_wire_bytes():
    p = bench.percentiles([5.0, 1.0, 4.0, 2.0, 3.0, 6.0, 7.0, 8.0, 9.0, 10.0])
    assert p == {"median": 5.5, "p10": 1.0, "p90": 9.0}
    assert bench.percentiles([2.0]) == {"median": 2.0, "p10": 2.0, "p90": 2.0}
    from weight_communication_gb300 import workloads as wl
    assert bench.wire_bytes(wl.QGZ_SINGLE_HOP)["int4_blocked"] == 0.515625
    assert bench.wire_bytes(wl.QGZ_HIERARCHICAL)["int4_blocked"] == 0.5078125
    assert bench.wire_bytes(wl.QGZ_HIERARCHICAL)["exchanges_per_step"] == 2
