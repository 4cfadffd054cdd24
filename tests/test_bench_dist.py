"""The replica (N > 1) path of bench.py on CPU: two gloo ranks, max-over-ranks
interval and whole-job throughput."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_setup()[:2] == (world, rank)
    ms, value = bench.aggregate(10.0 + 5.0 * rank, 897.1e9 * 20, world, dist, "cpu")
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregate_takes_max_interval():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    assert set(out.keys()) == {0, 1}
    for r in range(world):
        ms, value = out[r]
        assert ms == 15.0
        assert value == pytest.approx(897.1e9 * 20 * 2 / 15e-3 / 1e12)


def test_single_rank_aggregate():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.aggregate(5.0, 1e12, 1)
    assert ms == 5.0 and value == pytest.approx(200.0)


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _clock_line(t, sm, power_cap):
    import datetime
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    cap = "Active" if power_cap else "Not Active"
    return f"{ts}, 0, {sm}, 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, {cap}"


def test_clock_summary_keeps_samples_inside_the_timed_window():
    sys.path.insert(0, ROOT)
    import time

    import bench
    now = time.time()
    c = bench.ClockSampler(0)
    c.proc = _DoneProc()
    c.lines = [_clock_line(now - 2.0, 2070, False), _clock_line(now, 1900, True), _clock_line(now + 0.05, 1910, True),
               _clock_line(now + 3.0, 2070, False), "garbage line"]
    c.mark(now - 0.01, now + 0.06)
    r = c.stop()
    assert r["window"] == "timed window" and r["samples"] == 2
    assert r["sm_mhz"] == 1905.0 and r["sm_max_mhz"] == 2070.0 and r["reasons"] == ["sw_power_cap"]
    # no sample inside the window: the summary falls back to every sample and says so
    c.mark(now + 10.0, now + 11.0)
    r = c.stop()
    assert r["samples"] == 4 and r["window"].startswith("all samples")


def test_peaks_from_measured_file_or_fallback(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import json

    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks == bench.FALLBACK_PEAKS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": {"value": 7100.0}, "bf16_tflops": 2010.5, "bf16_tflops_sustained": {"value": 1790.0},
         "clocks": {"sm_mhz": 2070}}))
    peaks, src = bench.load_peaks()
    assert src == "measured"
    assert peaks == {"hbm_gbs": 7100.0, "bf16_tflops": 2010.5, "bf16_tflops_sustained": 1790.0}
    (tmp_path / "MEASURED_PEAKS.json").write_text("{not json")
    assert bench.load_peaks()[1] == "fallback"
