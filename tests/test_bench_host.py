"""bench.py's host-side logic, on CPU: the barrier and max-over-ranks timing of
the multi-process path over two gloo ranks, the clock-sample summary, and the
oracle arm's JSON line on one small bounded sample."""

import json
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import os

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench as b

    r, w, local = b._dist()
    d = b._init_dist(w)
    b.barrier(d)
    mx = b.reduce_max(1.5 + 2.0 * r, d)
    b.barrier(d)
    # every rank but 0 leaves the oracle arm without work
    ref = b.run_reference(None, r, w) if r != 0 else "rank0"
    results.put((r, w, local, mx, ref))
    d.destroy_process_group()


def test_two_gloo_ranks_reduce_max_and_barrier():
    ctx = mp.get_context("spawn")
    results = ctx.SimpleQueue()
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, results), nprocs=2, join=True,
                       start_method="spawn")
    got = sorted(results.get() for _ in range(2))
    assert got[0][:3] == (0, 2, 0) and got[1][:3] == (1, 2, 1)
    assert got[0][3] == got[1][3] == 3.5          # max over ranks of 1.5 + 2 * rank
    assert got[1][4] is None


def test_single_process_helpers_are_identities():
    assert bench._init_dist(1) is None
    assert bench.reduce_max(2.25, None) == 2.25
    bench.barrier(None)


def _row(ts, sm, smax, power, reasons=("Not Active",) * 4):
    return ", ".join([ts, "0", str(sm), str(smax), str(power), "0x0", *reasons])


def test_clock_summary_keeps_the_timed_window():
    import datetime

    def stamp(sec):
        return datetime.datetime(2026, 1, 1, 12, 0, sec).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]

    t = lambda sec: datetime.datetime(2026, 1, 1, 12, 0, sec).timestamp()
    lines = [
        _row(stamp(0), 900, 2070, 150.0),                                 # idle, before
        _row(stamp(2), 1965, 2070, 1300.0),
        _row(stamp(3), 1980, 2070, 1350.0, ("Not Active", "Not Active", "Not Active", "Active")),
        _row(stamp(4), 1995, 2070, 1380.0),
        _row(stamp(9), 600, 2070, 120.0, ("Active",) + ("Not Active",) * 3),  # after
        "garbage line",
    ]
    s = bench.parse_clock_samples(lines, t(1), t(5))
    assert s["samples"] == 3
    assert s["sm_mhz"] == 1980 and s["sm_max_mhz"] == 2070 and s["power_w"] == 1350.0
    assert s["reasons"] == ["sw_power_cap"]
    everything = bench.parse_clock_samples(lines)
    assert everything["samples"] == 5
    assert everything["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_reference_arm_json_line(capsys):
    bench.main(["--impl", "reference", "--steps", "1", "--cpu-seconds", "0", "--cpu-chunk", "2"])
    line = capsys.readouterr().out.strip().splitlines()[-1]
    out = json.loads(line)
    assert out["impl"] == "reference"
    assert out["unit"] == "TFLOP/s" and out["higher_is_better"] is True
    assert out["value"] > 0 and out["cpu_baseline"]["value"] == out["value"]
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["cores"] >= 1
    assert out["config"]["sample_rows"] == 2
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["e2e"]["d2h_bytes_per_step"] == 0


def test_nvml_window_summary_and_fp8_denominator():
    """The NVML sampler's summary keeps only samples inside the timed window
    and decodes the throttle-reason bits; the W8A8 roofline denominator is
    max(measured FP8, 2 x measured BF16) and says which one it is."""
    s = bench.NvmlSampler.__new__(bench.NvmlSampler)
    s.max_mhz = 2070.0
    s.samples = [(0.5, 900.0, 100.0, 0x0), (1.0, 1950.0, 1300.0, 0x4), (1.5, 1980.0, 1350.0, 0x4),
                 (2.0, 2000.0, 1390.0, 0x0), (3.0, 600.0, 90.0, 0x1)]
    w = s.window(0.9, 2.1)
    assert w["samples"] == 3 and w["sm_mhz"] == 1980.0 and w["reasons"] == ["sw_power_cap"]
    assert w["power_w"] == 1350.0 and w["sm_max_mhz"] == 2070.0
    peaks = {"bf16": 1871.8, "source": "measured", "hbm_gbs": 6751.7}
    d, note = bench.fp8_denominator(peaks, {"tflops": 4100.0, "how": "x"})
    assert d == 4100.0 and note.startswith("measured FP8")
    d, note = bench.fp8_denominator(peaks, {"tflops": 3000.0, "how": "x"})
    assert d == 2 * 1871.8 and "above the measured FP8 3000.0" in note
    d, _ = bench.fp8_denominator(peaks, {"tflops": None, "how": "unavailable"})
    assert d == 2 * 1871.8


def test_nvml_stop_without_a_timed_window():
    import threading

    s = bench.NvmlSampler.__new__(bench.NvmlSampler)
    s.samples, s.t_begin, s.t_end, s.max_mhz = [], None, None, None
    s._stop = threading.Event()
    s.thread = threading.Thread(target=lambda: None)
    s.thread.start()
    assert s.stop() == {}
