"""The benchmark's JSON line, checked on the CPU with the GPU measurement stubbed:
every key the line must carry, the types, and the figures derived from the
timings (whole-job rate, roofline fraction, end-to-end rate, launch count)."""
import json

import pytest

import bench
from weight_only_bit_q4_gb300 import metrics


def _fake_measure(args, wl, rank, world, local, sampler=None, with_e2e=True):
    us = 8.0 if wl["T"] == 1 else (20.0 if wl["T"] == 8 else 100.0)
    return dict(sample_us=[us] * 60, steps=args.steps, samples=60, copies=8,
                cold_us=[12.0] * 200, route="gemv" if wl["T"] == 1 else "tc_splitk", launches=1,
                clocks={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 5},
                e2e=dict(us=[32.0] * 100, memcpy_us=[36.0] * 100, eager_us=[40.0] * 100, host_entry=True, h2d=2 * wl["K"] * wl["T"], d2h=2 * wl["N"] * wl["T"]) if with_e2e else None,
                tile={"n": 0, "split_k": 1, "main_tiles": 0, "tail_split_k": 0}, ws_bytes=0)


@pytest.fixture
def line(monkeypatch, capsys):
    monkeypatch.setattr(bench, "measure_ours", _fake_measure)
    monkeypatch.setattr(bench, "cpu_baseline", lambda wl: {"value": 0.05, "unit": "GB/s", "cores": 8,
                                                           "kind": "oracle", "sample": "rows 0..9"})
    assert bench.main(["--steps", "10", "--warmup", "3"]) == 0
    out = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(out) == 1
    return json.loads(out[0])


def test_line_carries_every_key(line):
    for k, typ in [("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                   ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                   ("dtype", str), ("data", str), ("config", dict), ("roofline", dict), ("e2e", dict),
                   ("gpu_launches", int), ("clocks", dict), ("cpu_baseline", dict)]:
        assert isinstance(line[k], typ), k
    assert "vs_baseline" in line and line["vs_baseline"] is None
    assert line["config"]["workload"] == "q4_6144x5120_t1"
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in line["roofline"], k
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in line["e2e"], k
    for k in ("value", "unit", "cores", "kind", "sample"):
        assert k in line["cpu_baseline"], k
    assert line["warmup"] >= 3 and line["scaling"] == "weak" and line["data"] == "synthetic"


def test_derived_figures(line):
    mb = metrics.model_bytes(6144, 5120, 1)
    # median sample: 8 us per call
    assert line["ms_per_step"] == pytest.approx(0.008)
    assert line["steps"] == 10 and line["samples"] >= 50
    assert line["value"] == pytest.approx(mb / 8e-6 / 1e9, rel=1e-3)
    assert line["unit"] == "GB/s" and line["roofline"]["bound"] == "hbm"
    assert line["roofline"]["frac"] == pytest.approx(line["roofline"]["achieved"] / line["roofline"]["peak"], rel=1e-3)
    assert line["e2e"]["value"] == pytest.approx(mb / 32e-6 / 1e9, rel=1e-3)
    assert line["e2e"]["h2d_bytes_per_step"] == 2 * 5120 and line["e2e"]["d2h_bytes_per_step"] == 2 * 6144
    assert line["e2e"]["eager_us"] == pytest.approx(40.0) and line["e2e"]["memcpy_us"] == pytest.approx(36.0)
    assert "q4lin_linear_host" in line["e2e"]["method"]
    assert line["gpu_launches"] == 10 * 60


def test_secondary_records(line):
    # the small-T (T = 8) and large-T (T = 1024) records of the same weight, each with its own figures
    recs = line["records"]
    assert [r["workload"] for r in recs] == ["q4_6144x5120_t8", "q4_6144x5120_t1024"]
    r8, r1024 = recs
    assert r8["unit"] == "GB/s" and r8["roofline"]["bound"] == "hbm"
    assert r8["value"] == pytest.approx(metrics.model_bytes(6144, 5120, 8) / 20e-6 / 1e9, rel=1e-3)
    assert r1024["unit"] == "TFLOP/s" and r1024["roofline"]["bound"] == "tensor"
    assert r1024["value"] == pytest.approx(metrics.useful_flops(6144, 5120, 1024) / 100e-6 / 1e12, rel=1e-3)
    for r in recs:
        for k in ("us", "roofline", "cold_call", "clocks", "steps", "samples", "route", "tile"):
            assert k in r, k
        assert r["steps"] == 10


def test_sweep_spec_and_line():
    # --sweep: ranges and single values in order, duplicates dropped; one line per T with the
    # contract's fields and the change of the median against the previous T
    assert bench.parse_sweep("1:4:1,8,2:3,384,385") == [1, 2, 3, 4, 8, 384, 385]
    assert bench.parse_sweep("4:16:4") == [4, 8, 12, 16]
    with pytest.raises(SystemExit):
        bench.parse_sweep("0:4:1")
    r1 = bench.sweep_row("w_t1", "q4g64", 6144, 5120, 1, [8.0, 8.0, 9.0], 7200.0, None)
    mb = metrics.model_bytes(6144, 5120, 1)
    assert r1["median_us"] == 8.0 and r1["min_us"] == 8.0 and r1["delta_%"] is None
    assert r1["effective_GB/s"] == pytest.approx(mb / 8e-6 / 1e9, rel=1e-3)
    assert r1["DRAM_%"] == pytest.approx(100 * mb / 8e-6 / 1e9 / bench.DRAM_SPEC_GBS, rel=1e-3)
    assert r1["READ_%"] == pytest.approx(100 * mb / 8e-6 / 1e9 / 7200.0, rel=1e-3)
    assert r1["memory_floor_pct"] == pytest.approx(r1["DRAM_%"], rel=1e-3)   # both against the spec
    r2 = bench.sweep_row("w_t2", "q4g64", 6144, 5120, 2, [10.0, 10.0], 7200.0, r1["median_us"])
    assert r2["delta_%"] == pytest.approx(25.0)
    assert list(r2) == list(bench.SWEEP_COLUMNS)
