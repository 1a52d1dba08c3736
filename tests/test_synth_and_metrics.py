"""Input generator and benchmark-metric pins (CPU only)."""
import numpy as np
import pytest

from weight_only_bit_q4_gb300 import metrics, synth


def test_splitmix64_published_vector():
    # First outputs of splitmix64 seeded with 1234567 (the generator's reference C code).
    got = [int(v) for v in synth.splitmix64(1234567, 5)]
    assert got == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]
    # counter-based: any window equals the same slice of the sequence
    assert np.array_equal(synth.splitmix64(99, 3, start=4), synth.splitmix64(99, 7)[4:])


def test_generator_deterministic_and_distinct():
    a = synth.make_problem(64, 256, 4)
    b = synth.make_problem(64, 256, 4)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    c = synth.make_problem(64, 256, 4, x_seed=5)
    assert not np.array_equal(a[2], c[2])


def test_codes_uniform():
    wq = synth.packed_codes(256, 4096, 0)
    lo, hi = wq & 15, wq >> 4
    for q in (lo, hi):
        counts = np.bincount(q.reshape(-1), minlength=16)
        assert counts.min() > 0.9 * q.size / 16 and counts.max() < 1.1 * q.size / 16


def test_scales_and_activations_ranges():
    s = synth.group_scales(512, 1024, 0).view(np.float16).astype(np.float64)
    assert s.min() >= 1e-3 * (1 - 1e-3) and abs(np.median(s) - (0.02 * 0.6745 + 1e-3)) < 2e-3
    ln = synth.group_scales(2048, 1024, 0, "lognormal").view(np.float16).astype(np.float64)
    assert abs(np.median(np.log(ln)) - np.log(0.02)) < 0.05
    assert abs(np.std(np.log(ln)) - 0.5) < 0.05
    x = synth.activations(64, 1024, 0)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    assert abs(xf.mean()) < 0.02 and abs(xf.std() - 1) < 0.02


def test_outlier_channels():
    idx = synth.outlier_channels(5120, 3)
    assert len(idx) == 51 and len(set(idx.tolist())) == 51
    x = synth.activations(4, 5120, 3, outliers=True)
    xf = np.abs((x.astype(np.uint32) << 16).view(np.float32))
    assert xf[:, idx].mean() > 10 * np.delete(xf, idx, axis=1).mean()


def test_bf16_rounding_ties_to_even():
    f = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20], np.float32)
    bits = synth.float32_to_bf16_bits(f)
    assert bits.tolist() == [0x3F80, 0x3F82, 0x3F81]


def test_weight_bytes_printed(golden):
    for N, K, b, *_ in golden("format_bytes.txt"):
        assert metrics.q4_weight_bytes(int(N), int(K)) == int(b)


def test_metric_functions_reproduce_printed_table(golden):
    N, K = 6144, 5120
    rows = golden("q4_6144x5120_rtx5090_table.txt")
    assert len(rows) == 24
    for T, us, gbs, bw, tf, tc in rows:
        T, us = int(T), float(us) * 1e-6
        assert metrics.model_bytes(N, K, T) == 16711680 + 2 * 5120 * T + 2 * 6144 * T
        assert metrics.logical_gbs(N, K, T, us) == pytest.approx(float(gbs), abs=0.051)
        assert metrics.tflops(N, K, T, us) == pytest.approx(float(tf), abs=0.0051)
        assert metrics.logical_gbs(N, K, T, us) / 1792 * 100 == pytest.approx(float(bw), abs=0.0051)
        if tc != "-":
            assert metrics.tflops(N, K, T, us) / 209.5 * 100 == pytest.approx(float(tc), abs=0.0051)


def test_percentile():
    v = sorted(range(1, 101))
    assert metrics.percentile(v, 50) == 50 and metrics.percentile(v, 95) == 95


def test_sibling_format_bytes_per_group():
    # format table: Q5G64 42 B and Q6G64 50 B per 64 weights, W8G32 34 B per 32 (6144 x 5120 has 80 / 160 groups per row)
    assert metrics.weight_bytes("q4g64", 6144, 5120) == metrics.q4_weight_bytes(6144, 5120) == 6144 * 80 * 34
    assert metrics.weight_bytes("q5g64", 6144, 5120) == 6144 * 80 * 42
    assert metrics.weight_bytes("q6g64", 6144, 5120) == 6144 * 80 * 50
    assert metrics.weight_bytes("w8g32", 6144, 5120) == 6144 * 160 * 34
    assert metrics.weight_bytes("q6g64", 4304, 1152) == 4304 * 1152 // 64 * 50
    assert metrics.model_bytes(6144, 5120, 2, "w8g32") == 6144 * 160 * 34 + 4 * 5120 + 4 * 6144


def test_bench_format_workloads():
    import bench
    wl = bench.workload(bench.parse_args(["--qtype", "q5g64"]))
    assert (wl["name"], wl["N"], wl["K"], wl["T"], wl["qtype"]) == ("q5g64_6144x5120_t1", 6144, 5120, 1, "q5g64")
    wl = bench.workload(bench.parse_args(["--qtype", "w8g32", "--workload", "q4_34816x5120", "--t", "4"]))
    assert wl["name"] == "w8g32_34816x5120_t4"
    wl8 = bench.workload(bench.parse_args(["--qtype", "w8g32", "--workload", "q4_6144x5120", "--t", "8"]))
    assert wl8["name"] == "w8g32_6144x5120_t8"     # beyond four tokens: the warp-MMA route
    planes, s, x = bench.format_problem(dict(wl, N=40, K=256, T=2), rows=7)
    assert planes[0].shape == (7, 256) and s.shape == (7, 8) and x.shape == (2, 256)


def test_bench_linear_add_workload():
    import bench
    wl = bench.workload(bench.parse_args(["--op", "add", "--workload", "q4_6144x5120", "--t", "1024"]))
    assert wl["name"] == "q4_6144x5120_t1024_add" and wl["op"] == "add"
    # the residual is read once: 2 N T bytes on top of the layer's model bytes
    assert bench.op_bytes(wl) == metrics.model_bytes(6144, 5120, 1024) + 2 * 6144 * 1024
    with pytest.raises(SystemExit):
        bench.workload(bench.parse_args(["--op", "add", "--qtype", "q5g64"]))
    with pytest.raises(SystemExit):
        bench.workload(bench.parse_args(["--op", "add", "--route", "tc_fp16"]))
