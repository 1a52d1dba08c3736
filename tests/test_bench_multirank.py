"""The benchmark's multi-rank host path on two gloo ranks (CPU, measurement stubbed).

Under torchrun every rank times an independent replica on its own GPU; the line
reports the units all ranks processed over the slowest rank's time, and only rank 0
prints.  Here rank r reports 8 + 2r microseconds per call, so the line must carry
two replicas' bytes over 10 us.  The reference arm prints on rank 0 only as well.
"""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, outdir, impl):
    import contextlib
    import io
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench

    def fake_measure(args, wl, rk, wd, local, sampler=None, with_e2e=True):
        us = 8.0 + 2.0 * rk
        return dict(sample_us=[us] * 60, steps=args.steps, samples=60, copies=8, cold_us=[12.0] * 200,
                    route="gemv", launches=1, clocks={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [],
                                                      "samples": 5},
                    e2e=None, tile={"n": 0, "split_k": 1, "main_tiles": 0, "tail_split_k": 0}, ws_bytes=0)

    bench.measure_ours = fake_measure
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        argv = ["--gpus", str(world), "--steps", "10", "--warmup", "3", "--no-e2e", "--workload", "q4_6144x5120_t1"]
        if impl == "reference":
            argv += ["--impl", "reference", "--steps", "1", "--workload", "q4_512x1024_t8"]
        rc = bench.main(argv)
    with open(os.path.join(outdir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{rc}\n{buf.getvalue()}")


def _run(tmp_path, impl):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path), impl), nprocs=world,
                       start_method="spawn")
    outs = []
    for r in range(world):
        rc, *lines = open(tmp_path / f"rank{r}.txt").read().splitlines()
        assert rc == "0"
        outs.append([l for l in lines if l.startswith("{")])
    assert outs[1] == [] and len(outs[0]) == 1
    return json.loads(outs[0][0])


def test_two_gloo_ranks_report_the_slowest_replica(tmp_path):
    from weight_only_bit_q4_gb300 import metrics
    line = _run(tmp_path, "ours")
    mb = metrics.model_bytes(6144, 5120, 1)
    assert line["n_gpus"] == 2 and line["scaling"] == "weak"
    assert line["config"]["parallelism"] == "replicas"
    assert line["ms_per_step"] == pytest.approx(0.010)                       # the slower rank
    assert line["value"] == pytest.approx(2 * mb / 10e-6 / 1e9, rel=1e-3)    # both replicas' bytes
    assert "cpu_baseline" not in line                                       # N = 1 only


def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    line = _run(tmp_path, "reference")
    assert line["impl"] == "reference" and line["config"]["workload"] == "q4_512x1024_t8"
