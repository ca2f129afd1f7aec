"""Host logic of bench.py without a GPU: the multi-rank aggregation (two gloo
ranks on CPU) and the reference arm's JSON line."""

import json
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.slowest_rank_ms(1.0 + rank, dist)          # rank 1 is the slow one
    value = bench.whole_job_tflops(2e12, world, ms)
    out.put((rank, ms, value))
    dist.destroy_process_group()


def test_replicas_aggregate_to_slowest_rank_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in res:
        assert ms == pytest.approx(2.0)                     # max over ranks
        assert value == pytest.approx(2 * 2e12 / 2e-3 / 1e12)


def test_reference_arm_line(tmp_path):
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--reference-seconds", "3"], capture_output=True, text=True, timeout=900, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_nominal_peak_fractions():
    import bench
    nom = bench.nominal_peak(1000.0, 152, 2070.0, 1850.0)
    assert nom["peak_at_max_clock"] == round(152 * 8192 * 2070e6 / 1e12, 1)
    assert abs(nom["frac_at_kernel_clock"] - 1000.0 / (152 * 8192 * 1850e6 / 1e12)) < 1e-4
    assert "peak_at_kernel_clock" not in bench.nominal_peak(1000.0, 152, 2070.0, None)


def test_clock_windows_select_their_samples():
    """Each measured region gets the samples inside its own wall-clock window:
    median clock, maximum clock, the throttle reasons seen, sample count."""
    import bench
    c = bench.Clocks(0)
    c.rows = [(10.0 + 0.05 * i, 1900.0 + i, 2070.0, 500.0, ["sw_power_cap"] if i == 3 else []) for i in range(40)]
    w = c.window(10.01, 10.49)
    assert w["samples"] == 11 and w["sm_max_mhz"] == 2070.0     # t = 10.00 .. 10.50 (50 ms margin)
    assert w["sm_mhz"] == 1905.0 and w["reasons"] == ["sw_power_cap"]
    w2 = c.window(11.01, 11.49)
    assert w2["reasons"] == [] and w2["samples"] == 11
    assert bench.Clocks(0).window(0, 1)["samples"] == 0          # no sampler: an empty record, no failure


def test_oracle_full_problem_record():
    import bench
    from tensor_comm_gemm_gb300 import synth
    rec = bench.oracle_full(synth.workload(0), reps=2)
    assert rec["value"] > 0 and rec["cores"] >= 1 and rec["full_problem_s"] > 0
