"""The one-line JSON contract of bench.py.

The reference arm (the fp64 oracle on the host cores) runs on the CPU; the GPU arm is
checked on the GPU with a small workload. Both lines carry the same metric, unit and
config keys, and the timing rules they encode (at least three warm-up steps, L2 state,
clock record) are part of the line."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def run_bench(*args, timeout=900):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=timeout, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def check_common(line, impl_steps):
    import bench
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["n_gpus"] == 1 and line["steps"] == impl_steps and line["warmup"] >= 3
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["vs_baseline"] is None
    assert line["data"] == "synthetic"
    assert line["config"]["workload"] == "fixed_T17_H1"
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == bench.UNIT
    assert e2e["h2d_bytes_per_step"] >= 0 and e2e["d2h_bytes_per_step"] >= 0


def test_reference_arm_line():
    line = run_bench("--impl", "reference", "--steps", "2", "--warmup", "3", "--workload", "fixed_T17_H1")
    check_common(line, 2)
    assert line["impl"] == "reference" and line["dtype"] == "f64"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.gpu
def test_gpu_arm_line():
    line = run_bench("--steps", "2", "--warmup", "3", "--workload", "fixed_T17_H1", "--decode-requests", "4")
    check_common(line, 2)
    assert "impl" not in line or line["impl"] != "reference"
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert set(rf["kernel_ms"]) >= {"fwd_intra", "fwd_scan", "bwd_scan", "bwd_state", "bwd_wy", "bwd_pair"}
    assert line["gpu_launches"] > 0
    assert line["tflops_dense_tile"] > line["tflops"] > 0
    assert abs(line["gbs"] - line["value"] * 3590 / 1e9) < 1e-6 * line["gbs"] and 0 < line["pct_hbm_peak"] < 1
    assert line["e2e"]["h2d_bytes_per_step"] > 0 and line["e2e"]["d2h_bytes_per_step"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] > 0
    clk = line["clocks"]
    assert clk["sm_max_mhz"] > 0 and isinstance(clk["reasons"], list)
    assert line["decode"]["ms_per_step"] > 0


def test_clock_samples_are_taken_inside_the_timed_region():
    """The sampler keeps the samples whose nvidia-smi timestamp falls inside the timed region
    (or the nearest one when none does), and reports their median clock and the reasons."""
    import bench

    class FinishedProcess:   # stands in for the nvidia-smi process at stop()
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    cs = bench.ClockSampler(0)
    cs.proc = FinishedProcess()
    samples = [("2026/12/03 10:00:00.000", "1200", "Not Active"),
               ("2026/12/03 10:00:00.500", "2070", "Not Active"),
               ("2026/12/03 10:00:00.600", "2060", "Active"),
               ("2026/12/03 10:00:01.500", "900", "Not Active")]
    cs.rows = [[stamp, "0", mhz, "2070", "1000.0", "0x0", "Not Active", "Not Active", "Not Active", cap]
               for stamp, mhz, cap in samples]
    t0 = cs._when("2026/12/03 10:00:00.400")
    cs.t0, cs.t1 = t0, t0 + 0.3
    out = cs.stop()
    assert out["samples"] == 2 and out["sm_mhz"] == 2065.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    cs.t0 = cs.t1 = cs._when("2026/12/03 10:00:01.400")
    out = cs.stop()
    assert out["samples"] == 1 and out["sm_mhz"] == 900.0


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_two_ranks():
    """Launched as for a 2-GPU run: rank 0 alone times the oracle and prints one line; the
    other rank exits 0 without work."""
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port),
                        os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "3", "--workload", "fixed_T17_H1"],
                       capture_output=True, text=True, timeout=280, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
