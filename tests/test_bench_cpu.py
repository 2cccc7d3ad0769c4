"""Host-side pieces of the benchmark on CPU: the reference arm's JSON line
(the oracle timed on the host cores) and the clock-sample parser that decides
whether a timed region saw a throttle reason."""
import json
import os
import subprocess
import sys
import tempfile
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

CONTRACT_KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                 "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                 "cpu_baseline", "e2e")


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    t0 = time.perf_counter()
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3", "--ref-units", "4"], env=env,
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in CONTRACT_KEYS:
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["higher_is_better"] is False
    assert line["value"] > 0 and line["steps"] == 1 and line["warmup"] == 3
    assert line["config"]["workload"] == bench.WORKLOAD
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == line["value"]
    assert "4 of" in cpu["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # ms_per_step is the wall time of the sample that ran (it fits in the process's
    # own run time); value is that sample scaled to a whole layer-call
    wall_ms = (time.perf_counter() - t0) * 1e3
    assert 0 < line["ms_per_step"] * line["steps"] < wall_ms
    assert line["config"]["value_scale"] == pytest.approx(2048 / 4)
    assert line["value"] > line["ms_per_step"] * 1e3


def test_job_value_is_the_whole_jobs_time_per_layer_call():
    # one rank: 300 steps of 24 layer-calls in 620 ms
    assert bench.job_us_per_layer_call(620.0, 300, 24, 1) == pytest.approx(620e3 / 7200)
    # weak scaling: each of 4 ranks does the same work in the same time, so the
    # job does four times the layer-calls per microsecond
    one = bench.job_us_per_layer_call(620.0, 300, 24, 1)
    assert bench.job_us_per_layer_call(620.0, 300, 24, 4) == pytest.approx(one / 4)


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _parse(rows):
    s = bench.ClockSampler(0)
    s.proc = _DoneProc()
    s.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    s.file.write("\n".join(rows) + "\n")
    return s.stop()


def test_clock_samples_without_throttle():
    rows = [f"0, {mhz}, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, "
            f"Not Active" for mhz in (2070, 2055, 2070)]
    got = _parse(rows)
    assert got["sm_mhz"] == 2070 and got["sm_max_mhz"] == 2070
    assert got["reasons"] == [] and got["samples"] == 3
    assert got["power_w_max"] == 900.5


def test_clock_samples_report_each_active_reason_once():
    rows = [
        "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1500, 2070, 1200.0, 0x48, Not Active, Active, Not Active, Active",
        "0, 2070, 2070, 800.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 800.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    got = _parse(rows)
    assert got["samples"] == 3
    assert got["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert got["sm_mhz"] == 1980


def test_clock_sampler_without_nvidia_smi_reports_nothing():
    s = bench.ClockSampler(0)
    assert s.stop() is None


def test_algorithmic_bytes_follow_the_per_unit_formulas():
    """The roofline's byte count: per unit (request, head), with dk = dv = 128,
    bf16 q/k/v and fp32 gates, state and o,
      verify = 65536 + T (768 + 8) + T 512
      commit = [a > 0] 2 * 65536 + a (512 + 8)
      fused  = 65536 + [a > 0] 65536 + T (768 + 8 + 512)
    plus per-request metadata; bf16 o halves the o term."""
    from speculative_decode_gated_gb300 import inputs
    prob = inputs.make_custom(batch=3, heads=2, dk=128, dv=128, lengths=[16, 5, 9],
                              qkv_dtype="bf16", pool_slots=4, accepted=[0, 5, 3], seed=1,
                              name="bytes")
    T, a, H, B = prob.lengths.astype(int), prob.accepted.astype(int), 2, 3
    ragged_meta = 4
    verify = H * sum(65536 + t * (768 + 8) + t * 512 for t in T) + B * (4 + ragged_meta)
    commit = H * sum((x > 0) * 2 * 65536 + x * (512 + 8) for x in a) + B * (4 + 4 + ragged_meta)
    fused = H * sum(65536 + (x > 0) * 65536 + t * (768 + 8 + 512) for t, x in zip(T, a)) \
        + B * (4 + 4 + ragged_meta)
    assert bench.alg_bytes(prob, "verify") == verify
    assert bench.alg_bytes(prob, "commit") == commit
    assert bench.alg_bytes(prob, "fused") == fused
    assert bench.alg_bytes(prob, "verify", o_bytes=2) == verify - H * sum(T) * 128 * 2


def test_single_layer_workloads_cycle_instances_past_l2():
    """A single-layer workload runs as independent instances, all verifies
    before all commits, so that between an instance's verify and its commit
    the other instances' verifies move more than the 129 MB L2 (its
    checkpoints are then read from HBM again, as between layers in an
    engine); the multi-layer workload keeps its own layers."""
    from speculative_decode_gated_gb300 import inputs
    l2 = 129e6
    assert bench.instances_of(bench.WORKLOAD) == 1
    with pytest.raises(SystemExit):
        bench.instances_of(bench.WORKLOAD, 2)
    assert bench.instances_of("b32_h32_d128_t16", 1) == 1
    for name, _ in bench.PER_CONFIG:
        assert bench.instances_of(name) == bench.INSTANCES[name]
    for name, n in bench.INSTANCES.items():
        assert "layers" not in inputs.WORKLOADS[name]
        prob = inputs.make_problem(name)
        checkpoints = prob.units * prob.dk * prob.dv * 4
        if "ragged" in name:  # fused calls: an instance's next call follows the others' calls
            assert (n - 1) * bench.alg_bytes(prob, "fused") > l2 or checkpoints > 2 * l2
        else:
            assert checkpoints < l2 and (n - 1) * bench.alg_bytes(prob, "verify") > l2
