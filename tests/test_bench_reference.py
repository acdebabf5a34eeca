"""The benchmark's host-side logic, on the CPU: the reference arm (the CPU
oracle on the host cores: its JSON line, its sampler's coverage of the
experts, ranks other than 0 doing no work), the key of the stored DRAM
traffic figure, and the warm-up rule."""
import json
import os
import subprocess
import sys

import bench
from combine_counting_sort_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None, *args):
    env = dict(os.environ, **(extra_env or {}))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout


def test_reference_line_tiny_workload():
    out = _run(None, "--workload", "tiny", "--steps", "3", "--warmup", "3", "--ref-budget-s", "2")
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["steps"] == 3 and line["warmup"] == 3 and line["config"]["workload"] == "tiny"
    assert line["value"] > 0
    # value follows the estimated time of one whole step of T tokens; ms_per_step
    # is what each sampled step took, so steps x ms_per_step fits the run
    T = inputs.CONFIGS["tiny"].T
    assert abs(T / (line["ms_per_full_step_estimate"] / 1e3) - line["value"]) <= 0.01 * line["value"] + 0.01
    # (seconds_timed is printed to 10 ms, ms_per_step to 0.1 ms)
    assert line["steps"] * line["ms_per_step"] <= 1e3 * line["cpu_baseline"]["seconds_timed"] + 5.0 + line["steps"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_without_work():
    out = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--workload", "tiny", "--steps", "3",
               "--warmup", "3", "--ref-budget-s", "2")
    assert not [l for l in out.splitlines() if l.startswith("{")]


def test_sampler_times_every_nonempty_expert_once_before_repeating():
    cfg = inputs.CONFIGS["tiny"]
    s = bench.CpuSample(cfg)
    eo = s.L["expert_offset"]
    nonempty = {e for e in range(cfg.E) if eo[e + 1] > eo[e]}
    assert set(int(e) for e in s.order) == nonempty and len(s.order) == len(nonempty)
    for _ in range(len(s.order)):
        s.expert()
    s.fixed()
    assert len(s.t_experts) == len(nonempty)
    # with every expert timed once, the GEMM1 part of the estimate is their sum
    gemm_ms = s.step_ms() - 1e3 * s.t_fixed[0]
    assert abs(gemm_ms - 1e3 * sum(s.t_experts)) <= 1e-6 * gemm_ms


def test_traffic_key_follows_kernel_code_not_comments(tmp_path, monkeypatch):
    # the DRAM-traffic figure is keyed by a hash of the dominant kernel's
    # sources' code: editing a comment keeps it, editing code drops it (null
    # until recaptured); code of other kernels does not enter
    import shutil
    src = os.path.join(ROOT, "combine_counting_sort_gb300", "csrc")
    fake_root = tmp_path / "root"
    shutil.copytree(src, fake_root / "combine_counting_sort_gb300" / "csrc")
    monkeypatch.setattr(bench, "ROOT", str(fake_root))
    h0 = bench.kernel_source_hash()
    csrc = fake_root / "combine_counting_sort_gb300" / "csrc"
    other = csrc / "layout.cu"
    other.write_text(other.read_text() + "\nstatic int unused_probe;\n")
    assert bench.kernel_source_hash() == h0
    f = csrc / "gemm1.cuh"
    text = f.read_text()
    f.write_text(text + "\n// a comment\n/* another\n comment */\n")
    assert bench.kernel_source_hash() == h0
    f.write_text(text.replace("kGemmStages", "kGemmStages ", 1) + "\nstatic int unused_probe;\n")
    assert bench.kernel_source_hash() != h0


def test_bench_refuses_fewer_than_three_warmup_steps():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode != 0 and "warmup" in r.stderr


def test_roofline_peak_follows_the_timed_region():
    # a short region at full clocks is measured against the burst peak; only a
    # region long enough to hit the power cap, with the cap seen by
    # nvidia-smi, is measured against the sustained peak
    assert bench.roofline_peak_kind(0.047, {"reasons": []}) == "burst"
    assert bench.roofline_peak_kind(0.047, {"reasons": ["sw_power_cap"]}) == "burst"
    assert bench.roofline_peak_kind(1.2, {"reasons": []}) == "burst"
    assert bench.roofline_peak_kind(1.2, {"reasons": ["sw_power_cap"]}) == "sustained"
    assert bench.roofline_peak_kind(5.0, {"reasons": ["not sampled"]}) == "burst"
