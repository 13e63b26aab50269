"""bench.py's reference arm on the CPU: the oracle timed on the host cores
prints one JSON line with the benchmark contract's keys; ranks other than 0
exit without work.  (The GPU arm's line is checked on a GB300 by running
bench.py itself.)"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_fp32",
                           "--steps", "1", "--warmup", "1"], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=600)


def test_reference_arm_prints_the_contract_line():
    p = _run({"RANK": "0"})
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 1
    assert d["config"]["workload"] == "tiny_fp32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    p = _run({"RANK": "1"})
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""


def test_clock_summary_reads_the_sampled_gpu_and_its_throttle_reasons(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    # nvidia-smi --format=csv,noheader,nounits rows: index, sm, max sm, power,
    # active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    rows = [
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "1, 1100, 2070, 300.0, 0x0000000000000008, Active, Not Active, Not Active, Not Active",
        "0, 2040, 2070, 1390.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2055, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, [N/A], 2070, [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]",
    ]
    p = tmp_path / "clocks.csv"
    p.write_text("\n".join(rows) + "\n")
    s = bench.ClockSampler(str(p)).summary(0)
    assert s["sm_mhz"] == 2055.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]  # GPU 1's hw_slowdown is another GPU's
    assert s["samples"] == 4
    s1 = bench.ClockSampler(str(p)).summary(1)
    assert s1["sm_mhz"] == 1100.0 and s1["reasons"] == ["hw_slowdown"]


def test_cpu_oracle_sample_extrapolation_arithmetic():
    """A workload too large for the oracle is sampled (2 of its layers, 2 of
    its sequences, block 0 and a middle block) and the whole generation's
    time extrapolated: per block one refresh and (iterations - 1) cached
    iterations at the sampled per-refresh and per-iteration times."""
    sys.path.insert(0, ROOT)
    import bench
    from block_denoising_gb300 import inputs
    cfg = inputs.shrink(inputs.LLADA_8B, n_layers=4, d_model=256, n_heads=2, ffn=512, vocab=1024, mask_id=1023)
    run = inputs.RunConfig(batch=3, prompt_len=32, gen_length=64, block_length=16, threshold=0.9)
    assert not bench.tiny_sample(cfg, run)
    ipb = [3, 1, 4, 2]
    s = bench.oracle_sample(cfg, run, ipb)
    assert s["extrapolated"] is True and s["kind"] == "oracle" and s["cores"] >= 1
    r, i = s["us_per_refresh"] * 1e-6, s["us_per_iteration"] * 1e-6
    total = 4 * r + (sum(ipb) - 4) * i
    assert s["value"] == pytest.approx(3 * 64 / total, rel=1e-9)
    assert "2 of 4 layers" in s["sample"] and "2 of 3 sequences" in s["sample"] and "block 2" in s["sample"]
    u = bench.oracle_sample(cfg, run, None)      # without iteration counts: an upper bound
    assert u["value"] == pytest.approx(3 * 64 / (4 * u["us_per_refresh"] * 1e-6), rel=1e-9)


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    """Without nvidia-smi (here) the sampler records nothing and the summary
    reports no clocks instead of failing the run."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("PATH", str(tmp_path))
    with bench.ClockSampler(str(tmp_path / "c.csv")) as c:
        pass
    s = c.summary(0)
    assert s["sm_mhz"] is None and s["reasons"] == []
