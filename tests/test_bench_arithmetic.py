"""The benchmark's roofline arithmetic against figures worked out by hand from
the workload shapes: algorithmic bytes (K once, the window queries, the
gathered K / V rows read and written, the indices) and the MMA flops and exp
counts of the two score passes.  CPU only."""
import pytest

import bench
import synth


@pytest.mark.parametrize("name,score_bytes,total_bytes", [
    ("2", 33_816_576, 42_237_952),
    ("4", 268_959_744, 302_645_248),
    ("5b", 778_502_144, 786_923_520),
])
def test_algorithmic_bytes(name, score_bytes, total_bytes):
    cfg = synth.CONFIGS[name]
    assert bench.workload_bytes(cfg, synth.config_seqlens(name), 2) == (score_bytes, total_bytes)


@pytest.mark.parametrize("name,flops,exps", [
    ("2", 8.59e9, 33.6e6),
    ("4", 137.4e9, 537e6),
    ("5b", 199.2e9, 778e6),
])
def test_score_work(name, flops, exps):
    f, e = bench.score_work(synth.CONFIGS[name], synth.config_seqlens(name))
    assert f == pytest.approx(flops, rel=3e-3)
    assert e == pytest.approx(exps, rel=3e-3)


def test_score_work_skips_keep_all_sequences():
    cfg = synth.CONFIGS["2"]
    assert bench.score_work(cfg, [cfg["C"], cfg["C"] - 1]) == (0, 0)


def test_mufu_peak_is_derived_from_units_and_clock():
    _, _, mufu, kind = bench.compute_peaks(152)
    assert mufu == pytest.approx(32 * 152 * 2070e6 / 1e12)
    assert "152 SMs" in kind


def test_reference_arm_line():
    """bench.py --impl reference (the oracle on the host cores) prints one JSON
    line with the contract's keys; run on the tiny workload so it takes
    seconds."""
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--workload", "1", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("1:")
