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
