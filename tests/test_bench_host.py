"""Host-side logic of bench.py (no GPU): the clock summary that decides whether a timed run is kept,
the flop counts the TFLOP/s figures divide by, and the oracle's row sampling."""
import numpy as np
import pytest

import bench


def _line(sm, mx, hw="Not Active", hw_th="Not Active", sw_th="Not Active", cap="Not Active"):
    # index, clocks.sm, clocks.max.sm, power.draw, active mask, then the four reasons
    return f"0, {sm}, {mx}, 1200.5, 0x0, {hw}, {hw_th}, {sw_th}, {cap}"


def test_clock_summary_median_max_and_reasons():
    cs = bench.ClockSampler(0)
    cs.lines = [_line(1950, 2070), _line(2010, 2070, cap="Active"), _line(1990, 2070),
                "garbage", "0, [N/A], 2070, 0, 0x0, a, b, c, d"]
    s = cs.summary()
    assert s["sm_mhz"] == 1990 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


@pytest.mark.parametrize("field,name", [("hw", "hw_slowdown"), ("hw_th", "hw_thermal_slowdown"),
                                        ("sw_th", "sw_thermal_slowdown")])
def test_clock_summary_reports_each_rejecting_reason(field, name):
    cs = bench.ClockSampler(0)
    cs.lines = [_line(1500, 2070, **{field: "Active"}), _line(1600, 2070)]
    assert name in cs.summary()["reasons"]


def test_clock_summary_without_samples():
    cs = bench.ClockSampler(0)
    assert cs.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}


def test_forward_flops():
    assert bench.fwd_flops(1, 32, 131072, 128, False) == 4.0 * 32 * 131072 ** 2 * 128
    assert bench.fwd_flops(1, 32, 131072, 128, True) == bench.fwd_flops(1, 32, 131072, 128, False) / 2


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("causal", [True, False])
def test_row_flops_sum_to_the_visible_pairs(layout, causal):
    """Every layout is a permutation of positions, so the rows' visible keys add up to L(L+1)/2
    per head (causal) or L^2 (not), whatever the layout."""
    B, H, L, d, n = 1, 2, 96, 64, 3
    total = sum(bench.row_flops(r, B, H, L, d, n, causal, layout) for r in range(B * H * L))
    pairs = L * (L + 1) // 2 if causal else L * L
    assert total == 4.0 * d * pairs * B * H


def test_sample_rows_are_distinct_sorted_and_in_range():
    rows = bench.sample_rows(2, 4, 1000, 500, seed=3)
    assert len(rows) == 500 and np.all(np.diff(rows) > 0)
    assert rows[0] >= 0 and rows[-1] < 2 * 4 * 1000
    assert np.array_equal(rows, bench.sample_rows(2, 4, 1000, 500, seed=3))


def test_peak_fractions_published_and_per_clock():
    """The roofline's extra denominators: NVIDIA's published dense figure always, the per-clock peak
    (SMs x 8192 flop/clock x sampled MHz) only when a clock was sampled on a device."""
    roof = {"achieved": 1250.0}
    bench.add_peak_fractions(roof, {"sm_mhz": None})
    assert roof["per_clock_peak"] is None and roof["frac_of_per_clock_peak"] is None
    assert roof["published_peak"] == 2500.0 and roof["frac_of_published_peak"] == 0.5
    assert "sparsity" in roof["published_peak_source"]
    if not __import__("torch").cuda.is_available():
        assert bench.per_clock_peak_tflops(2000.0) is None


def test_visible_tile_flops_exceed_the_algorithmic_count_by_the_diagonal_halves():
    """Zigzag at 131072 / 8 shards: 65600 tile pairs per shard and head (closed form
    (2n-1)c^2 + c(c+1), c = 64), of which 2n*c = 1024 per head are diagonal tiles, counted whole
    here and as halves in the algorithmic count."""
    vis = bench.visible_tile_flops(1, 32, 131072, 128, 8, True, "zigzag")
    assert vis == 4.0 * 32 * 8 * 65600 * 128 * 128 * 128
    alg = bench.fwd_flops(1, 32, 131072, 128, True)
    # the algorithmic count 4 B H L^2 d / 2 is the off-diagonal tiles plus half of each diagonal one
    half_diag = 4.0 * 32 * 1024 * 128 * 128 * 128 / 2
    assert vis - alg == pytest.approx(half_diag, rel=1e-12)
    # non-causal: every tile is visible and the two counts agree
    assert bench.visible_tile_flops(2, 8, 8192, 128, 8, False, "contiguous") == bench.fwd_flops(2, 8, 8192, 128, False)


def test_ring_config_cuts_the_workload_into_one_shard_per_rank():
    """Both arms of an N-rank run report this config: the workload's sequence in N shards."""
    import argparse

    from sequence_sharded_exact_gb300 import synth

    args = argparse.Namespace(step="fwd", ring_groups=2, dist_backend="nccl")
    c = bench.ring_config(synth.WORKLOADS["zigzag_gqa_128k"], 8, args)
    assert c["n_shards"] == 8 and c["L"] == 131072 and "n8" in c["workload"]
    assert "16384 tokens each" in c["parallelism"] and "2 groups of 4" in c["parallelism"]
    assert "NCCL" in c["mode"]
