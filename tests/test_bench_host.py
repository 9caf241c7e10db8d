"""CPU tests of bench.py's host-side accounting: the kernel launches it
claims per layer call match the launch lists ncu recorded for the same
workloads (the forward: router, offsets, permute, GEMMs, combine; the
backward: 19 kernels at the default and decode workloads), and the
algorithmic FLOP and byte counts follow the definitions of the counting
rules (useful FLOP exclude padding rows)."""
import sys

import pytest

from routing_permute_grouped_gb300 import ledger, synth


@pytest.fixture(scope="module")
def bench():
    import os

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench as b

    return b


@pytest.mark.parametrize("name, skinny, fp8, expect", [
    ("default", False, False, 8),      # clustered split-K router 1, offsets 2 (histograms; scan
                                       # and scatter), 2 + 2 GEMMs (the permute in the shared
                                       # GEMM1's epilogue), combine
    ("decode", True, False, 7),        # split-K router 2 (partials + reduce: E = 256), small offsets
                                       # 1, permute, 2 GEMMs, combine
    ("decode", True, True, 8),         # + the e4m3 pairs of h between the GEMMs
    ("prerouted", False, False, 6),    # no router: offsets 2, permute, 2 GEMMs, combine
    ("default", False, True, 12),      # + widening routed and shared W13, W2
    ("imbalance_x4_p128", False, False, 7),  # fused router 1, offsets 2 (48 chunks x 64 experts),
                                             # permute, 2 GEMMs, combine
    ("tiny", False, False, 7),         # split-K router 2 (8 slices), small offsets 1, permute, 2
                                       # GEMMs, combine
])
def test_forward_launch_counts(bench, name, skinny, fp8, expect):
    assert bench.forward_launches(synth.WORKLOADS[name], skinny, fp8) == expect


def test_forward_launch_counts_with_large_chunk_tables(bench):
    # chunks x experts above 8192 (256 chunks of 2048 assignments x 256
    # experts): histograms, scan and scatter as three launches
    from routing_permute_grouped_gb300.synth import MoeShape

    s = MoeShape("big_table", T=65536, d=512, d_e=128, E=256, k=8)
    assert bench.forward_launches(s, False, False) == 1 + 3 + 1 + 2 + 1


@pytest.mark.parametrize("permute, combine, expect", [
    ("layer", "kernel", 8), ("kernel", "kernel", 9), ("gather", "kernel", 8), ("gemm", "kernel", 8),
    ("layer", "fused", 7), ("kernel", "fused", 8),
])
def test_forward_launch_counts_options(bench, permute, combine, expect):
    # the default workload's stage-call options: the permute as its own kernel
    # or inside a GEMM, the combine as its own kernel or in the shared GEMM2
    assert bench.forward_launches(synth.WORKLOADS["default"], False, False, permute,
                                  combine) == expect


@pytest.mark.parametrize("name, recompute, expect", [
    ("default", True, 19), ("decode", True, 19), ("default", False, 17), ("prerouted", True, 9),
])
def test_backward_launch_counts(bench, name, recompute, expect):
    assert bench.backward_launches(synth.WORKLOADS[name], recompute=recompute) == expect


def test_useful_flops_exclude_padding():
    s = synth.WORKLOADS["default"]
    # 2 * T*k * d * 3 d_e routed + 2 * T * d * 3 d_s shared
    routed = 2 * s.A * s.d * 3 * s.d_e
    assert ledger.routed_flops(s.A, s.d, s.d_e) == routed
    assert routed == 2_886_218_022_912


def test_clock_windows_and_normalised_rate(bench):
    """ClockSampler.summary picks the samples inside a region (median SM MHz,
    the reasons seen there), and clock_normalised scales a rate by the
    maximum over the median clock of the region."""
    c = bench.ClockSampler(0)
    c.source, c.period, c.sm_max = "nvml", 0.001, 2070.0
    c.power_limit = 1400.0
    c.samples = [(0.5, 2070.0, 0, 300.0), (1.1, 1800.0, 0x4, 1390.0), (1.2, 1900.0, 0x4, 1400.0),
                 (1.3, 2000.0, 0, None), (2.5, 1500.0, 0x8, 900.0)]
    c.window("timed", 1.0, 1.4)
    s = c.summary("timed")
    assert s["samples"] == 3 and s["sm_mhz"] == 1900.0 and s["reasons"] == ["sw_power_cap"]
    assert s["power_w_median"] == 1395.0 and s["power_w_max"] == 1400.0
    assert s["power_limit_w"] == 1400.0
    assert c.summary()["reasons"] == ["hw_slowdown", "sw_power_cap"]
    roof = {"achieved": 1700.0, "peak": 1935.5}
    n = bench.clock_normalised(1.6, roof, s)
    assert abs(n["stage_ms_x_mhz"] - 1.6 * 1900.0) < 1e-9
    assert abs(n["achieved_at_max_clock"] - 1700.0 * 2070.0 / 1900.0) < 1e-9
    assert bench.clock_normalised(1.6, roof, {"sm_mhz": None}) is None


@pytest.mark.parametrize("extra", [["--pass", "train"], ["--parallel", "ep"],
                                   ["--impl", "reference"]])
def test_graph_option_is_for_the_forward_only(extra):
    """--graph records the whole-layer forward; with another pass, the
    expert-parallel layer or the reference arm the argument parser refuses it
    before any device work."""
    import os
    import subprocess

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--graph", *extra],
                       capture_output=True, text=True, timeout=300, cwd=root)
    assert r.returncode == 2 and "--graph" in r.stderr
