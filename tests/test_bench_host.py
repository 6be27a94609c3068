"""Host arithmetic of bench.py: the work and byte counts the bench line's
throughput and roofline are computed from, and the rule that the recorded DRAM
traffic of the dominant GEMM kernel is reported only for the sources it was
captured on."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_gemm_flops_is_three_gemms_per_projection():
    m = bench.TOKENS
    assert bench.gemm_flops() == sum(3 * 2 * m * n * k for n, k in bench.PROJ.values())


def test_gemm_bytes_per_role():
    """Fprop: X [M,K] and W [N,K] codes, 1x128 and 128x128 scales, Y [M,N]
    bf16.  Dgrad swaps the roles of K and N on the token side; Wgrad reads
    both operands along the token axis with 128x1 scales."""
    m = bench.TOKENS
    n, k = 6144, 4096
    assert bench.gemm_algorithmic_bytes("fprop", n, k) == m * k + n * k + 4 * (m * k / 128 + n * k / 16384) + 2 * m * n
    assert bench.gemm_algorithmic_bytes("dgrad", n, k) == m * n + n * k + 4 * (m * n / 128 + n * k / 16384) + 2 * m * k
    assert bench.gemm_algorithmic_bytes("wgrad", n, k) == n * m + k * m + 4 * (m / 128) * (n + k) + 2 * n * k
    # square projection: Fprop and Dgrad move the same bytes
    assert bench.gemm_algorithmic_bytes("fprop", k, k) == bench.gemm_algorithmic_bytes("dgrad", k, k)


def test_quantiser_bytes_per_element():
    """3.03125 B per element for one code layout; the dual kernel writes both."""
    m = bench.TOKENS
    n, k = 4096, 4096
    assert bench.quant_bytes("quant_x_dual", n, k) == m * k * (2 + 1 + 1) + 2 * 4 * m * k / 128


def test_traffic_reported_only_for_captured_sources(monkeypatch):
    current = bench.gemm_sources_sha256()
    table = {f"{k}:{p}": 1000.0 * (i + 1) for i, (k, p) in enumerate(
        (k, p) for k in ("fprop", "dgrad") for p in bench.PROJ)}
    monkeypatch.setitem(bench.GEMM_TRAFFIC, "per_launch_bytes", table)
    monkeypatch.setitem(bench.GEMM_TRAFFIC, "sha256", current)
    traffic, _ = bench.gemm_traffic()
    assert traffic == sum(table.values()) / len(table)
    # a launch of the step without a capture: no figure
    monkeypatch.setitem(bench.GEMM_TRAFFIC, "per_launch_bytes", dict(list(table.items())[1:]))
    traffic, note = bench.gemm_traffic()
    assert traffic is None and note.startswith("null")
    # other sources than those captured: no figure
    monkeypatch.setitem(bench.GEMM_TRAFFIC, "per_launch_bytes", table)
    monkeypatch.setitem(bench.GEMM_TRAFFIC, "sha256", "0" * 64)
    traffic, note = bench.gemm_traffic()
    assert traffic is None and note.startswith("null")


def test_workloads_match_the_configured_shapes():
    """train-8b: the four 8B projections at 16384 tokens; train-32b: the four
    32B projections at 32768 tokens (2 x 16384)."""
    w8, w32 = bench.WORKLOADS["train-8b"], bench.WORKLOADS["train-32b"]
    assert w8["tokens"] == 16384 and w8["proj"] == {"qkv": (6144, 4096), "o": (4096, 4096),
                                                     "gate_up": (28672, 4096), "down": (4096, 14336)}
    assert w32["tokens"] == 32768 and w32["proj"] == {"qkv": (7168, 5120), "o": (5120, 5120),
                                                       "gate_up": (55296, 5120), "down": (5120, 27648)}
    assert w32["student_t"] and w32["outlier_scale"] == 100.0 and w32["dy_sigma"] == 1e-3
    # 32B step: 3 GEMMs x 2MNK over the four projections, about 95.9 TFLOP
    assert abs(bench.gemm_flops(w32["proj"], w32["tokens"]) / 1e12 - 95.9) < 0.1


def test_burst_peak_is_twice_the_bf16_burst():
    assert bench.fp8_burst_peak({"bf16_tflops": 1880.6}) == 2 * 1880.6
