"""CPU checks of the benchmark's host-side arithmetic: the per-call flop and byte
counts behind `value` and `roofline`, the traffic digest guard, and the clock
record parsing that decides whether a run is kept."""
import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from precision_grouped_gemm_gb300 import workloads as wl  # noqa: E402
from precision_grouped_gemm_gb300.layer import FP8_STEP_NAMES, fp8_layer_work, layer_work, mx_layer_work  # noqa: E402


def test_bf16_layer_work_deepseek_shape():
    # M = 24576 rows, H = 4096, I = 2048, G = 256: every tensor moved once, bf16
    M, G, Hd, I = 24576, 256, 4096, 2048
    w = layer_work(M, G, Hd, I)
    W1 = G * 2 * I * Hd * 2
    assert w["fc1_fwd_swiglu"][0] == 2.0 * M * 2 * I * Hd
    assert w["fc1_fwd_swiglu"][1] == M * Hd * 2 + W1 + M * I * 2 + M * 2 * I * 2 + 4 * G
    assert w["fc1_wgrad"][1] == M * Hd * 2 + M * 2 * I * 2 + W1 + 4 * G
    total_flops = sum(v[0] for v in w.values())
    assert total_flops == pytest.approx(18.0 * M * I * Hd)               # the metric's flop count
    assert total_flops / 1e12 == pytest.approx(3.711, abs=1e-3)
    assert sum(v[1] for v in w.values()) / 1e9 == pytest.approx(41.2, abs=0.05)
    lens, _ = wl.DSV4_BF16.group_lens()
    assert bench.layer_flops(lens, wl.DSV4_BF16) == pytest.approx(total_flops)


@pytest.mark.parametrize("fmt,c", [("e4m3", 1.0), ("e2m1", 0.5)])
def test_mx_layer_work_matches_bf16_flops_and_scales_bytes(fmt, c):
    M, G, Hd, I = 24576, 256, 4096, 2048
    M_pad = G * 128
    bf, mx = layer_work(M, G, Hd, I), mx_layer_work(fmt, M, G, Hd, I, M_pad)
    assert sum(v[0] for v in mx.values()) == pytest.approx(sum(v[0] for v in bf.values()))
    q = c + 1.0 / 32
    # the weight stream of the forward GEMMs shrinks from 2 B to q B per element
    W1 = G * 2 * I * Hd
    assert mx["fc1_fwd_swiglu"][1] - bf["fc1_fwd_swiglu"][1] == pytest.approx(
        (M * Hd + W1) * (q - 2) + M * I * q)
    # the column-wise quantizers read bf16 and write transposed codes; padding is not counted
    assert mx["q_x_col"][1] == M * Hd * 2 + Hd * M * q + 4 * G
    assert mx["fc1_wgrad"][1] == (2 * I + Hd) * M * q + W1 * 2 + 4 * G
    assert mx_layer_work(fmt, M, G, Hd, I, 2 * M_pad) == mx              # independent of the padding


def test_fp8_layer_work_matches_mxfp8_without_scales():
    # the FP8 tensor-wise layer does the same GEMMs as MXFP8 with no per-block scale bytes, plus
    # one read of each current-scaled tensor for its amax
    M, G, Hd, I = 24576, 256, 4096, 2048
    M_pad = G * 128
    f8, mx = fp8_layer_work(M, G, Hd, I, M_pad), mx_layer_work("e4m3", M, G, Hd, I, M_pad)
    assert tuple(f8) == FP8_STEP_NAMES
    assert sum(v[0] for v in f8.values()) == pytest.approx(sum(v[0] for v in mx.values()))
    W1 = G * 2 * I * Hd
    assert f8["fc1_fwd_swiglu"][1] == M * Hd + W1 + M * I * 2 + M * 2 * I * 2 + 4 * G
    assert mx["fc1_dgrad"][1] - f8["fc1_dgrad"][1] == pytest.approx((M * 2 * I + W1) / 32)
    assert f8["q_x_col"][1] == M * Hd * 2 + Hd * M + 4 * G
    assert fp8_layer_work(M, G, Hd, I, 2 * M_pad) == f8
    assert sum(f8[n][1] for n in ("s_x", "s_a", "s_dy", "s_dh")) == 2 * M * (Hd + I + Hd + 2 * I)
    assert bench.PEAK_RATIO["fp8"] == bench.PEAK_RATIO["e4m3"] and bench.ARITH["fp8"] == "e4m3"
    # library kernels per FP8 step: one per tensor scale, quantization and GEMM
    assert sum(bench.KERNELS_PER_CALL.get(n, 1) for n in FP8_STEP_NAMES) == 18


def test_kernel_traffic_only_for_matching_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps(
        {"source_digests": {"bf16": "abc", "mx": "def"},
         "workloads": {"W": {"fc1_wgrad": {"dram_bytes_per_launch": 123.0, "family": "bf16"}},
                       "Q": {"fc1_wgrad": {"dram_bytes_per_launch": 456.0, "family": "mx"},
                             "fc2_fwd": {"dram_bytes_per_launch": 789.0}}}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    import precision_grouped_gemm_gb300.build as build
    now = {"bf16": "abc", "mx": "def"}
    monkeypatch.setattr(build, "source_digest", lambda family: now[family])
    assert bench.kernel_traffic("W", "fc1_wgrad") == 123.0
    assert bench.kernel_traffic("Q", "fc1_wgrad") == 456.0
    assert bench.kernel_traffic("W", "fc2_wgrad") is None
    assert bench.kernel_traffic("Q", "fc2_fwd") is None       # no family recorded: not trusted
    now["mx"] = "changed"                                     # only the MX sources changed
    assert bench.kernel_traffic("W", "fc1_wgrad") == 123.0
    assert bench.kernel_traffic("Q", "fc1_wgrad") is None
    now["bf16"] = "changed"
    assert bench.kernel_traffic("W", "fc1_wgrad") is None


def test_digest_families_cover_the_kernels():
    # each family's digest changes with its own kernel sources and ignores the other family's
    import precision_grouped_gemm_gb300.build as build
    srcs = {n for n in os.listdir(build.CSRC) if n.endswith((".cu", ".cuh", ".h"))}
    assert {"gemm_bf16.cu", "gemm_bf16.cuh"} <= srcs - set(build.DIGEST_EXCLUDE["bf16"])
    assert {"gemm_mx.cu", "mx_quant.cu"} <= srcs - set(build.DIGEST_EXCLUDE["mx"])
    for fam in build.DIGEST_EXCLUDE:
        assert set(build.DIGEST_EXCLUDE[fam]) <= srcs
        assert len(build.source_digest(fam)) == 16
    assert build.source_digest("bf16") != build.source_digest("mx")


def test_clock_samples_parse_reasons_and_median():
    lines = [
        "0, 2062, 2070, 1003.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1995, 2070, 1398.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 640.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    r = bench.parse_clock_samples("\n".join(lines))
    assert r["samples"] == 3 and r["sm_mhz"] == 2062.0 and r["sm_max_mhz"] == 2070.0
    assert r["power_w_max"] == 1398.0 and r["reasons"] == ["sw_power_cap"]
    bad = bench.parse_clock_samples("0, 1400, 2070, 900, 0x8, Active, Not Active, Not Active, Not Active")
    assert bad["reasons"] == ["hw_slowdown"]
    assert bench.parse_clock_samples("")["sm_mhz"] is None


def test_generator_values_are_bounded_below_the_fp8_plants():
    # gen_f32 maps a sum of four 16-bit fields (0 .. 262140) to (s - 131070) * std / 37837.23,
    # so |v| <= 3.4641 std; the FP8 full-size test plants one element above that bound in each
    # current-scaled tensor, which makes the plant the tensor's amax
    import torch
    bound = 131070 / wl._IH4_SD
    assert bound == pytest.approx(3.4641, abs=1e-4)
    v = wl.gen_f32(wl.KEY_X, torch.arange(2048), 1024, 1.0, 7).abs()
    assert float(v.max()) <= bound and float(v.max()) > 0.6 * bound
    vb = wl.gen_bf16(wl.KEY_W1, torch.arange(2048), 1024, 0.02, 7).float().abs()
    assert float(vb.max()) <= bound * 0.02 * (1 + 2.0 ** -8)    # bf16 rounding at most half an ulp up
    for std, plant in ((1.0, 8.0), (0.02, 0.25), (0.5, 4.0), (0.25, 2.0)):
        assert bound * std * (1 + 2.0 ** -8) < plant
