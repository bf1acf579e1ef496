"""The benchmark's host logic on CPU: the roofline figures it reports (algorithmic work per
launch over time, against the stated peak), the whole-step model, the kernel-launch
count it claims, and the rule that a profile's DRAM traffic is reported only while the
kernel's sources still hash to what was captured."""

import os
import sys
from types import SimpleNamespace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6000.0, "source": "measured"}
SC = SimpleNamespace(n=1000, sh_degree=3)  # 236 parameter bytes per Gaussian
N_SM, MHZ = 152, 2000.0
FP32_TFLOPS = 2.0 * 128 * N_SM * MHZ * 1e6 / 1e12
FP32_TOPS = 128 * N_SM * MHZ * 1e6 / 1e12    # an FMA is one op
SFU_OPS = 16 * N_SM * MHZ * 1e6


def test_alu_roofline_of_the_raster_calls():
    # the op model: 40 fp32 ops + 2 SFU per contributing pair backward, 14 + 1 forward,
    # against SMs x 128 lanes (x 16 for the SFU) x the clock; flops reported beside it
    assert (bench.OPS_BWD_PER_E, bench.SFU_BWD_PER_E) == (40, 2)
    assert (bench.OPS_FWD_PER_E, bench.SFU_FWD_PER_E) == (14, 1)
    E = 10_000_000
    r = bench.roofline("gs_rasterize_bwd", 0.5, SC, 700, 3000, E, 100, 200, PEAKS, N_SM, MHZ)
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
    assert r["peak"] == pytest.approx(FP32_TOPS)
    assert r["achieved"] == pytest.approx(40 * E / 0.5e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert r["sfu_frac"] == pytest.approx(2 * E / 0.5e-3 / SFU_OPS)
    assert r["flop_model"]["frac"] == pytest.approx(48 * E / 0.5e-3 / 1e12 / FP32_TFLOPS)
    f = bench.roofline("gs_rasterize_fwd", 0.25, SC, 700, 3000, E, 100, 200, PEAKS, N_SM, MHZ)
    assert f["achieved"] == pytest.approx(14 * E / 0.25e-3 / 1e12)
    assert f["flop_model"]["frac"] == pytest.approx(22 * E / 0.25e-3 / 1e12 / FP32_TFLOPS)


def test_per_call_fractions_cover_every_call():
    E = 10_000_000
    per_call = {"gs_project": 0.08, "gs_bin_sort": 0.1, "gs_rasterize_fwd": 0.2,
                "gs_rasterize_bwd": 0.4, "gs_project_bwd": 0.09}
    out = bench.per_call_fractions(per_call, SC, 600, 5000, E, 100, 100, PEAKS, N_SM, MHZ)
    assert set(out) == set(per_call)
    for call, ms in per_call.items():
        r = bench.roofline(call, ms, SC, 600, 5000, E, 100, 100, PEAKS, N_SM, MHZ)
        assert out[call] == {"bound": r["bound"], "frac": r["frac"], "ms": ms}


def test_loss_roofline_counts_window_fmas_per_pixel():
    H, W = 840, 1297
    assert bench.LOSS_FLOPS_PER_PIXEL == 3 * (5 + 3) * 2 * 11 * 2
    r = bench.roofline("gs_loss_l1_ssim", 0.1, SC, 0, 0, 0, H, W, PEAKS, N_SM, MHZ)
    assert r["bound"] == "alu"
    assert r["achieved"] == pytest.approx(bench.LOSS_FLOPS_PER_PIXEL * H * W / 0.1e-3 / 1e12)


@pytest.mark.parametrize("call,expected", [
    # visible: M = 600 of N = 1000; G = 44 + 12 * 16 = 236 bytes of parameters
    ("gs_project", 44 * 1000 + 192 * 600 + 64 * 1000),
    ("gs_project_bwd", 36 * 600 + 236 * 600 + 236 * 1000 + 5 * 1000),
    ("gs_project_bwd_adam", 36 * 600 + 5 * 1000 + 6 * 236 * 1000 + 16 * 1000),
    ("gs_bin_sort", 8 * 600 * 8 + 8 * 5000 * 5),
])
def test_hbm_roofline_bytes(call, expected):
    r = bench.roofline(call, 0.01, SC, 600, 5000, 0, 100, 100, PEAKS, N_SM, MHZ)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6000.0
    assert r["achieved"] == pytest.approx(expected / 0.01e-3 / 1e9)


def test_step_roofline_sums_the_binding_term_of_each_phase():
    M, I, E, H, W = 600, 5000, 2_000_000, 100, 100
    out = bench.step_roofline(1.0, SC, M, I, E, H, W, PEAKS, N_SM, MHZ)
    assert set(out["phases_ms"]) == {"project", "bin_sort", "forward", "backward"}
    assert out["ms"] == pytest.approx(sum(out["phases_ms"].values()))
    assert out["frac"] == pytest.approx(out["ms"] / 1.0)
    fwd_ops = bench.OPS_FWD_PER_E * E / (FP32_TOPS * 1e12) * 1e3
    assert out["phases_ms"]["forward"] >= fwd_ops * (1 - 1e-12)
    assert out["phases_ms"]["backward"] == pytest.approx(
        max(bench.OPS_BWD_PER_E * E / (FP32_TOPS * 1e12),
            bench.SFU_BWD_PER_E * E / SFU_OPS,
            (48 * I + 36 * H * W + 36 * M + 236 * M + 236 * SC.n) / 6000e9) * 1e3)
    # with few contributing pairs the backward is bound by its bytes, which Adam raises
    # (parameters and both moments read and written instead of one gradient row)
    plain = bench.step_roofline(1.0, SC, M, I, 0, H, W, PEAKS, N_SM, MHZ)
    train = bench.step_roofline(1.0, SC, M, I, 0, H, W, PEAKS, N_SM, MHZ, train=True)
    assert "loss" in train["phases_ms"] and "loss" not in plain["phases_ms"]
    assert train["phases_ms"]["backward"] > plain["phases_ms"]["backward"]


def test_kernel_launch_count_of_both_binning_paths():
    # project, policy + forward, reset + backward, chain rule: 6 kernels around the sort
    # bucket path: 10 binning kernels plus one merge round per doubling of 4096 up to
    # min(n, capacity) -- 9 rounds on the 1.5M scene, 25 launches per step as the ncu
    # launch list of that scene counts them
    assert bench.kernel_launches(1000, 4000, 128, 128) == 10 + 6
    assert bench.kernel_launches(1_500_000, 1_900_000, 1297, 840) == 10 + 9 + 6 == 25
    # long lists: the two-stage radix sort, one tile pass per 8 bits of the tile index
    # (8160 tiles at 1920 x 1080: 13 bits, 2 passes)
    assert ((120 * 68) - 1).bit_length() == 13
    assert bench.kernel_launches(3_000_000, 9 << 20, 1920, 1080) == (3 + 4 + 3 + 1 + 2 + 2 + 2) + 6


def test_profile_traffic_only_while_sources_match(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    csrc = tmp_path / "differentiable_gaussian_splatting_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("gs_raster.cu", "gs_device.cuh", "gs_internal.h"):
        (csrc / f).write_text(f"// {f}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    digest = bench.sources_digest(["gs_raster.cu", "gs_device.cuh", "gs_internal.h"])
    page = prof / "raster_bwd_kernel_scene-1.5M-1297x840.md"
    page.write_text(f"- sources_sha256: `{digest}` (as captured)\n"
                    "- traffic_bytes_per_launch: 123456\n")
    assert bench.profiled_traffic("gs_rasterize_bwd") == 123456
    (csrc / "gs_raster.cu").write_text("// changed since the capture\n")
    assert bench.profiled_traffic("gs_rasterize_bwd") is None
    assert bench.profiled_traffic("gs_bin_sort") is None  # several kernels: no single profile


def test_l2_note_and_workload_config_follow_the_scene():
    import synthetic_scenes as ss

    small, _ = ss.make_config(1)
    big, _ = ss.make_config(3, n=300_000)  # 70.8 MB of parameters
    assert bench.l2_note(small, "gradients", 1).startswith("inputs smaller than L2")
    # 2 x 70.8 MB of parameters and gradients exceed the 129 MB L2; 1 x alone would not
    assert bench.l2_note(big, "gradients", 1).startswith("inputs larger than L2 (70.8 MB")
    assert bench.l2_note(big, "moments", 2).endswith("+ 142 MB moments)")
    args = SimpleNamespace(config=1, sh_bf16=False)
    cfg = bench.workload_config(args, small, 128, 128, 5713, "single")
    assert cfg["workload"] == ss.CONFIG_NAMES[1] and cfg["tile_pairs"] == 5713
    assert cfg["gaussians"] == small.n and cfg["image"] == "128x128"
    assert bench.workload_config(SimpleNamespace(config=1, sh_bf16=True), small, 128, 128, 5713,
                                 "single")["sh_storage"] == "bf16"


def test_clock_summary_reads_nvidia_smi_lines():
    """The clocks record of a bench line: median SM clock under load, the maximum, and every
    throttle reason seen Active in any sample (lines as nvidia-smi prints them with
    --format=csv,noheader,nounits); unreadable or short lines are skipped."""
    s = bench.ClockSampler(0)
    s.lines = [
        "2070, 2070, 812.50, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "1980, 2070, 1395.10, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2055, 2070, 990.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "[N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]",
        "2070, 2070",
    ]
    out = s.summary()
    assert out == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                   "samples": 3}
    s.lines = ["1500, 2070, 700.0, 0x88, Active, Not Active, Active, Not Active"]
    assert s.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    s.lines = []
    assert s.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_imbalance_reports_the_tile_load_against_the_per_cta_share():
    st = {"resident_ctas": 760, "n_total": 1_520_000, "n_max": 10_000, "nonempty_tiles": 4000,
          "n_min_nonempty": 2, "h": 3, "k": 4, "batches_tiles": 9000, "batches_chunks": 120,
          "batches_skipped_on_flag": 30, "batches_skipped_done": 5, "batches_discarded": 7}
    out = bench.imbalance(st, 4346)
    assert out["max_over_share"] == pytest.approx(10_000 / (1_520_000 / 760))
    assert out["max_over_min"] == pytest.approx(5000)
    assert out["n_mean"] == pytest.approx(1_520_000 / 4346)
    assert out["n_mean_nonempty"] == pytest.approx(380)
    assert (out["h"], out["k"], out["batches"]["discarded"]) == (3, 4, 7)


def test_chain_rule_bytes_count_the_touched_gaussians():
    # the chain rule reads grad2d and the parameters of the Gaussians the backward
    # touched (T <= M), and writes every gradient row
    r = bench.roofline("gs_project_bwd", 0.01, SC, 600, 5000, 0, 100, 100, PEAKS, N_SM, MHZ, T=250)
    assert r["achieved"] == pytest.approx((36 * 250 + 236 * 250 + 236 * 1000 + 5 * 1000)
                                          / 0.01e-3 / 1e9)


def test_raster_roofline_without_contributing_pairs():
    # an empty view (no pixel blends anything) reports zero, not a division error
    r = bench.roofline("gs_rasterize_bwd", 0.1, SC, 0, 0, 0, 100, 100, PEAKS, N_SM, MHZ)
    assert r["achieved"] == 0 and r["frac"] == 0
