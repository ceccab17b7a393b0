"""Host-side logic of bench.py that the reported numbers rest on (CPU only):
the algorithmic byte counts behind every GB/s and roofline fraction, the
DRAM-traffic lookup keyed by the kernel sources, and the clock sampler's
throttle-reason parsing."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from nvfp4_quant_gemma_gb300.workloads import (EXTRA_WORKLOADS, HEADLINE,  # noqa: E402
                                                WORKLOADS, all_workloads)


# Bytes one call must move, worked by hand from the shapes (e = 2 bytes per
# 16-bit element): inputs once, outputs once, the weight once; NVFP4 scale
# padding (rows M..round_up(M,128)) is never written and not counted.
HAND_BYTES = {
    # x + r + r' (3·2·M·H) + q (M·H) + w (2H)
    "decode_m16_h2048_bf16_fp8": 3 * 2 * 16 * 2048 + 16 * 2048 + 2 * 2048,
    # + y (2·M·H)
    "decode_m256_h4096_bf16_fp8_y": 4 * 2 * 256 * 4096 + 256 * 4096 + 2 * 4096,
    # x, r, r', y + codes M·H/2 + scales M·H/16
    "prefill_m2048_h5120_bf16_nvfp4_y": 4 * 2 * 2048 * 5120 + 2048 * 2560 + 2048 * 320 + 2 * 5120,
    "prefill_m16384_h8192_fp16_fp8": 3 * 2 * 16384 * 8192 + 16384 * 8192 + 2 * 8192,
    "prefill_m16384_h8192_fp16_nvfp4": 3 * 2 * 16384 * 8192 + 16384 * 4096 + 16384 * 512 + 2 * 8192,
    "prefill_m16384_h8192_fp16_fp8_nores": 2 * 16384 * 8192 + 16384 * 8192 + 2 * 8192,
    "prefill_m16384_h8192_fp16_nvfp4_nores": 2 * 16384 * 8192 + 16384 * 4096 + 16384 * 512 + 2 * 8192,
    # 4 partials + r + r' + y + codes + scales
    "parts4_m4096_h7168_bf16_nvfp4_y": (4 + 3) * 2 * 4096 * 7168 + 4096 * 3584 + 4096 * 448 + 2 * 7168,
    # MXFP8: codes M·H + E8M0 scales M·H/32
    "decode_m256_h4096_bf16_mxfp8_y": 4 * 2 * 256 * 4096 + 256 * 4096 + 256 * 128 + 2 * 4096,
    "prefill_m16384_h8192_fp16_mxfp8": 3 * 2 * 16384 * 8192 + 16384 * 8192 + 16384 * 256 + 2 * 8192,
    "prefill_m16384_h8192_fp16_nvfp4_plain": 3 * 2 * 16384 * 8192 + 16384 * 4096 + 16384 * 512 + 2 * 8192,
    # norm only: x, r, r', y
    "prefill_m16384_h8192_fp16_norm_y": 4 * 2 * 16384 * 8192 + 2 * 8192,
}


def test_every_workload_has_a_hand_count():
    assert set(HAND_BYTES) == set(all_workloads())
    assert HEADLINE in WORKLOADS and not set(WORKLOADS) & set(EXTRA_WORKLOADS)


@pytest.mark.parametrize("name", sorted(HAND_BYTES))
def test_algorithmic_bytes(name):
    assert all_workloads()[name].algorithmic_bytes() == HAND_BYTES[name]


def test_headline_is_the_largest_configuration():
    wl = WORKLOADS[HEADLINE]
    assert (wl.M, wl.H, wl.dtype, wl.mode, wl.write_y, wl.residual) == (16384, 8192, "fp16", "fp8",
                                                                         False, True)
    assert wl.algorithmic_bytes() == 939540480
    assert wl.algorithmic_bytes() == max(w.algorithmic_bytes() for w in WORKLOADS.values())


def test_both_arms_report_the_same_config():
    """The GPU arm and the reference arm build `config` from the workload
    alone, so the two lines of one workload carry identical configs."""
    wl = WORKLOADS[HEADLINE]
    a = bench.workload_config(wl, 1)
    assert a == bench.workload_config(wl, 1)
    assert a["workload"] == HEADLINE and a["l2"].startswith("inputs larger than L2")
    assert bench.workload_config(wl, 2)["parallelism"] == "replicas2"
    small = bench.workload_config(WORKLOADS["decode_m16_h2048_bf16_fp8"], 1)
    assert "rotate" in small["l2"] and not small["l2"].startswith("inputs larger")


def test_kernel_names_follow_the_launch_shape():
    wl = WORKLOADS[HEADLINE]
    assert bench.kernel_name(1, 1, 4, 1, wl) == \
        "gnq::row_kernel<__half, MODE_FP8, parts=false, VPT=4, fp32>"
    nv = WORKLOADS["prefill_m16384_h8192_fp16_nvfp4_nores"]
    assert bench.kernel_name(2, 0, 4, 2, nv) == \
        "gnq::stream_kernel_nvfp4<__half, MODE_NVFP4, parts=false, VPT=4, packed>"
    assert bench.kernel_name(1, 4, 1, 1, wl).endswith("x 4-CTA cluster")


def test_link_ceiling():
    link = {"h2d_GB_s": 400.0, "d2h_GB_s": 200.0, "bidirectional_GB_s": 500.0}
    # one way: max(4e8 / 400e9, 1e8 / 200e9) = 1 ms; both ways: 5e8 / 500e9 = 1 ms
    assert abs(bench.link_ceiling(10 ** 9, 4 * 10 ** 8, 10 ** 8, link) - 1000.0) < 1e-6
    link["bidirectional_GB_s"] = 250.0   # the two directions share the link: 2 ms
    assert abs(bench.link_ceiling(10 ** 9, 4 * 10 ** 8, 10 ** 8, link) - 500.0) < 1e-6
    link["step_mix_GB_s"] = 200.0        # the step's own two copies at once: 2.5 ms
    assert abs(bench.link_ceiling(10 ** 9, 4 * 10 ** 8, 10 ** 8, link) - 400.0) < 1e-6
    link["step_mix_GB_s"] = 1000.0       # faster than the other bounds: they decide
    assert abs(bench.link_ceiling(10 ** 9, 4 * 10 ** 8, 10 ** 8, link) - 500.0) < 1e-6


@pytest.mark.parametrize("M,chunks", [(16384, 8), (16384, 1), (1000, 8), (4096, 3), (129, 2),
                                      (100, 8), (1, 4), (128 * 5, 4)])
def test_row_blocks_cover_the_rows_at_tile_starts(M, chunks):
    blocks = bench.row_blocks(M, chunks)
    assert 1 <= len(blocks) <= chunks
    assert blocks[0][0] == 0 and blocks[-1][1] == M
    for (a, e), (a2, _) in zip(blocks, blocks[1:]):
        assert e == a2 and a < e
    assert all(a % 128 == 0 for a, _ in blocks)
    # as even as 128-row tiles allow: every block but the last is equal
    assert len({e - a for a, e in blocks[:-1]}) <= 1


def test_small_batch_sweep_bases():
    from nvfp4_quant_gemma_gb300.workloads import SMALL_M, sweep_workload
    assert {1, 128, 129, 192, 8192} <= set(SMALL_M)
    for mode in ("fp8", "nvfp4"):
        wl = sweep_workload(mode, 129)
        assert (wl.M, wl.H, wl.dtype, wl.mode, wl.residual, wl.write_y) == (129, 5120, "bf16",
                                                                             mode, True, True)


def _traffic_file(tmp_path, src_hash, rows):
    f = tmp_path / "dram_traffic.txt"
    f.write_text("# comment\n" + f"kernel_sources_sha256_16 {src_hash}\n"
                 + "".join(f"{k} {v}\n" for k, v in rows.items()))
    return str(f)


def test_traffic_only_for_the_current_kernel_sources(tmp_path, monkeypatch):
    good = _traffic_file(tmp_path, bench.kernel_hash(), {HEADLINE: 4222976, "other": "null"})
    monkeypatch.setattr(bench, "TRAFFIC_FILE", good)
    assert bench.recorded_traffic(HEADLINE) == 4222976.0
    assert bench.recorded_traffic("other") is None      # recorded as unknown
    assert bench.recorded_traffic("missing") is None
    (tmp_path / "stale").mkdir()
    stale = _traffic_file(tmp_path / "stale", "0" * 16, {HEADLINE: 4222976})
    monkeypatch.setattr(bench, "TRAFFIC_FILE", stale)
    assert bench.recorded_traffic(HEADLINE) is None     # sources changed since the capture
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "absent.txt"))
    assert bench.recorded_traffic(HEADLINE) is None


def test_kernel_hash_covers_every_kernel_source():
    csrc = os.path.join(ROOT, "nvfp4_quant_gemma_gb300", "csrc")
    files = {f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh"))}
    covered = {os.path.basename(f) for f in bench.KERNEL_SOURCES}
    assert files <= covered


def _sampler(lines, uuid="GPU-a"):
    s = bench.ClockSampler(uuid)
    s.lines = lines
    return s


def _line(uuid, sm, smax, power, *active):
    flags = ["Active" if a else "Not Active" for a in active]
    return ", ".join(["0", uuid, str(sm), str(smax), str(power), "0x0"] + flags)


def test_clock_summary_median_and_reasons():
    s = _sampler([
        _line("GPU-a", 2070, 2070, 500.0, False, False, False, False),
        _line("GPU-a", 1980, 2070, 900.0, False, False, False, True),   # power cap
        _line("GPU-a", 2070, 2070, 700.0, False, False, False, False),
        _line("GPU-b", 300, 2070, 100.0, True, True, True, True),       # another GPU
        "garbage line",
    ])
    out = s.summary()
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["samples"] == 3 and out["power_w_max"] == 900.0


def test_clock_summary_flags_thermal_slowdown_and_no_samples():
    s = _sampler([_line("GPU-a", 1500, 2070, 800.0, True, False, True, False)])
    assert s.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert _sampler([]).summary()["reasons"] == ["unavailable"]
