"""bench.py's host arithmetic on CPU: the roofline of a timed stage, the
algorithmic bytes of a MoE layer, the per-instantiation decode shares, the
job rate, the nvidia-smi clock record, and the guard that drops a profile's
DRAM bytes once its kernel source has changed.  Every expected value is
worked out by hand in the test or follows from a stated invariant."""
import os
import shutil
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_roofline_of_a_stage_at_either_peak():
    # 1 TFLOP at a 2000 TFLOP/s peak takes 500 us; 1 GB at 4000 GB/s takes 250 us
    r = bench._roof(flops=1e12, nbytes=1e9, seconds=1e-3, hbm=4000.0, fp4_peak=2000.0)
    assert r["tflops"] == 1000.0 and r["gbs"] == 1000.0
    assert r["frac_fp4_peak"] == 0.5
    assert r["bound"] == "tensor" and r["roofline_us"] == 500.0
    assert r["frac_roofline"] == 0.5 and r["bytes"] == 10 ** 9
    # the same stage with 4 GB: 1000 us of HBM time, so it runs at its roofline
    r = bench._roof(flops=1e12, nbytes=4e9, seconds=1e-3, hbm=4000.0, fp4_peak=2000.0)
    assert r["bound"] == "hbm" and r["roofline_us"] == 1000.0 and r["frac_roofline"] == 1.0


def test_roofline_of_the_prefill_gemm():
    # 2 M N K for M = 8192 and the fused qkv weight N = 7168, K = 5120
    flops = 2 * 8192 * 7168 * 5120
    assert flops == 601_295_421_440
    r = bench._roof(flops, 161_677_312, 0.1065e-3, 6768.1, 11348.4)
    assert r["bound"] == "tensor"
    assert abs(r["roofline_us"] - 52.99) < 0.01           # 601.3 GFLOP / 11.348 PFLOP/s
    assert abs(r["frac_fp4_peak"] - 0.4975) < 1e-4         # 5.646 / 11.348
    assert r["frac_roofline"] == r["frac_fp4_peak"]        # tensor-bound: the same fraction


class _FakeLib:
    """nvfp4_scale_bytes of the 128x4 swizzled layout: rows padded to 128, the
    16-element blocks of a row padded to 4."""

    @staticmethod
    def nvfp4_scale_bytes(rows, k):
        return -(-rows // 128) * 128 * (-(-(k // 16) // 4) * 4)


def test_moe_bytes_count_each_used_expert_once():
    E, H, I, topk = 4, 256, 128, 2
    ids = torch.tensor([[0, 2], [2, 2], [-1, 4]], dtype=torch.int32)   # experts 0 and 2; -1 and 4 dropped
    nbytes, used = bench._moe_bytes(_FakeLib, ids, 3, E, H, I, topk)
    assert used == 2
    # per expert: W13 codes 256 x 128 B + scales 256 x 16, W2 codes 256 x 64 B + scales 256 x 8
    expert = 32768 + 4096 + 16384 + 2048
    # x and out bf16 (2 x 3 x 256 x 2 B); the intermediate of 6 routes written and read once:
    # codes 6 x 64 B and scales padded to 128 rows x 8
    assert nbytes == 2 * expert + 3072 + 2 * (384 + 1024)


def test_decode_shares_weight_each_call_by_its_time():
    class WL:
        decode = [
            {"T": 1, "N": 8, "K": 128, "ncopy": 10, "bytes": 1000},
            {"T": 2, "N": 8, "K": 128, "ncopy": 30, "bytes": 1000},
            {"T": 16, "N": 8, "K": 128, "ncopy": 20, "bytes": 2000},
        ]
    times = {"T1_8x128": {"us": 1.0}, "T2_8x128": {"us": 2.0}, "T16_8x128": {"us": 3.5}}
    r = bench._decode_kernel_rooflines(WL, times, hbm=1.0)
    # two-group kernel: 10 x 1 us + 30 x 2 us = 70 us for 40 kB; 16-token kernel: 20 x 3.5 us = 70 us for 40 kB
    assert set(r) == {"gemv_ring_kernel<0, 2>", "gemv_ring_kernel<1, 3>"}
    for k in r:
        assert r[k]["share_of_decode_time"] == 0.5
        assert abs(r[k]["gbs"] - 40_000 / 70e-6 / 1e9) < 0.05
    assert bench._decode_kernel(4) == bench._decode_kernel(8) == "gemv_ring_kernel<0, 3>"


def test_job_rate_counts_every_replica():
    assert bench.job_throughput(1, 100.0, 4.0) == 25.0
    assert bench.job_throughput(4, 100.0, 4.0) == 100.0


def test_clock_record_median_max_and_reasons(tmp_path):
    p = tmp_path / "clocks.csv"
    na, act = "Not Active", "Active"
    rows = [
        f"0, 2070, 2070, 910.5, 0x0, {na}, {na}, {na}, {na}",
        f"0, 1980, 2070, 1390.2, 0x4, {na}, {na}, {na}, {act}",
        "0, [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]",   # unreadable sample: skipped
        f"0, 2055, 2070, 1200.0, 0x0, {na}, {na}, {na}, {na}",
    ]
    p.write_text("\n".join(rows) + "\n")
    s = bench.ClockSampler(0)
    s.path = str(p)
    out = s.summary()
    assert out["samples"] == 3 and out["sm_mhz"] == 2055.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    p.write_text(f"0, 1500, 2070, 800.0, 0x8, {na}, {act}, {na}, {na}\n")
    assert bench.ClockSampler.summary(s)["reasons"] == ["hw_thermal_slowdown"]


def test_profile_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    src = tmp_path / "kern.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    git = shutil.which("git")
    if git is None:
        pytest.skip("git is not installed")
    blob = subprocess.run([git, "hash-object", str(src)], capture_output=True, text=True, check=True).stdout.strip()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "k.md").write_text(
        f"# k\n\nsource-blob: kern.cu {blob}\ndram-bytes-per-launch: 12345\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._profile_traffic("k.md") == 12345          # the capture's source, unchanged
    src.write_bytes(b"__global__ void k() { }\n")
    assert bench._profile_traffic("k.md") is None            # edited since the capture
    assert bench._profile_traffic("missing.md") is None
