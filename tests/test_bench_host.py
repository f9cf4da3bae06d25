"""The bench's host-side arithmetic on the CPU: the algorithmic byte and flop
counts its rooflines divide by, the per-launch statistics, the rotation
depth, and the rule that the GEMM's DRAM traffic from the committed ncu
capture is reported only while the kernel source is the one captured."""

import json
import os
import shutil

import pytest

import bench
from mxfp8_norm_quant_gb300 import workloads as W


def test_byte_and_flop_counts():
    # norm-quant of the 32768 x 6144 residual: x in (2 B), codes out (1 B),
    # F8_128x4 scales (6144 / 32 = 192 columns, 128-row blocks), w once
    assert bench.norm_quant_bytes(32768) == 2 * 32768 * 6144 + 32768 * 6144 + 32768 * 192 + 2 * 6144
    assert bench.norm_quant_bytes(100) == 2 * 100 * 6144 + 100 * 6144 + 128 * 192 + 2 * 6144  # padded rows
    assert bench.norm_rowmajor_bytes(100) == 3 * 100 * 6144 + 100 * 192 + 2 * 6144
    assert bench.norm_bf16_bytes(100) == 4 * 100 * 6144 + 2 * 6144
    assert bench.quant_bytes(32768, 3072) == 3 * 32768 * 3072 + 32768 * 96
    assert bench.quant_bytes(1, 32) == 3 * 32 + 128 * 4                                  # 1 column padded to 4
    assert bench.gemm_flops(32768, 6144, 3072) == 2.0 * 32768 * 6144 * 3072
    # A, its scales, W, its scales, bf16 C
    assert bench.gemm_bytes(32768, 6144, 3072) == (32768 * 3072 + 32768 * 96 + 6144 * 3072 + 6144 * 96
                                                   + 2 * 32768 * 6144)


def test_per_launch_stats_and_rotation():
    med, lo, hi = bench.per_launch_stats([2.0, 1.0, 3.0], 10)           # ms per replay of 10 launches
    assert (med, lo, hi) == pytest.approx((200.0, 100.0, 300.0))       # us per launch
    assert bench.rotation(10 ** 12) == 20                                # at least 20 launches
    small = bench.rotation(1 << 20)
    assert small * (1 << 20) > 2.2 * bench.L2_BYTES                      # a replay moves more than 2.2x L2


def test_config_names_the_workload():
    cfg = bench.make_config(W.get_workload("m32768_stress"), 1)
    assert cfg["workload"] == "m32768_stress" and cfg["M"] == 32768 and cfg["N"] == 6144
    assert "model" not in cfg


def test_gemm_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "k_gemm_mxf8_traffic.json")))
    want = rec["workloads"]["m32768_stress"]["dram_bytes_per_launch"]["3072"]
    assert bench.gemm_traffic_per_launch("m32768_stress", 3072) == want
    assert bench.gemm_traffic_per_launch("m1024", 3072) is None          # no capture of that workload
    # a copy of the tree whose kernel source differs by one byte: no traffic
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    shutil.copy(os.path.join(bench.ROOT, "profiles", "k_gemm_mxf8_traffic.json"), root / "profiles")
    for f in rec["source_files"]:
        dst = root / f
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, f), dst)
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.gemm_traffic_per_launch("m32768_stress", 3072) == want
    with open(root / rec["source_files"][0], "ab") as fh:
        fh.write(b"\n")
    assert bench.gemm_traffic_per_launch("m32768_stress", 3072) is None
