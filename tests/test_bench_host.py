"""bench.py's host-side accounting (no GPU): algorithmic bytes, the roofline
traffic read back from the committed ncu summaries, argument parsing."""
import os

import torch

import bench
from mixture_experts_decode_gb300 import inputs


def test_layer_bytes_count_each_distinct_expert_once():
    cfg = inputs.QWEN3
    ids = torch.tensor([[0, 1, 2, 3, 4, 5, 6, 7], [0, 1, 2, 3, 8, 9, 10, 11]], dtype=torch.int32)
    b = bench.layer_bytes(cfg, ids, 2)
    assert b["U"] == 12
    expert = cfg.I * cfg.d * 33 // 32
    assert b["gate_up"] == 12 * 2 * expert + 2 * 2 * cfg.d + 4 * 2 * cfg.k + 2 * 2 * cfg.k * cfg.I
    assert b["down"] == 12 * expert + 2 * 2 * cfg.k * cfg.I + 8 * 2 * cfg.k + 2 * 2 * cfg.d
    assert b["layer"] == 12 * 3 * expert + 4 * 2 * cfg.d + 8 * 2 * cfg.k + 4 * 2 * cfg.k * cfg.I


def test_profiled_traffic_needs_the_current_kernel_source(tmp_path, monkeypatch):
    sha = bench.kernel_source_sha()
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    (tmp_path / "gate_up_qwen3_b32.md").write_text(
        f"kernel_source_sha: {sha}\ndram_bytes_per_launch: 123456\n")
    assert bench.profiled_traffic("gate_up", "qwen3_b32") == 123456.0
    (tmp_path / "down_qwen3_b32.md").write_text("kernel_source_sha: 0000000000000000\ndram_bytes_per_launch: 1\n")
    assert bench.profiled_traffic("down", "qwen3_b32") is None      # taken on other kernel source
    assert bench.profiled_traffic("down", "qwen3_b1") is None       # no summary


def test_committed_summaries_parse():
    for kernel in ("gate_up", "down"):
        path = os.path.join(bench.PROFILES, f"{kernel}_qwen3_b32.md")
        text = open(path).read()
        assert "kernel_source_sha:" in text and "dram_bytes_per_launch:" in text
        assert "--clock-control none" in text or "capture of" in text


def test_default_arguments_are_a_short_single_gpu_run():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.impl == "ours" and a.batch == 32 and a.config == "qwen3"
    assert a.warmup >= 3 and not a.no_sweep and a.profile is None
    p = bench.parse_args(["--profile", "grouped", "--batch", "256", "--steps", "2", "--warmup", "2"])
    assert p.profile == "grouped" and p.batch == 256
