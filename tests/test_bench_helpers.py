"""The benchmark's roofline arithmetic and its profiled-traffic lookup (CPU).

The roofline object reports the dominant stage (the longest per-launch
time) against the measured peak of what bounds it: the tensor pipe when the
attention's arithmetic intensity lies above the ridge point of the measured
peaks (and it computes in bf16), else HBM.  `achieved` is the algorithmic
work per launch over the stage's time, `frac` that over the peak.  The
DRAM traffic comes from the committed ncu summary only while the summary's
source hash matches the kernel source it was taken from.
"""
import hashlib
import os
from types import SimpleNamespace

import bench

PEAKS = {"hbm_gbs": 6777.3, "bf16_tflops": 1886.1}


def res(dtype, attn_bytes, attn_flops, ms):
    return {"w": SimpleNamespace(dtype=dtype),
            "work": {"draft_topk": 3_264_000, "tree_build": 0, "tree_attn": attn_bytes, "verify": 3_904_000,
                     "attn_flops": attn_flops},
            "stage_ms": ms}


def test_roofline_hbm_bound_attention():
    r = bench.roofline(res("bf16", 35_553_768, 2_049_851_392,
                           {"draft_topk": 0.0079, "tree_build": 0.011, "tree_attn": 0.0184, "verify": 0.007}),
                       PEAKS, "measured", "no-such-workload")
    assert r["kernel"] == "tree_attn" and r["bound"] == "hbm" and r["unit"] == "GB/s"
    want = 35_553_768 / 0.0184e-3 / 1e9
    assert abs(r["achieved"] - want) < 0.01
    assert abs(r["frac"] - want / PEAKS["hbm_gbs"]) < 1e-4
    assert r["traffic"] is None and r["algorithmic_per_launch"] == 35_553_768


def test_roofline_tensor_bound_attention():
    flops, nbytes = 524_192_923_648, 1_145_731_584        # intensity ~457 flop/B, above the ridge (~278)
    r = bench.roofline(res("bf16", nbytes, flops,
                           {"draft_topk": 0.35, "tree_build": 0.013, "tree_attn": 0.834, "verify": 0.237}),
                       PEAKS, "measured", "no-such-workload")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    want = flops / 0.834e-3 / 1e12
    assert abs(r["achieved"] - want) < 0.01
    assert abs(r["frac"] - want / PEAKS["bf16_tflops"]) < 1e-4
    assert r["algorithmic_per_launch"] == flops


def test_roofline_fp32_attention_is_hbm_and_dominant_stage_wins():
    flops, nbytes = 524_192_923_648, 1_145_731_584
    r = bench.roofline(res("f32", nbytes, flops,
                           {"draft_topk": 0.35, "tree_build": 0.013, "tree_attn": 0.834, "verify": 0.237}),
                       PEAKS, "measured", "no-such-workload")
    assert r["bound"] == "hbm"                            # no bf16 tensor path for fp32 inputs
    r = bench.roofline(res("bf16", nbytes, flops,
                           {"draft_topk": 0.9, "tree_build": 0.013, "tree_attn": 0.834, "verify": 0.237}),
                       PEAKS, "measured", "no-such-workload")
    assert r["kernel"] == "draft_topk" and r["bound"] == "hbm"
    assert abs(r["achieved"] - 3_264_000 / 0.9e-3 / 1e9) < 0.01


def test_profiled_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    csrc = tmp_path / "tree_speculative_decoding_eagle_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = csrc / "tree_attn_tc.cu"
    src.write_bytes(b"// kernel source, first version\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.md").write_text(
        "| stage | workload | bytes | source sha16 |\n|---|---|---|---|\n"
        f"| tree_attn | wl | 35131648 | {sha} |\n| verify | wl | 3997696 | 0000000000000000 |\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("tree_attn", "wl") == 35131648
    assert bench.profiled_traffic("tree_attn", "other") is None
    assert bench.profiled_traffic("verify", "wl") is None      # its source file is absent here
    assert bench.profiled_traffic("no_such_stage", "wl") is None
    src.write_bytes(b"// kernel source, changed since the capture\n")
    assert bench.profiled_traffic("tree_attn", "wl") is None


def test_committed_profile_rows_name_existing_stages():
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic.md")
    rows = [l for l in open(path) if l.startswith("| ") and l.count("|") == 5 and "sha16" not in l]
    stages = {l.split("|")[1].strip() for l in rows if not l.startswith("|---")}
    assert {"draft_topk", "tree_build", "tree_attn", "verify"} <= stages
