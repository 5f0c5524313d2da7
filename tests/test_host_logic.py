"""Host-side arithmetic of the benchmark and the binding (no GPU): the
algorithmic byte counts the roofline divides by, the workloads' shapes, and
the recall/acceptance summary computed from the kernels' flags."""
import torch

import bench
import synth


def test_lmhead_algorithmic_bytes():
    by, fl = bench.lmhead_algorithmic(synth.get("b32k8"))
    # W_lm + y in bf16, top-16 values/ids and lse of 256 rows
    assert by == 151936 * 2048 * 2 + 256 * 2048 * 2 + 256 * (16 * 8 + 4)
    assert fl == 2.0 * 256 * 151936 * 2048
    by8, fl8 = bench.lmhead_algorithmic(synth.get("b32k8e4m3"))
    # codes of W_lm and y, their fp32 row scales, the same outputs
    assert by8 == (151936 * 2048 + 256 * 2048 + 256 * (16 * 8 + 4) +
                   (151936 + 256) * 4)
    assert fl8 == fl


def test_stage_bytes_of_the_fused_cycle():
    w = synth.get("b32k8")
    sb = bench.stage_bytes(w, fused=True)
    assert set(sb) == {"conv+gate", "merge+pair_score+walk", "verify"}
    assert sb["verify"] == 32 * 9 * 151936 * 4
    sb8 = bench.stage_bytes(synth.get("b32k8e4m3"), fused=True)
    assert sb8["quantize_y"] == 256 * 2048 * (2 + 1) + 256 * 4


def test_verify_roofline_counts_the_rows_the_accepted_lengths_need():
    w = synth.get("b32k8")                      # T = 1: the draw row again
    row = 151936 * 4
    side = 256 * 16 * 8 + 256 * 4               # candidates, q, drafts
    assert bench.verify_algorithmic(w, 0.0) == 32 * 2 * row + side
    assert bench.verify_algorithmic(w, 3.0) == 32 * 5 * row + side
    g = synth.get("b1k8")                       # T = 0: no draw row
    assert bench.verify_algorithmic(g, 1.0) == 1 * 2 * row + 8 * 16 * 8 + 8 * 4
    r = bench.verify_roofline(w, 0.5, 25.0, 6791.4)
    assert r["bytes"] == bench.verify_algorithmic(w, 0.5)
    assert r["all_rows_bytes"] == 32 * 9 * row
    assert abs(r["GB/s"] - r["bytes"] / 25e-6 / 1e9) < 1e-6
    assert abs(r["frac"] * 6791.4 - r["GB/s"]) < 1e-6
    # fewer bytes needed than all rows until every draft is accepted
    assert r["frac"] < r["frac_all_rows"]
    full = bench.verify_roofline(w, 8.0, 25.0, 6791.4)
    assert full["bytes"] > full["all_rows_bytes"]   # all rows + draw rows


def test_lmhead_strips_match_the_pair_grid():
    # 256 rows: two row tiles, CTA pairs, 76 pairs in one row group
    assert bench.lmhead_strips(synth.get("b32k8")) == 76
    # 8 rows: one row tile, single CTAs, one strip per SM
    assert bench.lmhead_strips(synth.get("b1k8")) == 152


def test_workloads():
    for name in ("b32k8e4m3", "b32k8cale4m3"):
        w = synth.get(name)
        assert w.lm_e4m3 and w.dtype == "bf16" and (w.B, w.K) == (32, 8)
        assert "E4M3" in synth.describe(w)
    assert not synth.get("b32k8").lm_e4m3
    assert bench.aggregate(100, [0.5, 0.4], 2) == (400.0, 0.5)
    assert bench.rank_seed(2, 0) != bench.rank_seed(2, 1)


def test_recall_by_position_on_flags():
    from bench import recall_by_position
    flags = torch.tensor([[1, 1, 0, 1],
                          [1, 1, 1, 1],
                          [0, 1, 1, 1]], dtype=torch.int32)
    recall, accept = recall_by_position(flags)
    assert recall.tolist() == [2 / 3, 1.0, 2 / 3, 1.0]
    # leading runs of candidates that hold the target token: 2, 4, 0
    assert float(accept) == 2.0


def test_reference_arm_prints_one_json_line():
    """bench.py --impl reference (the oracle on the host cores) keeps the
    line's contract: metric, value, unit, impl, cpu_baseline and e2e."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run(
        [sys.executable, os.path.join(root, "bench.py"), "--impl",
         "reference", "--config", "tiny", "--steps", "1", "--warmup", "0",
         "--cpu-seconds", "1"], capture_output=True, text=True, timeout=600,
        cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["unit"] == "cycles/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny"
