"""Host-side accounting of bench.py (no GPU): the attended pairs of the Gather
0 layer against the oracle's query and key sets, compulsory bytes with
grouped heads, densities, and the reference arm's JSON line for the image
layer."""
import json
import os
import subprocess
import sys

import numpy as np

import bench
import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_image_pairs_match_oracle_sets():
    for h, w, nt, g in [(32, 32, 128, 2), (16, 24, 0, 1), (64, 32, 256, 8)]:
        prob = synth.image_gather0(H=1, img_h=h, img_w=w, n_text=nt, groups=g, D=64)
        pairs = sum(len(qt) * len(kt) for qt, kt in oracle.gather0_sets(h, w, nt, g))
        assert bench.image_visible_pairs(prob) == pairs
        assert bench.image_useful_flops(prob) == 4.0 * 64 * pairs
        assert np.isclose(bench.workload_density(prob, None), pairs / float(prob.N) ** 2)


def test_flux_shape_pairs():
    prob = synth.image_gather0()
    # every image query: 512 text keys + its 16 x 16 window; every text query:
    # 512 text keys + its Scatter group's 16384 / 8 image tokens
    assert bench.image_visible_pairs(prob) == 16384 * (512 + 256) + 512 * (512 + 2048)


def test_compulsory_bytes_grouped_heads():
    prob = synth.llm_window(H=4, H_kv=2, N=1024, D=128)
    q_and_o = 2 * 1 * 4 * 1024 * 128 * 2
    k_and_v = 2 * 1 * 2 * 1024 * 128 * 2
    lse = 1 * 4 * 1024 * 4
    assert bench.compulsory_bytes(prob) == q_and_o + k_and_v + lse


def test_reference_arm_image_layer_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "9",
           "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["dtype"] == "f64" and d["value"] > 0
    assert d["config"]["config_id"] == 9 and d["config"]["image"] == "128x128"
    assert "attended query-key pairs" in d["config"]["flops"]
    assert "(head, CQS)" in d["cpu_baseline"]["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_recorded_traffic_follows_the_kernel_source(monkeypatch):
    """ncu counters are reported only for the kernel they were taken on, only
    on the workload they were taken on and only in the row order used there."""
    import argparse
    with open(os.path.join(ROOT, "profiles", "forward_traffic.json")) as f:
        recs = json.load(f)
    key = sorted(recs)[0]
    rec = recs[key]
    args = argparse.Namespace(config=int(key[len("config"):]), heads=None, dense=False, crm=False,
                              scores="auto", order="auto", kv_gather="auto")
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: rec["kernel_hash"])
    assert bench.recorded_traffic(args, rec["order"]) == rec["dram_bytes_per_launch"]
    assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    other = "reordered" if rec["order"] == "identity" else "identity"
    assert bench.recorded_traffic(args, other) is None
    unrecorded = next(c for c in range(1, 10) if f"config{c}" not in recs)
    for change in (dict(heads=2), dict(dense=True), dict(order="identity"), dict(kv_gather="kernel"),
                   dict(scores="given"), dict(config=unrecorded)):
        assert bench.recorded_traffic(argparse.Namespace(**{**vars(args), **change}), rec["order"]) is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.recorded_traffic(args, rec["order"]) is None


def test_kernel_hash_ignores_comments_only(tmp_path, monkeypatch):
    """A comment edit keeps the hash; a code edit changes it."""
    src_dir = tmp_path / "long_context_mask_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    names = ("bsa_attn.cu", "bsa_ptx.cuh", "bsa_math.cuh", "bsa_gather0.cuh")
    for n in names:
        (src_dir / n).write_text("int f(int x) {\n  return x + 1;  // one\n}\n/* block */\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    (src_dir / names[0]).write_text("int f(int x) {\n  /* a note */ return x + 1;  // another\n}\n")
    assert bench.kernel_source_hash() == h0
    (src_dir / names[0]).write_text("int f(int x) {\n  return x + 2;\n}\n")
    assert bench.kernel_source_hash() != h0


def test_clock_summary_parses_samples():
    """The clocks record: median SM clock over the busy samples, the maximum,
    and every throttle reason seen active (nvidia-smi csv, no header/units)."""
    s = bench.ClockSampler("0")
    s.lines = [
        "345, 2070, 120.5, 0x0000000000000001, Not Active, Not Active, Not Active, Not Active",   # idle
        "1965, 2070, 1210.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "1980, 2070, 1190.2, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "1950, 2070, 1250.7, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "[N/A], 2070, [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]",                                # unreadable
        "garbage",
    ]
    d = s.summary()
    assert d == {"sm_mhz": 1965.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 4}
    s.lines.append("1500, 2070, 1300.0, 0x0000000000000048, Active, Not Active, Active, Not Active")
    assert s.summary()["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    s.lines = []
    assert s.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_tensor_peak_by_sequence_length():
    """A forward timed over a long back-to-back sequence (under the board's
    power limit) is compared with the sustained GEMM rate, a short one with
    the burst rate; the measured numbers are used when present."""
    peaks = {"bf16_tflops": 1909.3, "bf16_tflops_sustained": 1714.8}
    assert bench.tensor_peak(peaks, 20, 17.3) == (1714.8, "sustained")
    assert bench.tensor_peak(peaks, 20, 1.15) == (1909.3, "burst")
    assert bench.tensor_peak(peaks, 10, bench.SUSTAINED_AFTER_MS / 10) == (1714.8, "sustained")
    assert bench.tensor_peak({}, 1, 1.0) == (bench.FALLBACK_PEAKS["bf16_tflops"], "burst")
    assert bench.tensor_peak({}, 100, 10.0) == (bench.FALLBACK_PEAKS["bf16_tflops_sustained"], "sustained")


def test_cpu_baseline_full_heads(monkeypatch):
    """Workloads too large for the oracle are timed on whole heads (every
    query block of the first and the last head), not on a time budget."""
    prob = synth.CONFIGS[1]()
    monkeypatch.setattr(bench, "sample_heads", lambda p: (0, p.B * p.H - 1))
    lists = bench.host_lists(prob)
    v, s, b, threads = bench.time_oracle(prob, lists, budget_s=1e-9, full_heads=True)
    assert b == 2 * prob.nqb and v > 0 and threads >= 1
    _, _, b_budget, _ = bench.time_oracle(prob, lists, budget_s=1e-9)
    assert b_budget < b
