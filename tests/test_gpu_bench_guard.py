"""The benchmark's step takes the row order the reorder guard picks
(WaveAlign, "A. Design Rationale", "E. Runtime Coordination"): it measures the
listed blocks, the forward's rate and the reordering costs on the GPU, asks
bsa_reorder_guard, and reports the decision in its JSON line."""
import argparse
import json
import os
import subprocess
import sys

import pytest
import torch

import bench
import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _choose(prob, pooled):
    args = argparse.Namespace(crm=False, kv_gather="auto")
    peaks, _ = bench.load_peaks()
    flush = torch.empty(bench.L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    return bench.choose_order(prob, torch.device("cuda"), args, pooled, peaks, flush)


def test_kv_that_fits_l2_keeps_the_input_order():
    order, g = _choose(synth.threshold(H=4), pooled=False)
    assert g["miss_fraction"] == 0.0
    assert g["order"] == "input" and order == "identity"
    assert g["listed_blocks"] > 0 and g["measured_forward_ms_input_order"] > 0


def test_kv_beyond_l2_is_reordered():
    """One head of the 401K-token long-video workload: its K/V (205 MB) exceed
    the L2 share, and at the measured rates the wave sort pays."""
    prob = synth.long_video(H=1)
    order, g = _choose(prob, pooled=True)
    assert g["miss_fraction"] > 0.3
    assert g["order"] in ("wave", "spectral")
    assert order == bench.ORDER_OF_GUARD[g["order"]]
    assert g["t_wave_ms"] + g["wave_cost_ms"] < g["t_input_ms"]


def test_bench_line_reports_the_guard_decision():
    r = subprocess.run([sys.executable, "bench.py", "--config", "2", "--heads", "2", "--steps", "3",
                        "--warmup", "3", "--no-cpu-baseline"], cwd=ROOT, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    ro = line["row_order"]
    assert ro["chosen_by"] == "reorder guard"
    assert ro["order"] == bench.ORDER_OF_GUARD[ro["guard"]["order"]] == "identity"
    assert set(ro["forward_ms"]) == {"identity", "reordered"}
