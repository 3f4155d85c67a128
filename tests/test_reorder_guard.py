"""bsa_reorder_guard: the row-reordering decision (host arithmetic, no GPU).

The guard estimates the forward's latency for the input order, the NNZ wave
sort and the spectral order plus wave sort, and keeps the input order unless
a reordering's saving beats its cost (WaveAlign, "A. Design Rationale" and
"E. Runtime Coordination").  These checks run the C entry point with the L2
size given, so no device is queried.
"""
import ctypes

import pytest

import long_context_mask_gb300 as bsa
from long_context_mask_gb300 import binding

GB300_L2 = 126.5e6
H100_L2 = 50e6


def guard(**kw):
    return bsa.reorder_guard(**kw)


def pairs(heads, nb, density):
    return int(heads * nb * nb * density)


@pytest.mark.parametrize("name,args,order", [
    # threshold-map workload: one head's K/V (16.8 MB) fits the L2 share
    ("threshold", dict(heads=12, nqb=256, nkb=256, D=128, listed_blocks=210699), "input"),
    # dynamic workload: 60.8 MB per head, still inside half of GB300's L2
    ("dynamic", dict(heads=24, nqb=928, nkb=928, D=128, listed_blocks=3094000), "input"),
    # long video: 205.5 MB per head, reuse must come from the row order
    ("long video", dict(heads=2, nqb=3136, nkb=3136, D=128, listed_blocks=2950000), "wave"),
])
def test_decisions_on_the_gb300_workloads(name, args, order):
    r = guard(l2_bytes=GB300_L2, tensor_tflops=1500, hbm_gbs=6790, **args)
    assert r["order"] == order, (name, r)


def test_page_sequence_lengths_on_h100():
    """WaveAlign "F. Other Factors": reordering skipped at 25K, 49K and 98K
    tokens and enabled from 197K (Wan2.1, 40 heads of 128, H100's 50 MB L2);
    the overhead is taken as a few percent of the attention call."""
    decisions = {}
    for kt in (25, 49, 98, 197, 401):
        nb = kt * 1000 // 128
        listed = pairs(40, nb, 0.15)
        t = listed * 4 * 128 * 128 * 128 / 600e12 * 1e3  # ms at 600 TFLOP/s
        r = guard(heads=40, nqb=nb, nkb=nb, D=128, listed_blocks=listed, l2_bytes=H100_L2,
                  tensor_tflops=600, hbm_gbs=3350, wave_ms=0.02 * t, spectral_ms=0.03 * t)
        decisions[kt] = r["order"]
    assert decisions == {25: "input", 49: "input", 98: "input", 197: "wave", 401: "wave"}


def test_fitting_kv_is_never_reordered():
    for nb in (16, 128, 400):
        r = guard(heads=8, nqb=nb, nkb=nb, D=128, listed_blocks=pairs(8, nb, 0.3), l2_bytes=1e9,
                  wave_ms=0.0, spectral_ms=0.0)
        assert r["miss_fraction"] == 0.0
        assert r["order"] == "input"
        assert r["t_input_ms"] == r["t_wave_ms"] == r["t_spectral_ms"]


def test_gain_grows_with_density_and_shrinking_l2():
    nb = 3136
    gains = []
    for d in (0.02, 0.07, 0.15, 0.3):
        r = guard(heads=2, nqb=nb, nkb=nb, D=128, listed_blocks=pairs(2, nb, d), l2_bytes=GB300_L2)
        gains.append(r["t_input_ms"] - r["t_wave_ms"])
    assert all(b >= a for a, b in zip(gains, gains[1:])) and gains[-1] > 0
    misses = [guard(heads=2, nqb=nb, nkb=nb, D=128, listed_blocks=1000, l2_bytes=l2)["miss_fraction"]
              for l2 in (1e9, 200e6, 100e6, 50e6)]
    assert misses == sorted(misses) and misses[0] == 0.0 and misses[-1] > 0.8


def test_density_skip_with_a_fixed_overhead():
    """A fixed per-call overhead (the page's reorderers cost milliseconds)
    skips reordering at low densities and keeps it at high ones, as in
    "F. Other Factors" (skipped at 1.7 % and 6.7 %, enabled from 14.5 %)."""
    nb = 401408 // 128
    orders = {}
    for d in (0.017, 0.067, 0.145, 0.3):
        r = guard(heads=40, nqb=nb, nkb=nb, D=128, listed_blocks=pairs(40, nb, d), l2_bytes=H100_L2,
                  tensor_tflops=600, hbm_gbs=3350, wave_ms=60.0, spectral_ms=60.0)
        orders[d] = r["order"]
    assert orders[0.017] == "input" and orders[0.3] != "input"
    assert list(orders.values()).index("wave") <= 2  # enabled by 14.5 %


def test_costs_and_the_spectral_stage():
    base = dict(heads=2, nqb=3136, nkb=3136, D=128, listed_blocks=2950000, l2_bytes=GB300_L2,
                tensor_tflops=6000, hbm_gbs=6790)
    # still memory bound after the wave sort at this tensor rate: the spectral
    # stage's larger cut pays when it is cheap
    assert guard(wave_ms=0.01, spectral_ms=0.01, **base)["order"] == "spectral"
    # and not when it costs more than it saves
    assert guard(wave_ms=0.01, spectral_ms=1e3, **base)["order"] == "wave"
    # nothing pays when both are dearer than the whole call
    assert guard(wave_ms=1e4, spectral_ms=1e4, **base)["order"] == "input"
    # negative costs ask for the estimate, which is small and positive
    r = guard(**base)
    assert 0 < r["wave_cost_ms"] < r["spectral_cost_ms"] < 5


def test_rejects_bad_arguments():
    lib = binding.load_library()
    r = binding.GuardResult()
    for bad in (dict(heads=0), dict(kv_heads=3), dict(nQB=0), dict(D=0), dict(listed_blocks=-1),
                dict(l2_bytes=-1.0), dict(hbm_gbs=float("nan"))):
        a = dict(heads=2, kv_heads=2, nQB=4, nKB=4, D=64, listed_blocks=4, l2_bytes=1e6,
                 tensor_tflops=0.0, hbm_gbs=0.0, wave_ms=-1.0, spectral_ms=-1.0)
        a.update(bad)
        args = binding.GuardArgs(*[a[f] for f, _ in binding.GuardArgs._fields_])
        assert lib.bsa_reorder_guard(ctypes.byref(args), ctypes.byref(r)) == 1, bad
    assert lib.bsa_reorder_guard(None, ctypes.byref(r)) == 1
