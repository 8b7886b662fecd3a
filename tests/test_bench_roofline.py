"""bench.py's roofline arithmetic on the host: the bound follows the ridge
(arithmetic intensity against peak FLOP/s over peak bytes/s), achieved is the
algorithmic work over the measured time, and a tensor-bound line takes the
sustained bf16 peak only when its timed loop ran under the power cap."""
import pytest

import bench
from all_gather_gemm_agmm_gb300.inputs import WORKLOADS

PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}


def test_decode_is_hbm_bound():
    w = WORKLOADS["c2_decode"]
    assert w.flops / w.unique_bytes < PEAKS["bf16_tflops"] * 1e12 / (PEAKS["hbm_gbs"] * 1e9)
    s = 10e-6
    r = bench.roofline_of(w, s, PEAKS, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(w.unique_bytes / s / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / PEAKS["hbm_gbs"])
    # the power-cap switch concerns the tensor peak only
    assert bench.roofline_of(w, s, PEAKS, "measured", sustained=True)["peak"] == PEAKS["hbm_gbs"]
    # roofline time: the unique bytes at the copy bandwidth
    assert r["roofline_time_us"] == pytest.approx(w.unique_bytes / (PEAKS["hbm_gbs"] * 1e9) * 1e6)


@pytest.mark.parametrize("sustained", [False, True])
def test_prefill_is_tensor_bound(sustained):
    w = WORKLOADS["c4_prefill"]
    s = 1.2e-3
    r = bench.roofline_of(w, s, PEAKS, "measured", sustained=sustained)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(w.flops / s / 1e12)
    peak = PEAKS["bf16_tflops_sustained"] if sustained else PEAKS["bf16_tflops"]
    assert r["peak"] == peak
    assert r["frac"] == pytest.approx(r["achieved"] / peak)
    assert r["frac_of_burst"] == pytest.approx(r["achieved"] / PEAKS["bf16_tflops"])
    assert r["frac_of_sustained"] == pytest.approx(r["achieved"] / PEAKS["bf16_tflops_sustained"])
    assert r["peak_kind"].startswith("sustained" if sustained else "burst")
    assert r["flops_per_launch"] == 2 * 16384 * 8192 * 7168


def test_no_sustained_figure_keeps_burst():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0}
    r = bench.roofline_of(WORKLOADS["c4_prefill"], 1.2e-3, peaks, "measured", sustained=True)
    assert r["peak"] == peaks["bf16_tflops"] and r["peak_kind"] == "burst"


def test_sweep_bounds_split_at_the_ridge():
    # with the measured peaks' ridge (~278 FLOP/B) the sweep's M <= 256 points
    # are HBM-bound and the rest tensor-bound
    peaks, _ = bench.load_peaks()
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    for name, w in WORKLOADS.items():
        if not name.startswith("sweep_"):
            continue
        bound = bench.roofline_of(w, 1e-3, peaks, "measured")["bound"]
        assert bound == ("hbm" if w.flops / w.unique_bytes < ridge else "tensor")
        assert (bound == "hbm") == (w.M <= 256), name


def test_sweep_sample_spans_the_sweep():
    # the default benchmark line times fused against unfused on these points
    pts = [WORKLOADS[n] for n in bench.SWEEP_SAMPLE]
    assert {w.P for w in pts} == {2, 4, 8}
    assert {w.m_per_device for w in pts} == {8, 32, 128, 1000, 4096}
    assert {w.rhs_transpose for w in pts} == {False, True}
    peaks, _ = bench.load_peaks()
    bounds = {bench.roofline_of(w, 1e-3, peaks, "measured")["bound"] for w in pts}
    assert bounds == {"hbm", "tensor"}
