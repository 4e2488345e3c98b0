"""Host logic of bench.py (no GPU): the clock summary, the dominant kernel's
roofline arithmetic, and the shape keys."""
import json
import os

import pytest

import bench
from memory_bound_weight_gb300 import workloads as wl


def row(sm, mx, *reasons):
    flags = ["Active" if r else "Not Active" for r in reasons] or ["Not Active"] * 4
    return ["2026/12/02 00:00:00.000", str(sm), str(mx), "900.0", "0x0"] + flags


def test_clock_summary():
    s = bench.ClockSampler(0)
    s.rows = [(1.0, row(2070, 2070, 0, 0, 0, 0)), (2.0, row(2060, 2070, 0, 0, 0, 1)),
              (3.0, row(2070, 2070, 0, 0, 0, 0)), (9.0, row(800, 2070, 1, 0, 0, 0)), (2.5, ["bad", "row"])]
    out = s.summary(0.5, 3.5)
    assert out == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3,
                   "window": "timed region"}
    # a timed region shorter than the sampling period takes the samples within 1 s of it
    near = s.summary(8.5, 8.6)
    assert near["window"] == "timed region +/- 1 s" and near["reasons"] == ["hw_slowdown"] and near["sm_mhz"] == 800.0
    assert s.summary(20.0, 21.0) is None


class FakeStep:
    def __init__(self, fmt, M):
        self.fmt, self.M = fmt, M


def test_roofline_of_the_dominant_kernel_hbm_bound():
    peak = 6778.3
    shapes = {(0, 11264, 2048): 5.0, (0, 2048, 2048): 1.7}
    counts = {(0, 11264, 2048): 22, (0, 2048, 2048): 44}
    times = {bench.skey(sh): {"us": us, "copies": 8, "launches": 40} for sh, us in shapes.items()}
    plans = {bench.skey(sh): "lat ..." for sh in shapes}
    r = bench.roofline_fields(FakeStep(wl.FMT_INT4_G64, 1), 0.29, 1900.0, peak, "measured", 123, plans, 89,
                              (0, 11264, 2048), counts, times)
    kb = wl.call_bytes(wl.FMT_INT4_G64, 1, wl.Mat("", 11264, 2048))
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["traffic"] == 123
    assert r["bytes_alg_per_launch"] == kb
    assert r["achieved"] == pytest.approx(kb / 5.0e-6 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / peak)
    assert r["share_of_step"] == pytest.approx(22 * 5.0 / (22 * 5.0 + 44 * 1.7))
    assert r["frac_of_nominal_hbm"] == pytest.approx(r["achieved"] / bench.NOMINAL_HBM_GBS)


def test_roofline_switches_to_the_tensor_bound_when_the_contraction_is_longer():
    tc, _ = bench.tensor_peak()
    sh = (0, 18944, 3584)
    times = {bench.skey(sh): {"us": 100.0, "copies": 8, "launches": 40}}
    for M, bound in ((16, "hbm"), (1024, "tensor")):
        r = bench.roofline_fields(FakeStep(wl.FMT_BF16, M), 1.0, 1.0, 6778.3, "measured", None,
                                  {bench.skey(sh): "tcgen05 ..."}, 1, sh, {sh: 1}, times)
        assert r["bound"] == bound, M
        fl = wl.call_flops(M, wl.Mat("", *sh[1:]))
        assert r["tensor_frac"] == pytest.approx(fl / 100e-6 / 1e12 / tc)
        if bound == "tensor":
            assert r["unit"] == "TFLOP/s" and r["frac"] == pytest.approx(r["tensor_frac"])


def test_peaks_come_from_the_measured_file():
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        pytest.skip("no MEASURED_PEAKS.json")
    d = json.load(open(path))
    assert bench.hbm_peak()[0] == float(d["hbm_gbs"])
    assert bench.tensor_peak()[0] == float(d["bf16_tflops_sustained"])


def test_shape_keys():
    assert bench.skey((0, 2048, 5632)) == "2048x5632"
    assert bench.skey((wl.FUSE_NORM | wl.FUSE_GLU, 5632, 2048)) == "5632x2048+norm+glu"
    assert bench.skey((wl.FUSE_RESIDUAL, 2048, 2048)) == "2048x2048+res"
