"""Host-side logic of bench.py (no GPU): the roofline entry names the roof
that binds the decode kernel."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6700.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def test_hbm_bound_decode():
    # 80 MB and 18 GFLOP in 30 us: 2667 GB/s (0.40 of HBM), 608 TFLOP/s (0.32 of tensor)
    r = bench.roofline_entry(80e6, 18.25e9, 0.030, PEAKS, 80.5e6, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 80e6 / 30e-6 / 1e9) < 1e-9
    assert abs(r["frac"] - r["achieved"] / 6700.0) < 1e-12
    assert r["traffic"] == 80.5e6


def test_tensor_bound_decode():
    # speculative decode: 720 MB and 310 GFLOP in 300 us: 0.36 of HBM, 0.54 of tensor
    r = bench.roofline_entry(720e6, 310e9, 0.300, PEAKS, None, "measured")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - 310e9 / 300e-6 / 1e12) < 1e-9
    assert abs(r["frac"] - r["achieved"] / 1900.0) < 1e-12
    assert r["frac"] > 720e6 / 300e-6 / 1e9 / 6700.0
