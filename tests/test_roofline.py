"""Host-side roofline arithmetic, pinned to the A100 figures on the QServe pages."""
import pytest

from w4a8_quantized_serving_qoq_gb300 import roofline


def test_a100_crossover_is_78():
    # A100: FP16 312 TOPS, INT8 624 TOPS, 2 TB/s -> W4A16 vs W8A8 cross at m = 78
    m = roofline.w4a16_w8a8_crossover(2e12, 312e12, 624e12)
    assert m == pytest.approx(78.0, abs=1e-6)


def test_bytes_and_ops():
    assert roofline.w4a8_bytes(1, 4096, 4096) == 4096 * 4096 // 2 + 4096
    assert roofline.gemm_ops(4096, 28672, 4096) == 2 * 4096 * 28672 * 4096
    # metadata, scales and output on top of the algorithmic bytes
    assert roofline.w4a8_bytes_full(2, 256, 512, 128) == 256 * 256 + 1024 + 256 * 4 * 2 + 512 + 4 + 2 * 2 * 256


def test_bound_switches_at_ridge():
    bw, peak = 6.8e12, 1.9e15
    r = roofline.ridge_m(bw, peak)
    assert 60 < r < 80
    assert roofline.bound(8, 28672, 4096, bw, peak) == "hbm"
    assert roofline.bound(4096, 28672, 4096, bw, peak) == "tensor"
