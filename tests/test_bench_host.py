"""Host-side helpers of the benchmark (no GPU): the roofline bound and the
code-only hash that keys the captured decode DRAM traffic to the kernel."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_roofline_takes_the_slower_unit():
    # 6.6945 MB at 6694.5 GB/s is 1 us; 1.8928 GFLOP at 1892.8 TFLOP/s is 1 us
    t, bound = bench.roofline_us(6.6945e6, 0.0, 6694.5, 1892.8)
    assert t == pytest.approx(1.0) and bound == "hbm"
    t, bound = bench.roofline_us(6.6945e6, 2 * 1.8928e9, 6694.5, 1892.8)
    assert t == pytest.approx(2.0) and bound == "tensor"
    # the wide shape at M = 8192 is tensor-bound (292.7 us), the default never is
    K, r, HC, HS = 32768, 512, 8, 4096
    w = 2 * (r + HC) * K + 2 * K * r + 2 * K
    a = 2 * K + 2 * HS + 4 * HC + 2 * K + 4 * HC + 4 * HC + 4 * r + 2 * HS
    t, bound = bench.roofline_us(w + 8192 * a, 8192 * 2 * K * (2 * r + HC), 6694.5, 1892.8)
    assert bound == "tensor" and t == pytest.approx(292.7, abs=0.1)
    t, bound = bench.roofline_us(bench.WEIGHT_BYTES + 65536 * bench.ACT_BYTES_PER_TOKEN,
                                 65536 * bench.FLOPS_PER_TOKEN, 6694.5, 1892.8)
    assert bound == "hbm"


def test_code_only_ignores_prose_but_not_code():
    src = "int a = 1;  // one\n/* block\n comment */\nint b = 2;\n\n"
    assert bench.code_only(src) == "int a = 1;\nint b = 2;"
    assert bench.code_only(src.replace("// one", "// another remark")) == bench.code_only(src)
    assert bench.code_only(src.replace("b = 2", "b = 3")) != bench.code_only(src)


def test_decode_hash_is_stable_and_sixty_four_hex():
    h = bench.decode_sources_sha256()
    assert h == bench.decode_sources_sha256() and len(h) == 64
    traffic, source = bench.decode_traffic_per_launch()
    assert (traffic is None) == source.startswith("null")
    assert traffic is None or traffic > 1e7


def test_stale_traffic_is_null_with_its_reason(monkeypatch):
    monkeypatch.setitem(bench.DECODE_TRAFFIC, "sources_sha256", "0" * 64)
    traffic, source = bench.decode_traffic_per_launch()
    assert traffic is None and "changed" in source
