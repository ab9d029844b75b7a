"""The roofline accounting of bench.py: the algorithmic flops and bytes per stage follow the
per-(batch, head) counts of the scope table (query-landmark dot counted once, tutorial ch. 6:
N(2m + sk) scores), and the reported bound is the larger of the tensor and HBM times."""
import pytest

import bench
from sparse_top_landmark_gb300 import workloads as W


def _mb(x):
    return x / 1e6


def _gf(x):
    return x / 1e9


def test_long_64k_counts():
    w = W.WORKLOADS["long_64k"]          # B*H = 8, N = 64K, d = 64, m = k = 128, bf16
    work = bench.stage_work(w)
    assert _mb(work["pool"][1]) == pytest.approx(67.2, abs=0.1)
    assert _gf(work["landmark"][0]) == pytest.approx(17.18, abs=0.01)
    assert _mb(work["landmark"][1]) == pytest.approx(134.9, abs=0.5)
    assert _gf(work["route"][0]) == pytest.approx(8.59, abs=0.01)      # 2Nmd: the QQ~^T half
    assert _mb(work["bucket"][1]) == pytest.approx(6.3, abs=0.1)
    assert _gf(work["expert"][0]) == pytest.approx(17.18 + 8.59, abs=0.02)


def test_long_1m_counts():
    w = W.WORKLOADS["long_1m"]           # B*H = 2, N = 1M, d = 64, m = k = 512, bf16
    work = bench.stage_work(w)
    assert _mb(work["pool"][1]) == pytest.approx(268.6, abs=0.5)
    assert _gf(work["landmark"][0]) == pytest.approx(274.9, abs=0.1)
    assert _gf(work["expert"][0]) == pytest.approx(274.9 + 137.4, abs=0.2)


def test_top_s_scales_the_per_query_terms():
    w = W.WORKLOADS["long_64k"]
    w2 = bench.workload_of("long_64k", 2)
    a, b = bench.stage_work(w), bench.stage_work(w2)
    assert b["landmark"] == a["landmark"] and b["pool"] == a["pool"]
    assert b["expert"][0] - a["expert"][0] == pytest.approx(a["expert"][0] - 2.0 * 8 * 65536 * 128 * 64)
    assert b["bucket"][1] > a["bucket"][1]
    assert w2.name == "long_64k_s2" and w2.s == 2


def test_roofline_entry_picks_the_slowest_stage_and_its_bound():
    w = W.WORKLOADS["long_1m"]
    pk = {"hbm": 6800.0, "tc": 1900.0, "tc_sus": 1700.0, "src": "measured"}
    stages = {"pool": 1e-4, "landmark": 2e-4, "route": 1e-4, "bucket": 1e-4, "expert": 8e-4}
    ent, per = bench.roofline_entry(w, stages, pk)
    fl, _ = bench.stage_work(w)["expert"]
    assert ent["kernel"] == "expert" and ent["bound"] == "tensor"
    assert ent["achieved"] == pytest.approx(fl / 8e-4 / 1e12)
    assert ent["frac"] == pytest.approx(ent["achieved"] / 1900.0)
    assert per["pool"]["frac"] == pytest.approx(bench.roofline_s(*bench.stage_work(w)["pool"], pk)
                                                / 1e-4)
    w64 = W.WORKLOADS["long_64k"]
    ent64, _ = bench.roofline_entry(w64, {"pool": 5e-4, "landmark": 1e-5, "route": 1e-5,
                                          "bucket": 1e-5, "expert": 1e-5}, pk)
    assert ent64["kernel"] == "pool" and ent64["bound"] == "hbm" and ent64["unit"] == "GB/s"
