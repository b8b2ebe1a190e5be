"""The benchmark's byte accounting (the roofline's numerator) against the per-step totals that
follow from the workload definitions: every index page of each row (8704 B) plus the K and V pages
of the k_eff selected pages (8704 B MXFP4, 16896 B FP8-KV, per KV head). Host only."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_attention_decode_mxfp4_gb300 import workloads as wl  # noqa: E402


def total(w, ctx):
    idx, kv = bench.algorithmic_bytes(w, ctx)
    return idx + kv


def test_fixed_workloads():
    assert total(wl.config(1), [1024]) == 8 * 8704 + 4 * 2 * 8704 == 139_264
    assert total(wl.config(2), [16384] * 4) == 5_570_560
    assert total(wl.config(3), [65536] * 4) == 22_151_168
    # 1919 full pages + 75 tokens = 1920 pages per row
    assert total(wl.config(4), [245707] * 2) == 35_651_584


def test_largest_sweep_shape_and_short_rows():
    w = wl.shrink(wl.config(2), B=4, max_ctx=262144, topk=128)
    assert total(w, [262144] * 4) == 80_216_064
    # rows shorter than k pages select every page they have; a row of Q tokens has one page
    w = wl.shrink(wl.config(2), B=2, topk=16)
    assert total(w, [1000, 8]) == (8 + 1) * 8704 + (8 + 1) * 2 * 8704


def test_split_count_is_not_in_the_bytes():
    a = wl.shrink(wl.config(2), num_splits=1)
    b = wl.shrink(wl.config(2), num_splits=16)
    assert total(a, [16384] * 4) == total(b, [16384] * 4)


def test_traffic_record_is_ignored_for_another_workload_or_source(monkeypatch):
    assert bench.recorded_traffic("no_such_workload") is None
    assert bench.recorded_traffic("no_such_workload", reuse=True) is None
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda: "0" * 64)
    assert bench.recorded_traffic("verify_b4_q8_h16_ctx16384_k16") is None
