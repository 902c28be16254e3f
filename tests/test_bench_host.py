"""Host-side logic of bench.py (no GPU): the FLOP conventions and the workload tables."""
import importlib
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture()
def bench():
    sys.path.insert(0, ROOT)
    mod = importlib.import_module("bench")
    yield importlib.reload(mod)  # a fresh module: select_workload rebinds module globals


def brute_pairs(Tq, Tk, causal, window):
    pos = np.arange(Tq)[:, None] + (Tk - Tq)
    key = np.arange(Tk)[None, :]
    vis = np.ones((Tq, Tk), dtype=bool)
    if causal:
        vis &= key <= pos
    if window >= 0:
        vis &= key >= pos - window
    return int(vis.sum())


@pytest.mark.parametrize("Tq,Tk,causal,window", [
    (1, 1, True, -1), (4, 4, True, -1), (5, 5, True, 1), (3, 5, False, -1), (1, 300, True, -1),
    (17, 300, True, -1), (300, 300, True, 0), (300, 300, True, 63), (200, 1000, True, 129),
    (128, 128, False, -1)])
def test_visible_pairs_brute_force(bench, Tq, Tk, causal, window):
    assert bench.visible_pairs(Tq, Tk, causal, window) == brute_pairs(Tq, Tk, causal, window)


def test_flop_conventions(bench):
    B, H, N, d = 2, 3, 256, 64
    assert bench.fwd_flops(B, H, N, d, False) == 4.0 * B * H * bench.visible_pairs(N, N, False, -1) * d
    # causal: the N^2 / 2 convention (the diagonal's N extra pairs are not counted)
    assert bench.fwd_flops(B, H, N, d, True) == 2.0 * B * H * N * N * d
    assert bench.visible_pairs(N, N, True, -1) == N * (N + 1) // 2
    assert bench.bwd_flops(B, H, N, d, True) == 2.5 * bench.fwd_flops(B, H, N, d, True)


def test_workload_tables(bench):
    assert bench.WORKLOAD["B"] == 4 and bench.WORKLOAD["H"] == 16 and bench.WORKLOAD["N"] == 2048
    assert bench.WORKLOAD["d"] == 64 and not bench.WORKLOAD["causal"]
    names = [c["name"].split(":")[0] for c in bench.CONFIGS]
    assert names == ["1", "2", "3", "4", "4r", "5"]
    for e in bench.EXTENSIONS:
        assert e["Hq"] % e["Hkv"] == 0 and e["Tq"] <= e["Tk"]
        assert e["window"] < 0 or e["causal"]
        assert e["d"] in (64, 128)
    cfg = bench.workload_config()
    assert cfg["workload"] == bench.WORKLOAD["name"] and cfg["parallelism"] == "single"


def test_select_workload(bench):
    bench.select_workload("5")
    assert (bench.WORKLOAD["B"], bench.WORKLOAD["H"], bench.WORKLOAD["N"], bench.WORKLOAD["d"]) == (4, 16, 4096, 128)
    assert bench.WORKLOAD["causal"] and "B4 H16 N4096 d128" in bench.METRIC
