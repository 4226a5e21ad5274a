"""The selection-quality measurements (eviction_gb300/metrics.py) on hand-made
kept sets, where the answers are known by construction."""
import numpy as np

from eviction_gb300 import metrics as m


def test_region_tokens_skip_inactive_and_empty():
    start = np.array([[10, 50, 90]])
    length = np.array([[5, 0, 7]])
    active = np.array([[True, True, False]])
    assert m.region_tokens(start, length, active) == [(0, 10, 15)]


def test_wipe_out_rate():
    # unit 0 holds tokens 0..19 before; region [2, 5) keeps token 3, region [10, 13) is
    # wiped out, region [30, 40) was never in the cache (not counted)
    before = np.array([np.arange(20)])
    after = np.array([[0, 1, 3, 15, 16, -1]])
    regions = [(0, 2, 5), (0, 10, 13), (0, 30, 40)]
    rate, present = m.wipe_out_rate(regions, before, after)
    assert present == 2 and rate == 0.5


def test_kept_set_iou():
    a = np.array([[1, 2, 3, 4], [5, 6, -1, -1]])
    b = np.array([[3, 4, 5, 6], [5, 6, -1, -1]])
    # unit 0: |{3,4}| / |{1..6}| = 1/3; unit 1: identical = 1
    assert abs(m.kept_set_iou(a, b) - (1 / 3 + 1) / 2) < 1e-12


def test_compact_ids():
    ids = np.array([[100, 101, 102, 103], [7, 8, 9, 10]])
    kept = np.array([[0, 2, 3], [1, -1, -1]])
    nk = np.array([3, 1])
    out = m.compact_ids(ids, kept, nk)
    assert out.tolist() == [[100, 102, 103], [8, -1, -1]]
