"""The benchmark's CPU-oracle sample: the workload cut to its leading
candidates keeps every score those candidates had in the whole workload (the
chain-rule sums read the same hidden rows), whole sets keep their set rules,
and a set cut short becomes a choice set of its leading candidates."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
import workloads as wk  # noqa: E402


@pytest.fixture(scope="module")
def whole():
    wl = wk.custom(d=64, V=300, n_sets=7, K=(2, 6), length=(1, 4), seed=11)
    return wl, oracle.score_workload(wl)


@pytest.mark.parametrize("c1", [1, 2, 5, 9, 10**6])
def test_subset_keeps_scores_of_its_candidates(whole, c1):
    wl, ref = whole
    sub = bench._subset(wl, c1)
    c1 = min(c1, wl.n_cand)
    assert sub.n_cand == c1
    assert sub.set_offsets[0] == 0 and sub.set_offsets[-1] == c1
    assert np.all(np.diff(sub.set_offsets) >= 1)
    # only the rows the sample's tokens read, renumbered densely
    assert sub.N == np.unique(wl.tok_row[:wl.cand_offsets[c1]]).size
    res = oracle.score_workload(sub)
    np.testing.assert_array_equal(res.s, ref.s[:c1])
    for k in range(sub.n_sets):
        a, b = int(sub.set_offsets[k]), int(sub.set_offsets[k + 1])
        whole_set = (a, b) == (int(wl.set_offsets[k]), int(wl.set_offsets[k + 1]))
        if whole_set:
            assert sub.kind[k] == wl.kind[k]
            np.testing.assert_array_equal(res.q[a:b], ref.q[a:b])
            assert res.decision[k] == ref.decision[k]
        else:
            assert k == sub.n_sets - 1 and sub.kind[k] == wk.KIND_CHOICE


def test_subset_of_restricted_pass_keeps_union():
    r = wk.binary_restricted(base=wk.binary_batch(n_questions=4, d=64, V=300))
    sub = bench._subset(r, 3)
    assert sub.union_ids is r.union_ids and sub.mode == r.mode
    res = oracle.score_workload(sub)
    np.testing.assert_array_equal(res.s, oracle.score_workload(r).s[:3])


def test_clock_summary_covers_the_timed_passes():
    """Clock statistics come from the samples received during the marked
    passes; a pass shorter than the sampling period takes the first sample
    after its start; idle samples outside them are not counted."""
    idle = ["2070", "2070", "150", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]
    busy = ["1800", "2070", "1300", "0x4", "Not Active", "Not Active", "Not Active", "Active"]
    c = bench.ClockSampler(None)
    c.rows = [(0.0, idle), (0.2, idle), (0.4, busy), (0.6, busy), (0.8, idle), (1.0, busy), (1.2, idle)]
    c.mark(0.3, 0.7)          # two samples inside
    c.mark(0.9, 0.95)         # none inside: the first after its start
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1800.0 and s["reasons"] == ["sw_power_cap"]
    assert abs(s["window_s"] - 0.45) < 1e-9
