"""Host-side aggregation of the per-CTA profile records (no GPU): records
built by hand in the layout ep_profile_begin documents."""
import numpy as np

import combine_ep_plan_gb300 as ep


def rec(kind, seq, cta, t0, ta, tb, tc, t1, units, nbytes):
    return [(kind << 56) | (seq << 32) | cta, t0, ta, tb, tc, t1, units, nbytes]


def test_summary_groups_by_launch_in_order():
    rows = [
        rec(1, 0, 0, 1000, 1500, 2000, 2600, 4000, 256, 0),
        rec(1, 0, 1, 1010, 1600, 2100, 2600, 3900, 100, 0),
        rec(1, 0, 2, 1020, 0, 1030, 2610, 3800, 0, 0),       # a CTA without a tile
        rec(2, 1, 0, 5000, 0, 0, 0, 6000, 7, 7000),
        rec(2, 1, 1, 5100, 0, 0, 0, 7000, 7, 9000),
        rec(5, 2, 0, 8000, 0, 0, 0, 8500, 3, 4000),
    ]
    s = ep.summarize_profile(np.array(rows, dtype=np.uint64).view(np.int64))
    assert [r["kernel"] for r in s] == ["plan", "dispatch_bf16", "combine"]
    plan, disp, comb = s
    assert plan["ctas"] == 3 and plan["units"] == 356 and plan["bytes"] == 0
    assert plan["span_ns"] == 4000 - 1000
    # stage marks: medians of the non-zero marks, from the launch's first start
    assert plan["scan_ns"] == np.median([500, 600])  # CTAs with a tile only
    assert plan["barrier1_ns"] == np.median([1000, 1100, 30])
    assert plan["barrier2_ns"] == np.median([1600, 1600, 1610])
    assert disp["ctas"] == 2 and disp["units"] == 14 and disp["bytes"] == 16000
    assert disp["span_ns"] == 2000 and disp["gbs"] == 8.0
    assert disp["cta_ns_median"] == np.median([1000, 1900]) and disp["cta_ns_max"] == 1900
    assert comb["gbs"] == 4000 / 500


def test_summary_of_nothing_is_empty():
    assert ep.summarize_profile(np.zeros((0, 8), np.int64)) == []
