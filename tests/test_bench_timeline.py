"""Host-side statistics of bench.py's stream timeline, on hand-made trace
events (Chrome trace format: ts and dur in microseconds)."""
import bench


def _ev(tid, name, block, ts, dur):
    return {"name": f"{name} {block}", "tid": tid, "ts": float(ts), "dur": float(dur), "args": {"block": block}}


def test_switch_gaps_counts_only_visits_whose_weights_were_resident():
    W, C = "weight stream", "compute stream"
    ev = [
        _ev(W, "H2D", 0, 0, 100), _ev(C, "FWD", 0, 100, 400),        # first visit: nothing before it
        _ev(W, "H2D", 1, 100, 200), _ev(C, "FWD", 1, 503, 400),      # ready at 300 < 500: gap 3
        _ev(W, "H2D", 2, 300, 700), _ev(C, "FWD", 2, 1000, 400),     # copy ends at 1000 > 903: not counted
        _ev(W, "H2D", 3, 1000, 100), _ev(C, "FWD", 3, 1900, 100),    # ready: gap 500 (a wait on something else)
        _ev("gradient stream", "D2H", 3, 2000, 50),
        _ev(W, "H2D_EXP", 3, 1950, 10),                               # expert copies are not the weights' copy
        _ev(C, "BWD", 3, 2001, 100),                                  # block 3's copy ended long ago: gap 1
    ]
    s = bench.switch_gaps(ev)
    assert s["pairs"] == 3
    assert sorted([3.0, 500.0, 1.0])[1] == s["median_us"] == 3.0
    assert s["max_us"] == 500.0 and s["over_100us"] == 1


def test_switch_gaps_without_resident_pairs_is_none():
    ev = [_ev("compute stream", "FWD", 0, 0, 10)]
    assert bench.switch_gaps(ev) is None


def test_union_and_overlap():
    assert bench._union([(0, 2), (1, 3), (5, 6)]) == 4
    assert bench._overlap([(0, 2)], [(1, 3)]) == 1
