"""The stream timeline (mt_trace) on real device timestamps.

Besides checking that every copy, compute and export of a step is recorded,
it checks on the device clock the orderings the three events exist for (the
hotdry.top page, section on the event-driven synchronisation protocol): a
visit's compute starts only after its weights landed (Weights-Ready), and a
block's gradient export starts only after its backward finished
(Backward-Done).
"""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import host_memory_centric_gb300 as mt  # noqa: E402
from host_memory_centric_gb300 import configs, inputs  # noqa: E402

EPS = 2e-3  # ms: event timestamp resolution


@pytest.mark.parametrize("name,steady", [("tiny", False), ("tiny_moe", False), ("tiny", True)])
def test_timeline_records_the_protocol_order(name, steady):
    """steady: recording starts while the previous step is still in flight
    (no drain), as for a timeline of training in its steady state."""
    c = configs.get(name, n_layers=3)
    L = c["n_layers"]
    m = mt.Model(c, seed=3)
    m.set_tokens(inputs.tokens_for(c, 0))
    m.train_step(0)  # first step: lazy loading and caches out of the way
    m.sync()
    m.set_tokens(inputs.tokens_for(c, 1))
    if steady:
        m.train_step(1)
        m.set_tokens(inputs.tokens_for(c, 2))
    m.trace(True)
    m.train_step(2 if steady else 1)
    m.sync()
    ev = m.trace_events()
    m.trace(False)
    m.close()
    # host Adam jobs of the previous step that ended after recording started are recorded too
    ev = [e for e in ev if e["tid"] != "host Adam" or e["args"]["step"] == (2 if steady else 1)]
    by = {}
    for e in ev:
        by.setdefault((e["tid"], e["name"].split()[0]), []).append(e)
    h2d = by[("weight stream", "H2D")]
    comp = [e for e in ev if e["tid"] == "compute stream"]
    d2h = by[("gradient stream", "D2H")]
    # one stream-in and one compute per visit; the embedding's backward copies nothing but is still a span
    assert len(comp) == 2 * L + 3 and len(h2d) == 2 * L + 3
    assert len(d2h) == L + 2  # every decoder block, the head and the embedding export once
    assert len(by[("host Adam", "ADAM")]) == L + 2
    if name == "tiny_moe":
        assert len(by[("weight stream", "H2D_EXP")]) == L  # routed experts of each decoder forward
    end = lambda e: (e["ts"] + e["dur"]) / 1e3
    start = lambda e: e["ts"] / 1e3
    # visit v: its weights (H2D span v) land before its compute (compute span v) starts
    for w, k in zip(h2d, comp):
        assert w["args"]["block"] == k["args"]["block"]
        assert start(k) >= end(w) - EPS, (w, k)
    # a block's gradient export starts after its backward (or the head's fused visit) ends
    last = {}
    for k in comp:
        if k["name"].startswith(("BWD", "HEAD")):
            last[k["args"]["block"]] = k
    for g in d2h:
        k = last[g["args"]["block"]]
        assert start(g) >= end(k) - EPS, (k, g)
