"""CPU tests of the static schedule's pipeline model (mt_schedule_simulate,
mt_schedule_plan).

The model simulates consecutive steps of the layer-streamed pipeline: the
just-in-time pack (chunked, each chunk's copy starting once it is packed),
the host-to-device copy, the compute, the gradient export into K slabs and
host Adam sharing host memory with DMA and the pack, with the event
protocol's dependencies.  It is checked against what fixes it independently:
* with the host side free (instant Adam, no pack, ample slabs) its per-visit
  compute-stream waits are the oracle's transfer-model schedule, itself pinned
  to the per-layer transfer times the pages print;
* its steady-state step is never shorter than any single resource's total
  work (compute, each link direction, host Adam at its rate) and never longer
  than all of them one after another;
* a single resource that dominates sets the step;
* Adam's rate under shared host memory is what the bandwidth leaves.
The planner must choose different slab counts for different measured inputs.
"""
import numpy as np
import pytest

import host_memory_centric_gb300 as mt
from host_memory_centric_gb300 import configs


def visit_inputs(name, pin_store=False, c_layer=0.02, **over):
    """Per-visit arrays of one step of a config, as the library builds them:
    H2D bytes (weights, plus the checkpoint at a segment's first backward
    visit), packed bytes, exported gradient bytes and Adam elements."""
    c = configs.get(name, **over)
    cfg = mt.make_config(c)
    plan = mt.visit_plan(cfg)
    lay = mt.layout(cfg)
    T, H = c["micro"] * c["batch"] * c["seq"], c["hidden"]
    kind = np.array([k for k, _ in plan], np.int32)
    block = np.array([j for _, j in plan], np.int32)
    wb = np.array([2 * lay[j]["n_pad"] for j in block], np.float64)
    copies = ~((block == 0) & (kind == 3))
    b = np.where(copies, wb, 0.0)
    # the backward visit of a layer whose input is a host checkpoint also loads it
    b += np.where((kind == 3) & (block >= 1), 2.0 * T * H, 0.0)
    p = np.zeros_like(b) if pin_store else np.where(copies, wb, 0.0)
    exp = (kind == 1) | (kind == 3)
    d = np.where(exp, wb, 0.0)
    a = np.where(exp, np.array([lay[j]["n_pad"] for j in block], np.float64), 0.0)
    cc = np.full(len(plan), c_layer)
    cc[kind == 3] *= 3.0
    return kind, block, b, p, d, cc, a


def sim(args, K=64, **rates):
    kind, block, b, p, d, cc, a = args
    si = mt.sched_in(kind, block, b, p, d, cc, a, **rates)
    return mt.schedule_simulate(si, K)


def test_host_free_pipeline_is_the_transfer_model(orc):
    """Instant Adam, a pinned store and ample slabs: the wait before each
    visit computes is max(0, d[v-2]/BW_d2h + b[v]/BW_h2d - c[v-1]), the
    oracle's schedule, wherever the previous visit itself did not wait."""
    kind, block, b, p, d, cc, a = visit_inputs("7.6b", pin_store=True)
    rng = np.random.default_rng(5)
    cc = rng.uniform(0.004, 0.03, len(cc))
    short = np.arange(4, len(cc) - 1, 5)
    cc[short] = 1e-4  # the visit after a short one cannot hide its copy
    bw_h, bw_d = 2.1e11, 1.9e11
    out, stall = sim((kind, block, b, p, d, cc, a), bw_h2d=bw_h, bw_d2h=bw_d, adam_rate=0.0)
    ref, _ = orc.schedule(b, d, cc, np.zeros_like(cc), bw_h, bw_d)
    ok = 0
    for v in range(3, len(cc)):
        if stall[v - 1] > 0 or ref[v - 1] > 0:
            continue
        assert stall[v] == pytest.approx(ref[v], abs=1e-9), v
        ok += 1
    assert ok > 30
    assert np.count_nonzero(ref[short + 1] > 0) >= len(short) - 2


@pytest.mark.parametrize("pin", [True, False])
def test_period_between_resource_bounds(pin):
    rng = np.random.default_rng(7)
    for trial in range(12):
        args = list(visit_inputs("1.2b", pin_store=pin, c_layer=float(rng.uniform(0.001, 0.02))))
        rates = dict(bw_h2d=float(rng.uniform(5e10, 3e11)), bw_d2h=float(rng.uniform(5e10, 3e11)),
                     pack_rate=float(rng.uniform(3e10, 2e11)), adam_rate=float(rng.uniform(2e9, 2e10)))
        K = int(rng.integers(1, 16))
        out, stall = sim(args, K, **rates)
        kind, block, b, p, d, cc, a = args
        per = out["period_ms"] / 1e3
        lower = max(cc.sum(), b.sum() / rates["bw_h2d"], d.sum() / rates["bw_d2h"], a.sum() / rates["adam_rate"],
                    p.sum() / rates["pack_rate"])
        upper = (cc.sum() + b.sum() / rates["bw_h2d"] + d.sum() / rates["bw_d2h"] + a.sum() / rates["adam_rate"]
                 + p.sum() / rates["pack_rate"])
        assert lower * (1 - 1e-9) <= per <= upper * (1 + 1e-9), (trial, lower, per, upper)
        assert out["stall_ms"] >= 0 and np.all(stall >= 0)
        # the compute stream is busy for sum(c) of every period
        assert out["stall_ms"] / 1e3 == pytest.approx(per - cc.sum(), rel=1e-6, abs=1e-9)


def test_dominant_resource_sets_the_step():
    args = visit_inputs("7.6b", pin_store=True, c_layer=0.01)
    kind, block, b, p, d, cc, a = args
    # host Adam far slower than everything else: the step is Adam's work plus
    # at most the part of the step in which no gradient exists yet
    out, _ = sim(args, K=64, bw_h2d=1e13, bw_d2h=1e13, adam_rate=1.6e8)
    t_adam = a.sum() / 1.6e8
    assert t_adam <= out["period_ms"] / 1e3 <= t_adam + cc.sum()
    assert out["adam_busy_ms"] / 1e3 == pytest.approx(t_adam, rel=0.05)
    # compute far slower: the step is the compute and nothing waits
    out, _ = sim(args, K=64, bw_h2d=1e13, bw_d2h=1e13, adam_rate=1e13)
    assert out["period_ms"] / 1e3 == pytest.approx(cc.sum(), rel=1e-3)
    # the pack far slower (just in time): every visit waits for its own pack
    args = visit_inputs("7.6b", pin_store=False, c_layer=0.001)
    kind, block, b, p, d, cc, a = args
    out, _ = sim(args, K=64, bw_h2d=1e13, bw_d2h=1e13, adam_rate=1e13, pack_rate=1e9)
    assert out["period_ms"] / 1e3 == pytest.approx(p.sum() / 1e9, rel=0.02)


def test_shared_host_memory_slows_adam():
    """With host memory shared, Adam runs at what the bandwidth leaves after
    the period's DMA and pack traffic, never faster than on an idle host."""
    args = visit_inputs("7.6b", pin_store=False, c_layer=0.006)
    kind, block, b, p, d, cc, a = args
    free, _ = sim(args, K=16, adam_rate=8.5e9, pack_rate=1.2e11)
    shared, _ = sim(args, K=16, adam_rate=8.5e9, pack_rate=1.2e11, host_bw=3.0e11)
    assert free["adam_gelem_s"] == pytest.approx(8.5, rel=1e-9)
    assert shared["adam_gelem_s"] < free["adam_gelem_s"]
    assert shared["period_ms"] > free["period_ms"]
    per = shared["period_ms"] / 1e3
    left = 3.0e11 - (b.sum() + d.sum() + 2 * p.sum()) / per
    assert shared["adam_gelem_s"] * 1e9 == pytest.approx(min(8.5e9, max(left, 0.75e11) / 28), rel=2e-3)


def test_plan_sizes_slabs_from_adam_rate():
    """Slow host Adam needs more slabs in flight than fast host Adam."""
    args = visit_inputs("7.6b", pin_store=True, c_layer=0.006)
    fast = mt.schedule_plan(mt.sched_in(*args, adam_rate=5e11), 32)
    slow = mt.schedule_plan(mt.sched_in(*args, adam_rate=8.5e9), 32)
    assert fast["K"] < slow["K"], (fast, slow)
    # the chosen K is within 0.5 % of the best period and no smaller K is
    for pl, rates in ((fast, dict(adam_rate=5e11)), (slow, dict(adam_rate=8.5e9))):
        best = min(sim(args, K, **rates)[0]["period_ms"] for K in range(1, 33))
        assert pl["period_ms"] <= best * 1.005 + 1e-12
        if pl["K"] > 1:
            assert sim(args, pl["K"] - 1, **rates)[0]["period_ms"] > best * 1.005


def test_schedule_rejects_bad_input():
    args = visit_inputs("tiny", pin_store=True)
    si = mt.sched_in(*args)
    with pytest.raises(mt.MtError):
        mt.schedule_simulate(si, 0)
    si = mt.sched_in(*args, bw_h2d=0.0)
    with pytest.raises(mt.MtError):
        mt.schedule_plan(si, 4)
