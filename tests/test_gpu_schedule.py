"""The static schedule inside a model (mt_get_schedule): mt_init_model sizes
the gradient slab pool from its plan when n_grad_slabs is 0, and plans again
on the first step's measured per-visit compute times."""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import host_memory_centric_gb300 as mt  # noqa: E402
from host_memory_centric_gb300 import configs, inputs  # noqa: E402


@pytest.mark.parametrize("pin", [0, 1])
def test_init_allocates_the_planned_slab_pool(pin):
    c = configs.get("tiny", n_layers=3)
    planned = mt.Model(c, seed=1, pin_store=pin)  # n_grad_slabs = 0: the schedule decides
    p0 = planned.schedule(0)
    K = p0["K"]
    assert K >= 1 and p0["measured"] == 0
    assert p0["bw_h2d_gbs"] > 0 and p0["bw_d2h_gbs"] > 0 and p0["adam_gelem_s_idle"] > 0
    assert planned.schedule(1) is None  # no step has run yet
    fixed = mt.Model(c, seed=1, pin_store=pin, n_grad_slabs=K)
    more = mt.Model(c, seed=1, pin_store=pin, n_grad_slabs=K + 1)
    slab = max(b["off_G"] - b["off_W"] for b in planned.layout)  # one slab holds the largest G region
    assert planned.stats()["pinned_bytes"] == fixed.stats()["pinned_bytes"]
    assert more.stats()["pinned_bytes"] - fixed.stats()["pinned_bytes"] == slab
    # the first step's per-visit compute times give the second plan, for the same K
    planned.set_tokens(inputs.tokens_for(c, 0))
    planned.train_step(0)
    planned.sync()
    p1 = planned.schedule(1)
    assert p1 is not None and p1["measured"] == 1 and p1["K"] == K and p1["period_ms"] > 0
    for m in (planned, fixed, more):
        m.close()


def test_steps_driven_by_hand_leave_the_measured_plan_unset():
    """The first-step plan needs mt_train_step's per-visit timing; driving
    the visits by hand leaves it unset and must not disturb later launches."""
    c = configs.get("tiny", n_layers=2)
    m = mt.Model(c, seed=2)
    m.set_tokens(inputs.tokens_for(c, 0))
    for v, (kind, j) in enumerate(mt.visit_plan(m.cfg)):
        m.stream_in(j, v % 2)
        view = m.bind(j, v % 2)
        (m.step_backward if kind == 3 else m.step_forward)(view)
        if kind in (1, 3):
            m.adam_host(j, m.stream_out(j, v % 2), 1)
    m.sync()
    assert m.schedule(1) is None
    m.set_tokens(inputs.tokens_for(c, 1))
    assert m.train_step(1) > 0  # no stale error from the unrecorded timing events
    m.sync()
    m.close()
