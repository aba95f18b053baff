"""Host-side arithmetic of bench.py: the step-roofline FLOP count and
parameter count against a recount from the block's shapes and against the
library's layout, and the stream-timeline statistics on hand-made trace events
(Chrome trace format: ts and dur in microseconds)."""
import pytest

import bench
from host_memory_centric_gb300 import configs


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


def _recount(c):
    """Tensor FLOPs of one step, enumerated op by op: every projection runs
    forward, again in the block recompute, and twice in the backward (input
    and weight gradient), 2 t out in each; causal attention per head costs
    hd S^2 per product (half of the S x S square, 2 FLOP per multiply-add):
    QK^T and PV forward, the same in the recompute, and in the backward the
    recomputed scores, dP, dV, dQ and dK; the LM head runs forward, input and
    weight gradient once."""
    L, H, nh, nkv, hd, F, V = (c[k] for k in ("n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "ffn",
                                              "vocab"))
    B, S, M = c["batch"], c["seq"], c["micro"]
    t = B * S
    projections = [((nh + 2 * nkv) * hd, H), (H, nh * hd), (2 * F, H), (H, F)]
    per_layer = 0
    for out, inp in projections:
        fwd = 2 * t * out * inp
        per_layer += fwd + fwd + (fwd + fwd)  # forward, recompute, dgrad + wgrad
    causal_product = B * nh * hd * S * S  # 2 * hd * S^2 / 2 per head and sequence
    per_layer += (2 + 2 + 5) * causal_product
    head = 3 * 2 * t * H * V
    return M * (L * per_layer + head)


@pytest.mark.parametrize("name", ["tiny", "1.2b", "7.6b", "14.7b", "lc32k", "lc512k"])
def test_model_numbers_match_op_recount_and_layout(name):
    import host_memory_centric_gb300 as mt
    c = configs.get(name)
    P, F_exec, _ = bench.model_numbers(c)
    assert F_exec == _recount(c)
    cfg = mt.make_config(c)
    lay = mt.layout(cfg)
    assert P == sum(r * cc for b in lay for (_o, r, cc) in b["tensors"]) == sum(b["n_real"] for b in lay)


def test_model_numbers_checkpoint_interval_adds_segment_forwards():
    c = configs.get("lc512k")
    _, f1, _ = bench.model_numbers(c, 1)
    _, f4, _ = bench.model_numbers(c, 4)
    L, t, S = c["n_layers"], c["batch"] * c["seq"], c["seq"]
    P_mm = c["hidden"] * (c["n_heads"] + 2 * c["n_kv_heads"]) * c["head_dim"] + \
        c["n_heads"] * c["head_dim"] * c["hidden"] + 3 * c["hidden"] * c["ffn"]
    rebuilt = L - 7  # 28 layers in segments of 4: 7 stored boundaries, 21 layers rebuilt
    assert f4 - f1 == rebuilt * (2 * t * P_mm + 2 * c["batch"] * c["n_heads"] * c["head_dim"] * S * S)


@pytest.mark.parametrize("name", ["tiny_moe", "moe"])
def test_moe_parameter_count_matches_layout(name):
    import host_memory_centric_gb300 as mt
    c = configs.get(name)
    P, _, _ = bench.model_numbers(c)
    lay = mt.layout(mt.make_config(c))
    assert P == sum(r * cc for b in lay for (_o, r, cc) in b["tensors"])
