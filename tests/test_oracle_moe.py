"""Pins of the oracle's routed mixture-of-experts layer.

The lilting.ch page (MoE section) says only that a router picks a few of the
experts per token and that only those experts' weights travel; the layer
itself is read as the GPT-OSS-style top-k MoE (softmax over the selected
logits, SwiGLU experts, no router bias, no auxiliary loss).  Each pin below
ties it to something other than its own formula: central finite differences
of the whole step, exact reductions to the dense layer (one expert; identical
experts), invariance under renumbering the experts, hand-computable routing
and gates, and the stated margin.
"""
import math

import numpy as np
import pytest

from host_memory_centric_gb300 import inputs
from tests import protocol_check

MOE_FD = dict(n_layers=1, hidden=16, n_heads=2, n_kv_heads=1, head_dim=8, ffn=8, vocab=37,
              batch=1, seq=7, micro=2, rope_base=1e4, rms_eps=1e-6, init_std=0.02,
              n_experts=4, top_k=2, expert_ffn=8)


def _weights(orc, shape, seed, scale=0.3):
    rng = np.random.default_rng(seed)
    W = []
    for b in orc.layout(shape):
        w = np.zeros(b["n_pad"])
        for (eo, r, cc) in b["tensors"]:
            if cc == 1:
                w[eo:eo + r] = 1.0 + 0.2 * rng.standard_normal(r)
            else:
                w[eo:eo + r * cc] = scale * rng.standard_normal(r * cc)
        W.append(w)
    return W


def _tok(shape, seed=5):
    return inputs.tokens(seed, 0, shape["micro"], shape["batch"], shape["seq"], shape["vocab"])


def test_moe_block_layout(orc):
    """Decoder block = W_qkv, W_o, W_router [E, H], W_experts [E, 3 Fe H], gamma1, gamma2;
    one expert is one contiguous row; the parameter count adds up by hand."""
    s = MOE_FD
    H, E, Fe = s["hidden"], s["n_experts"], s["expert_ffn"]
    lay = orc.layout(s)[1]
    shapes = [(r, c) for (_, r, c) in lay["tensors"]]
    assert shapes == [((2 + 2 * 1) * 8, H), (H, 2 * 8), (E, H), (E, 3 * Fe * H), (H, 1), (H, 1)]
    per_layer = 4 * 8 * H + H * 16 + E * H + E * 3 * Fe * H + 2 * H
    assert orc.param_count(s) == per_layer + 2 * s["vocab"] * H + H


def test_moe_step_finite_differences(orc):
    """Central differences of the fp64 step loss against the hand-derived
    backward, for every tensor including the router and all experts; the
    routing margin is far above the perturbation, so no selection flips."""
    shape = MOE_FD
    W = _weights(orc, shape, 21)
    tok = _tok(shape)
    loss, G = orc.step_fwd_bwd(shape, W, tok, dtype=np.float64)
    margin = orc.last_route_margin()
    assert 1e-3 < margin < math.inf
    rng = np.random.default_rng(22)
    h = 1e-5
    for j, b in enumerate(orc.layout(shape)):
        for (eo, r, cc) in b["tensors"]:
            n = r * cc
            g = G[j][eo:eo + n]
            rms = math.sqrt(float((g ** 2).mean())) + 1e-30
            for e in rng.choice(n, min(24, n), replace=False):
                Wp = [w.copy() for w in W]; Wm = [w.copy() for w in W]
                Wp[j][eo + e] += h; Wm[j][eo + e] -= h
                fd = (orc.step_fwd_bwd(shape, Wp, tok, np.float64)[0]
                      - orc.step_fwd_bwd(shape, Wm, tok, np.float64)[0]) / (2 * h)
                assert abs(fd - g[e]) / max(abs(g[e]), rms) <= 1e-6, (j, eo, e, fd, g[e])


def _dense_from_moe(orc, moe_shape, Wm, expert):
    """Dense-shape weights whose MLP is expert `expert` of the MoE weights."""
    dshape = {k: v for k, v in moe_shape.items() if k not in ("n_experts", "top_k", "expert_ffn")}
    dshape["ffn"] = moe_shape["expert_ffn"]
    H, Fe = moe_shape["hidden"], moe_shape["expert_ffn"]
    Wd = []
    for j, (bm, bd) in enumerate(zip(orc.layout(moe_shape), orc.layout(dshape))):
        w = np.zeros(bd["n_pad"])
        if 1 <= j <= moe_shape["n_layers"]:
            tm, td = bm["tensors"], bd["tensors"]
            for t in (0, 1, 4, 5):
                (om, r, c), (od, _, _) = tm[t], td[t]
                w[od:od + r * c] = Wm[j][om:om + r * c]
            row = Wm[j][tm[3][0] + expert * 3 * Fe * H:][:3 * Fe * H]
            w[td[2][0]:td[2][0] + 2 * Fe * H] = row[:2 * Fe * H]
            w[td[3][0]:td[3][0] + H * Fe] = row[2 * Fe * H:]
        else:
            w[:] = Wm[j][:bd["n_pad"]]
        Wd.append(w)
    return dshape, Wd


def test_single_expert_is_the_dense_layer(orc):
    """E = k = 1: the gate is 1, the layer is the dense SwiGLU MLP, and the
    router gets an exactly zero gradient."""
    shape = dict(MOE_FD, n_experts=1, top_k=1)
    Wm = _weights(orc, shape, 31)
    tok = _tok(shape)
    loss_m, Gm = orc.step_fwd_bwd(shape, Wm, tok, dtype=np.float64)
    dshape, Wd = _dense_from_moe(orc, shape, Wm, 0)
    loss_d, Gd = orc.step_fwd_bwd(dshape, Wd, tok, dtype=np.float64)
    assert loss_m == pytest.approx(loss_d, rel=1e-13)
    lm, ld = orc.layout(shape)[1]["tensors"], orc.layout(dshape)[1]["tensors"]
    H, Fe = shape["hidden"], shape["expert_ffn"]
    router = Gm[1][lm[2][0]:lm[2][0] + H]
    assert not np.any(router)
    row = Gm[1][lm[3][0]:lm[3][0] + 3 * Fe * H]
    np.testing.assert_allclose(row[:2 * Fe * H], Gd[1][ld[2][0]:ld[2][0] + 2 * Fe * H], rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(row[2 * Fe * H:], Gd[1][ld[3][0]:ld[3][0] + H * Fe], rtol=1e-10, atol=1e-14)
    for t in (0, 1, 4, 5):
        (om, r, c), (od, _, _) = lm[t], ld[t]
        np.testing.assert_allclose(Gm[1][om:om + r * c], Gd[1][od:od + r * c], rtol=1e-10, atol=1e-14)


def test_identical_experts_equal_one_dense_mlp(orc):
    """With every expert equal, the gates (which sum to one) weight the same
    output: loss equals the dense layer's, the router gradient vanishes and
    the expert gradients sum to the dense gradient."""
    shape = dict(MOE_FD, n_experts=4, top_k=3)
    Wm = _weights(orc, shape, 41)
    H, Fe, E = shape["hidden"], shape["expert_ffn"], shape["n_experts"]
    eo = orc.layout(shape)[1]["tensors"][3][0]
    row0 = Wm[1][eo:eo + 3 * Fe * H].copy()
    for e in range(E):
        Wm[1][eo + e * 3 * Fe * H:eo + (e + 1) * 3 * Fe * H] = row0
    tok = _tok(shape)
    loss_m, Gm = orc.step_fwd_bwd(shape, Wm, tok, dtype=np.float64)
    dshape, Wd = _dense_from_moe(orc, shape, Wm, 0)
    loss_d, Gd = orc.step_fwd_bwd(dshape, Wd, tok, dtype=np.float64)
    assert loss_m == pytest.approx(loss_d, rel=1e-12)
    ro = orc.layout(shape)[1]["tensors"][2][0]
    assert np.abs(Gm[1][ro:ro + E * H]).max() < 1e-13
    ex = Gm[1][eo:eo + E * 3 * Fe * H].reshape(E, -1).sum(axis=0)
    ld = orc.layout(dshape)[1]["tensors"]
    dense = np.concatenate([Gd[1][ld[2][0]:ld[2][0] + 2 * Fe * H], Gd[1][ld[3][0]:ld[3][0] + H * Fe]])
    np.testing.assert_allclose(ex, dense, rtol=1e-10, atol=1e-14)


def test_renumbering_experts_permutes_gradients(orc):
    """Permuting the experts (router rows with expert rows) leaves the loss
    unchanged and permutes the router and expert gradients the same way."""
    shape = MOE_FD
    W = _weights(orc, shape, 51)
    tok = _tok(shape)
    loss, G = orc.step_fwd_bwd(shape, W, tok, dtype=np.float64)
    H, Fe, E = shape["hidden"], shape["expert_ffn"], shape["n_experts"]
    t = orc.layout(shape)[1]["tensors"]
    ro, eo = t[2][0], t[3][0]
    perm = np.array([2, 0, 3, 1])
    Wp = [w.copy() for w in W]
    Wp[1][ro:ro + E * H] = W[1][ro:ro + E * H].reshape(E, H)[perm].ravel()
    Wp[1][eo:eo + E * 3 * Fe * H] = W[1][eo:eo + E * 3 * Fe * H].reshape(E, -1)[perm].ravel()
    lossp, Gp = orc.step_fwd_bwd(shape, Wp, tok, dtype=np.float64)
    assert lossp == pytest.approx(loss, rel=1e-13)
    np.testing.assert_allclose(Gp[1][ro:ro + E * H].reshape(E, H), G[1][ro:ro + E * H].reshape(E, H)[perm],
                               rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(Gp[1][eo:eo + E * 3 * Fe * H].reshape(E, -1),
                               G[1][eo:eo + E * 3 * Fe * H].reshape(E, -1)[perm], rtol=1e-10, atol=1e-15)


def _layer_inputs(T, H, E, Fe, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((T, H)), rng.standard_normal((T, H)), 0.3 * rng.standard_normal((E, H)),
            0.3 * rng.standard_normal((E, 3 * Fe * H)), rng.standard_normal((T, H)))


def test_routing_and_gates_by_hand(orc):
    """yn = the first unit vector, so the logits are column 0 of W_router:
    the top-k, the tie rule (lower index first), the gates (softmax of the
    chosen logits) and the margin are known by hand."""
    T, H, E, Fe, k = 2, 8, 5, 8, 2
    _, x1, Wr, We, dout = _layer_inputs(T, H, E, Fe, 61)
    yn = np.zeros((T, H)); yn[:, 0] = 1.0
    Wr[:, 0] = [0.5, 2.0, -1.0, 2.0, 1.5]   # experts 1 and 3 tie at the top
    out, dyn, dWr, dWe, idx, gate, margin = orc.moe_layer(yn, x1, Wr, We, dout, k, Fe)
    assert idx.tolist() == [[1, 3], [1, 3]]
    np.testing.assert_allclose(gate, 0.5, rtol=0, atol=1e-15)
    assert margin == pytest.approx(2.0 - 1.5, abs=1e-15)
    Wr[:, 0] = [0.5, 2.0, -1.0, 1.0, 1.5]
    out, dyn, dWr, dWe, idx, gate, margin = orc.moe_layer(yn, x1, Wr, We, dout, 3, Fe)
    assert idx.tolist() == [[1, 4, 3]] * 2
    z = np.exp([2.0, 1.5, 1.0]); z /= z.sum()
    np.testing.assert_allclose(gate, np.tile(z, (2, 1)), rtol=1e-14)
    assert margin == pytest.approx(1.0 - 0.5, abs=1e-15)
    # experts never chosen (0 and 2) get exactly zero gradient
    dWe = dWe.reshape(E, -1)
    assert not np.any(dWe[[0, 2]]) and np.all(np.any(dWe[[1, 3, 4]] != 0, axis=1))


def test_zero_router_ties_pick_the_first_experts(orc):
    """W_router = 0: every logit ties, so every token takes experts 0..k-1 with
    gates 1/k, and the output is the mean of those experts' outputs; the
    reported margin is zero."""
    T, H, E, Fe, k = 6, 16, 4, 8, 2
    yn, x1, Wr, We, dout = _layer_inputs(T, H, E, Fe, 71)
    Wr[:] = 0
    out, dyn, dWr, dWe, idx, gate, margin = orc.moe_layer(yn, x1, Wr, We, dout, k, Fe)
    assert (idx == np.arange(k)).all() and margin == 0.0
    np.testing.assert_allclose(gate, 1.0 / k, rtol=1e-15)
    # out - x1 is the average of the two experts run alone (k = 1 with one-hot routers)
    single = []
    for e in range(k):
        o = np.empty_like(yn)
        for t in range(T):
            w = np.zeros((E, H)); w[e, 0] = 1e3 * np.sign(yn[t, 0])  # expert e alone, gate 1
            o[t] = orc.moe_layer(yn[t:t + 1], x1[t:t + 1], w, We, dout[t:t + 1], 1, Fe)[0][0]
        single.append(o - x1)
    np.testing.assert_allclose(out - x1, 0.5 * (single[0] + single[1]), rtol=1e-12, atol=1e-14)


def test_all_experts_selected_has_no_margin_and_fd(orc):
    """top_k = E: no selection (margin +inf); the layer is smooth, and central
    differences of a scalar of its output match its backward for yn, the
    router and the experts."""
    T, H, E, Fe = 3, 8, 3, 8
    yn, x1, Wr, We, dout = _layer_inputs(T, H, E, Fe, 81)
    out, dyn, dWr, dWe, idx, gate, margin = orc.moe_layer(yn, x1, Wr, We, dout, E, Fe)
    assert margin == math.inf
    np.testing.assert_allclose(gate.sum(axis=1), 1.0, rtol=1e-14)
    f = lambda yn_, Wr_, We_: float((orc.moe_layer(yn_, x1, Wr_, We_, dout, E, Fe)[0] * dout).sum())
    rng = np.random.default_rng(82)
    h = 1e-6
    for name, arr, grad in (("yn", yn, dyn), ("Wr", Wr, dWr), ("We", We, dWe)):
        for i in rng.choice(arr.size, 12, replace=False):
            p, m = arr.copy(), arr.copy()
            p.flat[i] += h; m.flat[i] -= h
            args_p = {"yn": (p, Wr, We), "Wr": (yn, p, We), "We": (yn, Wr, p)}[name]
            args_m = {"yn": (m, Wr, We), "Wr": (yn, m, We), "We": (yn, Wr, m)}[name]
            fd = (f(*args_p) - f(*args_m)) / (2 * h)
            assert fd == pytest.approx(grad.flat[i], rel=1e-6, abs=1e-9), (name, i)


def test_fp32_moe_layer_tracks_fp64(orc):
    T, H, E, Fe, k = 16, 32, 6, 16, 2
    args = _layer_inputs(T, H, E, Fe, 91)
    d = orc.moe_layer(*args, k, Fe)
    f = orc.moe_layer(*args, k, Fe, dtype=np.float32)
    assert (d[4] == f[4]).all()
    for a, b in zip(d[:4], f[:4]):
        assert np.linalg.norm(a - b) <= 1e-5 * np.linalg.norm(a)


@pytest.mark.parametrize("jit,ckpt,ci,nbuf", [(1, 1, 1, 2), (0, 1, 1, 2), (0, 0, 2, 2), (1, 1, 2, 1)])
def test_moe_protocol_race_free(orc, jit, ckpt, ci, nbuf):
    shape = dict(MOE_FD, n_layers=3)
    lines = orc.protocol(shape, 3, 2, bool(ckpt), bool(jit), ci, nbuf)
    protocol_check.check(lines)
    per_step = [l for l in lines if l.startswith("1 ")]
    count = lambda op: sum(1 for l in per_step if f" {op} " in l)
    assert count("H2D_EXP") == count("FWD_EXP") == count("WAIT_RT") == 3  # one per decoder forward


def test_moe_protocol_checker_catches_missing_expert_wait(orc):
    shape = dict(MOE_FD, n_layers=2)
    lines = orc.protocol(shape, 2, 2, True, False)
    bad = [l for l in lines if " WAIT_ER " not in l]
    with pytest.raises(AssertionError):
        protocol_check.check(bad)
    bad = [l for l in lines if " WAIT_RT " not in l]
    with pytest.raises(AssertionError):
        protocol_check.check(bad)
