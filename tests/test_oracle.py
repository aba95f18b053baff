"""Pins of the CPU oracle against things other than itself.

Each test ties one oracle function to the pages, to a closed form, to an
invariant, to an independent library routine (numpy / scipy / torch CPU) or
to finite differences, so that a dropped term, a wrong sign or index or a
transposed operand in the oracle fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

from host_memory_centric_gb300 import configs, inputs
from tests import protocol_check

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

FD_SHAPE = dict(n_layers=1, hidden=16, n_heads=2, n_kv_heads=1, head_dim=8, ffn=32, vocab=37,
                batch=1, seq=7, micro=2, rope_base=1e4, rms_eps=1e-6, init_std=0.02)


# ------------------------------------------------------------------ generator
def test_splitmix64_published_vector(orc):
    vals = [int(l) for l in open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt"))
            if l.strip() and not l.startswith("#")]
    assert [orc.splitmix64(1234567, i) for i in range(5)] == vals


def test_splitmix64_token_module_matches_published_vector():
    vals = [int(l) for l in open(os.path.join(GOLDEN, "splitmix64_seed1234567.txt"))
            if l.strip() and not l.startswith("#")]
    got = inputs.splitmix64(1234567, np.arange(5, dtype=np.uint64))
    assert [int(v) for v in got] == vals


def test_tokens_uniform_range():
    t = inputs.tokens(1234, 0, 2, 3, 1000, 37)
    assert t.shape == (2, 3, 1000) and t.dtype == np.int32
    assert t.min() >= 0 and t.max() < 37
    counts = np.bincount(t.ravel(), minlength=37)
    # chi-square against uniform, 36 dof: 99.99% quantile is about 76
    chi2 = ((counts - t.size / 37) ** 2 / (t.size / 37)).sum()
    assert chi2 < 76


def test_box_muller_is_standard_normal(orc):
    scipy_stats = pytest.importorskip("scipy.stats")
    key = orc.splitmix64(99, 5)
    z = np.array([orc.normal(key, e) for e in range(40000)])
    assert abs(z.mean()) < 0.03 and abs(z.std() - 1) < 0.03
    assert scipy_stats.kstest(z, "norm").pvalue > 1e-3


def test_box_muller_from_published_uniform_mapping(orc):
    # cos branch of Box-Muller on the 53-bit uniforms of two consecutive outputs
    key = orc.splitmix64(7, 3)
    for e in (0, 1, 17, 1000):
        a, b = (int(v) for v in inputs.splitmix64(key, np.array([2 * e, 2 * e + 1], np.uint64)))
        u1 = ((a >> 11) + 1) * 2.0 ** -53
        u2 = (b >> 11) * 2.0 ** -53
        assert orc.normal(key, e) == pytest.approx(math.sqrt(-2 * math.log(u1)) * math.cos(2 * math.pi * u2),
                                                    rel=1e-14, abs=1e-14)


def test_bf16_rne_matches_torch(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(2000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 2000),
                        np.array([0.0, -0.0, 1.0, np.inf, -np.inf, 1e-40, -3e-39, 65504.0, 3.4e38],
                                 np.float32)]).astype(np.float32)
    # exact ties: mantissa low half = 0x8000
    ties = (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.bf16_rne(x), ref)
    assert np.array_equal(orc.bf16_rne_fast(x), ref)
    nan = orc.bf16_rne(np.array([np.nan], np.float32))[0]
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x7F) != 0


# ------------------------------------------------------------------ layout / accounting
def closed_form_params(c):
    L, H, nh, nkv, hd, F, V = (c[k] for k in ("n_layers", "hidden", "n_heads", "n_kv_heads",
                                              "head_dim", "ffn", "vocab"))
    mlp = 3 * H * F
    if c.get("n_experts", 0):  # router [E, H] and E experts of W_gu [2Fe, H] + W_down [H, Fe]
        mlp = c["n_experts"] * H + c["n_experts"] * 3 * H * c["expert_ffn"]
    return L * (H * (nh + 2 * nkv) * hd + nh * hd * H + mlp + 2 * H) + 2 * V * H + H


@pytest.mark.parametrize("name", list(configs.CONFIGS))
def test_param_count_closed_form(orc, name):
    c = configs.get(name)
    assert orc.param_count(c) == closed_form_params(c)


def test_moe_shape_at_full_depth_is_gpt_oss_20b_sized(orc):
    """The ``moe`` shape at GPT-OSS-20B's depth (24 layers) has about 21B
    parameters, the published size of that model (no biases, sinks or
    sliding windows here, so a little below)."""
    p = orc.param_count(configs.get("moe", n_layers=24))
    assert 20.5e9 < p < 21.5e9


def test_param_counts_match_public_model_sizes(orc):
    # Qwen2.5-7B publishes 7.61B parameters including 129,024 QKV bias terms
    # (28 layers x (3584 + 512 + 512)); the shape here has no biases.
    p7 = orc.param_count(configs.get("7.6b"))
    assert p7 == 7_615_487_488
    assert p7 + 28 * (3584 + 2 * 512) == 7_615_616_512
    p14 = orc.param_count(configs.get("14.7b"))
    assert p14 == 14_769_689_600


def test_sixteen_bytes_per_param_table(orc):
    rows = [l.split() for l in open(os.path.join(GOLDEN, "state_accounting.txt"))
            if l.strip() and not l.startswith("#")]
    per = {r[0]: int(r[2]) for r in rows[:5]}
    assert sum(per.values()) == 16
    models = {r[0]: (float(r[1]), float(r[2])) for r in rows[5:]}
    # the page's own rows are 16 B x printed params (rounded by the page)
    for name, (bparams, gb) in models.items():
        assert abs(16 * bparams - gb) <= 0.02 * gb, name
    # our two Qwen shapes land on the page's "about" figures
    for cfg, name in (("7.6b", "Qwen2.5-7B"), ("14.7b", "Qwen2.5-14B")):
        P = orc.param_count(configs.get(cfg))
        state_gb = sum(per.values()) * P / 1e9
        assert abs(state_gb - models[name][1]) / models[name][1] < 0.01, (cfg, state_gb)


def test_layout_tiny_by_hand(orc):
    c = configs.get("tiny")
    lay = orc.layout(c)
    assert len(lay) == 4
    H, V, F = 256, 1024, 1024
    emb = lay[0]
    assert emb["tensors"] == [(0, V, H)]
    assert emb["n_pad"] == V * H
    assert emb["off_W"] == 0 and emb["off_G"] == 2 * V * H and emb["off_master"] == 4 * V * H
    assert emb["off_m"] == 8 * V * H and emb["off_v"] == 12 * V * H and emb["bytes"] == 16 * V * H
    dec = lay[1]
    qkv = (4 + 8) * 64
    expect = [(0, qkv, H)]
    o = qkv * H
    expect.append((o, H, 256)); o += H * 256
    expect.append((o, 2 * F, H)); o += 2 * F * H
    expect.append((o, H, F)); o += H * F
    expect.append((o, H, 1)); o += H
    expect.append((o, H, 1)); o += H
    assert dec["tensors"] == expect
    assert dec["n_real"] == o and dec["n_pad"] == o
    assert dec["store_off"] == emb["bytes"]
    head = lay[3]
    assert head["tensors"] == [(0, H, 1), (256, V, H)]
    assert head["n_pad"] == 256 + V * H


@pytest.mark.parametrize("name", ["tiny", "1.2b", "7.6b", "14.7b"])
def test_layout_invariants(orc, name):
    c = configs.get(name)
    lay = orc.layout(c)
    off = 0
    for b in lay:
        assert b["store_off"] == off and b["store_off"] % 4096 == 0
        off += b["bytes"]
        regions = [b["off_W"], b["off_G"], b["off_master"], b["off_m"], b["off_v"], b["bytes"]]
        assert all(r % 4096 == 0 for r in regions) and regions == sorted(regions)
        assert b["off_G"] - b["off_W"] >= 2 * b["n_pad"] and b["off_m"] - b["off_master"] >= 4 * b["n_pad"]
        end = 0
        for (eo, r, cc) in b["tensors"]:
            assert eo % 128 == 0 and eo >= end
            end = eo + r * cc
        assert end <= b["n_pad"] and b["n_pad"] % 128 == 0
        assert b["n_real"] == sum(r * cc for (_, r, cc) in b["tensors"])
    assert off == orc.store_bytes(c)


def test_init_block_values(orc):
    c = configs.get("tiny")
    m = orc.init_block(c, 42, 1)
    lay = orc.layout(c)[1]
    eo, r, cc = lay["tensors"][0]
    w = m[eo:eo + r * cc]
    assert abs(w.mean()) < 2e-3 and abs(w.std() - 0.02) < 1e-3
    for t in (4, 5):  # RMSNorm gains start at 1
        eo, r, cc = lay["tensors"][t]
        assert np.all(m[eo:eo + r] == 1.0)
    # element e of tensor t of block j = 0.02 * normal(stream key of (j, t), e)
    key = orc.splitmix64(42, 1 + 64 * 1 + 2)
    eo = lay["tensors"][2][0]
    for e in (0, 5, 999):
        assert m[eo + e] == np.float32(0.02 * orc.normal(key, e))


# ------------------------------------------------------------------ per-op pins
def fd_grad(f, x, idx, h=1e-6):
    xp = x.copy(); xp.flat[idx] += h
    xm = x.copy(); xm.flat[idx] -= h
    return (f(xp) - f(xm)) / (2 * h)


def test_rmsnorm_closed_form_and_fd(orc):
    H = 24
    c = 3.5
    x = np.full((1, H), c)
    g = np.linspace(0.5, 1.5, H)
    y, r = orc.rmsnorm_fwd(x, g, eps=1e-6)
    assert np.allclose(y[0], g * c / math.sqrt(c * c + 1e-6), rtol=1e-14)
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, H)); g = rng.standard_normal(H); dy = rng.standard_normal((5, H))
    y, r = orc.rmsnorm_fwd(x, g)
    dx, dg = orc.rmsnorm_bwd(dy, x, g, r)
    f = lambda xx: float((orc.rmsnorm_fwd(xx, g)[0] * dy).sum())
    for i in rng.choice(x.size, 12, replace=False):
        assert fd_grad(f, x, i) == pytest.approx(dx.flat[i], rel=1e-6, abs=1e-9)
    fg = lambda gg: float((orc.rmsnorm_fwd(x, gg)[0] * dy).sum())
    for i in range(0, H, 5):
        assert fd_grad(fg, g, i) == pytest.approx(dg[i], rel=1e-6, abs=1e-9)


def test_linear_matches_numpy(orc):
    rng = np.random.default_rng(2)
    X = rng.standard_normal((9, 13)); W = rng.standard_normal((7, 13)); dY = rng.standard_normal((9, 7))
    assert np.allclose(orc.linear_fwd(X, W), X @ W.T, rtol=1e-13, atol=1e-13)
    assert np.allclose(orc.linear_dgrad(dY, W), dY @ W, rtol=1e-13, atol=1e-13)
    assert np.allclose(orc.linear_wgrad(dY, X), dY.T @ X, rtol=1e-13, atol=1e-13)


def test_rope_properties(orc):
    rng = np.random.default_rng(3)
    n_seq, S, nh, hd = 2, 6, 3, 8
    x = rng.standard_normal((n_seq * S, nh * hd))
    y = orc.rope(x, n_seq, S, nh, hd, 1e4)
    # position 0 of each sequence is the identity
    assert np.array_equal(y[0], x[0]) and np.array_equal(y[S], x[S])
    # each (i, i + hd/2) pair keeps its norm
    xr = x.reshape(-1, nh, 2, hd // 2); yr = y.reshape(-1, nh, 2, hd // 2)
    assert np.allclose(np.hypot(xr[:, :, 0], xr[:, :, 1]), np.hypot(yr[:, :, 0], yr[:, :, 1]), rtol=1e-13)
    # inverse undoes forward
    assert np.allclose(orc.rope(y, n_seq, S, nh, hd, 1e4, inverse=True), x, rtol=1e-12, atol=1e-12)
    # closed form at position p, frequency i: angle = p * base^(-2i/hd), rotate-half pairing
    p, i, h = 4, 1, 2
    ang = p * 1e4 ** (-2 * i / hd)
    a, b = x[p, h * hd + i], x[p, h * hd + hd // 2 + i]
    assert y[p, h * hd + i] == pytest.approx(a * math.cos(ang) - b * math.sin(ang), rel=1e-13)
    assert y[p, h * hd + hd // 2 + i] == pytest.approx(b * math.cos(ang) + a * math.sin(ang), rel=1e-13)


def _attn_dense(qkv, n_seq, S, nh, nkv, hd):
    from scipy.special import softmax
    q = qkv[:, :nh * hd].reshape(n_seq, S, nh, hd)
    k = qkv[:, nh * hd:(nh + nkv) * hd].reshape(n_seq, S, nkv, hd)
    v = qkv[:, (nh + nkv) * hd:].reshape(n_seq, S, nkv, hd)
    grp = nh // nkv
    k = np.repeat(k, grp, axis=2); v = np.repeat(v, grp, axis=2)
    s = np.einsum("nihd,njhd->nhij", q, k) / math.sqrt(hd)
    mask = np.tril(np.ones((S, S), bool))
    s = np.where(mask, s, -np.inf)
    p = softmax(s, axis=-1)
    return np.einsum("nhij,njhd->nihd", p, v).reshape(n_seq * S, nh * hd)


def test_attention_against_dense_softmax_and_special_cases(orc):
    pytest.importorskip("scipy")
    rng = np.random.default_rng(4)
    n_seq, S, nh, nkv, hd = 2, 9, 4, 2, 8
    qkv = rng.standard_normal((n_seq * S, (nh + 2 * nkv) * hd))
    o, lse = orc.attention_fwd(qkv, n_seq, S, nh, nkv, hd)
    assert np.allclose(o, _attn_dense(qkv, n_seq, S, nh, nkv, hd), rtol=1e-12, atol=1e-12)
    # first position attends only to itself: o = v of its kv head
    v0 = qkv[0, (nh + nkv) * hd:].reshape(nkv, hd)
    assert np.allclose(o[0].reshape(nh, hd), np.repeat(v0, nh // nkv, axis=0), rtol=1e-13)
    # equal keys -> uniform weights -> prefix mean of v
    qkv2 = qkv.copy()
    qkv2[:, nh * hd:(nh + nkv) * hd] = 0.3
    o2, lse2 = orc.attention_fwd(qkv2, n_seq, S, nh, nkv, hd)
    v = qkv2[:S, (nh + nkv) * hd:].reshape(S, nkv, hd)
    pref = np.cumsum(v, axis=0) / np.arange(1, S + 1)[:, None, None]
    assert np.allclose(o2[:S].reshape(S, nh, hd), np.repeat(pref, nh // nkv, axis=1), rtol=1e-12)


def test_attention_backward_fd(orc):
    rng = np.random.default_rng(5)
    n_seq, S, nh, nkv, hd = 1, 6, 4, 2, 4
    qkv = rng.standard_normal((n_seq * S, (nh + 2 * nkv) * hd))
    do = rng.standard_normal((n_seq * S, nh * hd))
    o, lse = orc.attention_fwd(qkv, n_seq, S, nh, nkv, hd)
    d = orc.attention_bwd(qkv, o, lse, do, n_seq, S, nh, nkv, hd)
    f = lambda x: float((orc.attention_fwd(x, n_seq, S, nh, nkv, hd)[0] * do).sum())
    for i in rng.choice(qkv.size, 30, replace=False):
        assert fd_grad(f, qkv, i) == pytest.approx(d.flat[i], rel=1e-6, abs=1e-9)


def test_swiglu_and_fd(orc):
    gu = np.array([[0.0, 1.0, 2.0, 3.0]])  # g = [0, 1], u = [2, 3]
    h = orc.swiglu_fwd(gu)
    assert h[0, 0] == 0.0  # silu(0) = 0
    assert h[0, 1] == pytest.approx(1.0 / (1 + math.exp(-1.0)) * 3.0, rel=1e-15)
    rng = np.random.default_rng(6)
    gu = rng.standard_normal((3, 10)); dh = rng.standard_normal((3, 5))
    d = orc.swiglu_bwd(gu, dh)
    f = lambda x: float((orc.swiglu_fwd(x) * dh).sum())
    for i in range(gu.size):
        assert fd_grad(f, gu, i) == pytest.approx(d.flat[i], rel=1e-6, abs=1e-10)


def test_cross_entropy_closed_forms_and_fd(orc):
    n_seq, S, V = 2, 5, 11
    tok = np.arange(n_seq * S, dtype=np.int32) % V
    loss, dl = orc.cross_entropy(np.zeros((n_seq * S, V)), tok, n_seq, S, n_seq * (S - 1))
    assert loss == pytest.approx(math.log(V), rel=1e-15)
    assert np.all(dl[S - 1] == 0) and np.all(dl[2 * S - 1] == 0)  # no target on last positions
    rng = np.random.default_rng(7)
    z = rng.standard_normal((n_seq * S, V))
    tok = rng.integers(0, V, n_seq * S).astype(np.int32)
    loss, dl = orc.cross_entropy(z, tok, n_seq, S, 8.0)
    from scipy.special import logsumexp
    ref = sum(logsumexp(z[n * S + p]) - z[n * S + p, tok[n * S + p + 1]]
              for n in range(n_seq) for p in range(S - 1)) / 8.0
    assert loss == pytest.approx(ref, rel=1e-13)
    f = lambda x: orc.cross_entropy(x, tok, n_seq, S, 8.0)[0]
    for i in rng.choice(z.size, 20, replace=False):
        assert fd_grad(f, z, i) == pytest.approx(dl.flat[i], rel=1e-6, abs=1e-10)


# ------------------------------------------------------------------ whole step
def _random_weights(orc, shape, seed, scale=0.3, dtype=np.float64):
    rng = np.random.default_rng(seed)
    W = []
    for b in orc.layout(shape):
        w = np.zeros(b["n_pad"], dtype=dtype)
        for (eo, r, cc) in b["tensors"]:
            if cc == 1:
                w[eo:eo + r] = 1.0 + 0.2 * rng.standard_normal(r)
            else:
                w[eo:eo + r * cc] = scale * rng.standard_normal(r * cc)
        W.append(w)
    return W


def test_full_step_finite_differences(orc):
    """Central differences of the step loss in the fp64 instance (h = 1e-5,
    32 elements per tensor) against the hand-derived backward."""
    shape = FD_SHAPE
    W = _random_weights(orc, shape, 11)
    tok = inputs.tokens(5, 0, shape["micro"], shape["batch"], shape["seq"], shape["vocab"])
    loss, G = orc.step_fwd_bwd(shape, W, tok, dtype=np.float64)
    rng = np.random.default_rng(12)
    h = 1e-5
    worst = 0.0
    for j, b in enumerate(orc.layout(shape)):
        for (eo, r, cc) in b["tensors"]:
            n = r * cc
            g = G[j][eo:eo + n]
            rms = math.sqrt(float((g ** 2).mean())) + 1e-30
            for e in rng.choice(n, min(32, n), replace=False):
                Wp = [w.copy() for w in W]; Wm = [w.copy() for w in W]
                Wp[j][eo + e] += h; Wm[j][eo + e] -= h
                fd = (orc.step_fwd_bwd(shape, Wp, tok, np.float64)[0]
                      - orc.step_fwd_bwd(shape, Wm, tok, np.float64)[0]) / (2 * h)
                err = abs(fd - g[e]) / max(abs(g[e]), rms)
                worst = max(worst, err)
                assert err <= 1e-6, (j, eo, e, fd, g[e])
    assert worst < 1e-6


def test_zero_head_gives_ln_vocab(orc):
    shape = configs.get("tiny")
    W = [orc.init_block(shape, 1, j) for j in range(4)]
    eo, r, cc = orc.layout(shape)[3]["tensors"][1]
    W[3][eo:eo + r * cc] = 0.0
    tok = inputs.tokens_for(shape, 0)
    loss, G = orc.step_fwd_bwd(shape, W, tok, dtype=np.float32)
    assert loss == pytest.approx(6.931471805599453, rel=1e-12)  # ln 1024
    # logits are all zero so every decoder gradient vanishes except the head's
    assert np.all(G[1] == 0) and np.all(G[0] == 0)


def test_random_init_loss_near_ln_vocab(orc):
    shape = configs.get("tiny")
    W = [orc.init_block(shape, 1, j) for j in range(4)]
    loss, _ = orc.step_fwd_bwd(shape, W, inputs.tokens_for(shape, 0), dtype=np.float32)
    assert abs(loss - math.log(1024)) < 0.05


def test_forward_hidden_embedding_identity_layers_and_causality(orc):
    """Hidden states after block j: block 0 is the embedding gather; a decoder
    layer with W_o = 0 and W_down = 0 adds nothing to its residual stream;
    and causal attention makes position p depend only on tokens 0..p of its
    own sequence."""
    shape = configs.get("tiny")
    L, H = shape["n_layers"], shape["hidden"]
    W = [orc.init_block(shape, 3, j) for j in range(L + 2)]
    tok = inputs.tokens_for(shape, 0)
    flat = tok.reshape(-1)
    E = W[0][:shape["vocab"] * H].reshape(shape["vocab"], H)
    h0 = orc.forward_hidden(shape, W, tok, 0)
    assert np.array_equal(h0, E[flat])
    lay = orc.layout(shape)
    Wz = [w.copy() for w in W]
    for j in range(1, L + 1):
        for t in (1, 3):  # W_o, W_down
            o, r, cc = lay[j]["tensors"][t]
            Wz[j][o:o + r * cc] = 0.0
    assert np.array_equal(orc.forward_hidden(shape, Wz, tok, L), h0)
    # causality: change the token at position p of sequence 0
    hL = orc.forward_hidden(shape, W, tok, L)
    S, p = shape["seq"], 77
    tok2 = tok.copy().reshape(-1, S)
    tok2[0, p] = (tok2[0, p] + 1) % shape["vocab"]
    hL2 = orc.forward_hidden(shape, W, tok2.reshape(tok.shape), L)
    assert np.array_equal(hL2[:p], hL[:p])            # earlier positions of that sequence
    assert not np.array_equal(hL2[p:S], hL[p:S])      # the changed position and later ones move
    assert np.array_equal(hL2[S:], hL[S:])            # the other sequence is untouched


def test_adam_f32_closed_form_and_torch(orc):
    """Adam on an FP32 gradient (the host-accumulation path): constant g gives
    a step of -lr g / (|g| + eps) every step; on BF16-representable gradients
    it equals the BF16-gradient Adam bit for bit; random FP32 gradients match
    torch.optim.Adam."""
    g = np.array([0.1234567, -3.3e-5, 7.77, 0.0], np.float32)
    master = np.array([0.1, 0.2, -0.3, 0.4], np.float32)
    m = np.zeros(4, np.float32); v = np.zeros(4, np.float32)
    for step in (1, 2, 3):
        before = master.copy()
        w = orc.adam_f32(g, master, m, v, step)
        assert np.allclose(master - before, -1e-3 * g / (np.abs(g) + 1e-8), rtol=2e-5, atol=1e-10)
        assert np.array_equal(w, orc.bf16_rne(master))
    rng = np.random.default_rng(12)
    gb = orc.bf16_rne((rng.standard_normal(256) * 1e-2).astype(np.float32))
    m1, v1, m2, v2 = (np.zeros(256, np.float32) for _ in range(4))
    p1 = (0.02 * rng.standard_normal(256)).astype(np.float32); p2 = p1.copy()
    for step in (1, 2):
        w1 = orc.adam(gb, p1, m1, v1, step)
        w2 = orc.adam_f32(orc.bf16_to_f32(gb), p2, m2, v2, step)
        assert np.array_equal(p1, p2) and np.array_equal(w1, w2)
    torch = pytest.importorskip("torch")
    n = 1000
    p0 = (0.02 * rng.standard_normal(n)).astype(np.float32)
    master = p0.copy(); m = np.zeros(n, np.float32); v = np.zeros(n, np.float32)
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.Adam([tp], lr=1e-3, betas=(0.9, 0.999), eps=1e-8, foreach=False)
    for step in (1, 2, 3):
        g32 = (rng.standard_normal(n) * 1e-2).astype(np.float32)
        orc.adam_f32(g32, master, m, v, step)
        tp.grad = torch.from_numpy(g32.copy())
        opt.step()
    assert np.allclose(master, tp.detach().numpy(), rtol=1e-5, atol=1e-8)


def test_micro_batch_copies_give_single_batch_gradient(orc):
    s1 = dict(FD_SHAPE, micro=1)
    s2 = dict(FD_SHAPE, micro=3)
    W = _random_weights(orc, s1, 21)
    tok1 = inputs.tokens(9, 0, 1, s1["batch"], s1["seq"], s1["vocab"])
    tok3 = np.concatenate([tok1] * 3, axis=0)
    l1, G1 = orc.step_fwd_bwd(s1, W, tok1, np.float64)
    l3, G3 = orc.step_fwd_bwd(s2, W, tok3, np.float64)
    assert l3 == pytest.approx(l1, rel=1e-13)
    for a, b in zip(G1, G3):
        assert np.allclose(a, b, rtol=1e-11, atol=1e-14)


def test_fp32_instance_tracks_fp64(orc):
    shape = dict(FD_SHAPE, micro=1)
    W = _random_weights(orc, shape, 31, scale=0.1)
    tok = inputs.tokens(3, 0, 1, shape["batch"], shape["seq"], shape["vocab"])
    ld, Gd = orc.step_fwd_bwd(shape, W, tok, np.float64)
    lf, Gf = orc.step_fwd_bwd(shape, [w.astype(np.float32) for w in W], tok, np.float32)
    assert lf == pytest.approx(ld, rel=1e-6)
    for a, b in zip(Gd, Gf):
        assert np.linalg.norm(a - b) <= 1e-5 * np.linalg.norm(a) + 1e-12


# ------------------------------------------------------------------ Adam
def test_adam_closed_forms(orc):
    g = np.array([0.5, -0.25, 1e-3, 0.0], dtype=np.float32)
    gb = orc.bf16_rne(g)
    gq = orc.bf16_to_f32(gb)
    master = np.array([0.1, 0.2, -0.3, 0.4], np.float32)
    m = np.zeros(4, np.float32); v = np.zeros(4, np.float32)
    start = master.copy()
    for step in (1, 2, 3):
        before = master.copy()
        w = orc.adam(gb, master, m, v, step)
        # constant gradient: m_hat = g, v_hat = g^2 every step -> delta = -lr g/(|g|+eps)
        expect = -1e-3 * gq / (np.abs(gq) + 1e-8)
        assert np.allclose(master - before, expect, rtol=2e-5, atol=1e-10)
        assert np.array_equal(w, orc.bf16_rne(master))
    assert master[3] == start[3]  # g = 0 -> no change


def test_adam_matches_torch_optim(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(8)
    n = 1000
    p0 = (0.02 * rng.standard_normal(n)).astype(np.float32)
    master = p0.copy(); m = np.zeros(n, np.float32); v = np.zeros(n, np.float32)
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.Adam([tp], lr=1e-3, betas=(0.9, 0.999), eps=1e-8, foreach=False)
    for step in (1, 2, 3):
        gb = orc.bf16_rne((rng.standard_normal(n) * 1e-2).astype(np.float32))
        orc.adam(gb, master, m, v, step)
        tp.grad = torch.from_numpy(orc.bf16_to_f32(gb).copy())
        opt.step()
    ref = tp.detach().numpy()
    assert np.linalg.norm(master - ref) <= 1e-6 * np.linalg.norm(ref)


# ------------------------------------------------------------------ protocol / schedule
@pytest.mark.parametrize("ckpt,jit", [(1, 1), (1, 0), (0, 1), (0, 0)])
@pytest.mark.parametrize("slabs", [1, 2, 12])
def test_protocol_is_race_free(orc, ckpt, jit, slabs):
    shape = configs.get("tiny", n_layers=3)
    lines = orc.protocol(shape, 3, slabs, bool(ckpt), bool(jit))
    protocol_check.check(lines)
    L = 3
    per_step = [l for l in lines if l.startswith("1 ")]
    assert sum(1 for l in per_step if " H2D " in l) == (L + 2) + L  # embedding bwd copies nothing
    assert sum(1 for l in per_step if " D2H " in l) == L + 2
    assert sum(1 for l in per_step if " ADAM_ENQ " in l) == L + 2


@pytest.mark.parametrize("L,ci", [(3, 2), (3, 3), (5, 2), (7, 3)])
@pytest.mark.parametrize("ckpt,nbuf", [(1, 2), (0, 2), (1, 1), (0, 1)])
def test_protocol_segments_race_free(orc, L, ci, ckpt, nbuf):
    shape = configs.get("tiny", n_layers=L)
    lines = orc.protocol(shape, 3, 2, bool(ckpt), True, ci, nbuf)
    protocol_check.check(lines)
    per_step = [l for l in lines if l.startswith("1 ")]
    nseg = -(-L // ci)
    count = lambda op: sum(1 for l in per_step if f" {op} " in l)
    assert count("RECOMP") == L - nseg  # every decoder layer but the top of each segment is rebuilt once
    assert count("H2D") == (L + 2) + L + (L - nseg)
    assert count("D2H_CKPT") == (nseg if ckpt else 0)
    assert count("H2D_CKPT") == (nseg if ckpt else 0)
    assert count("D2H") == L + 2 and count("ADAM_ENQ") == L + 2
    bufs = {int(l.split()[4]) for l in per_step if " H2D " in l}
    assert bufs == set(range(nbuf))


@pytest.mark.parametrize("passes,ckpt", [(2, 1), (3, 0), (2, 0)])
def test_protocol_host_accumulation_passes(orc, passes, ckpt):
    """One pass of every block per micro-batch: each pass exports, only the
    last pass's exports run Adam, and only the first pass waits for Adam."""
    L = 3
    shape = configs.get("tiny", n_layers=L)
    lines = orc.protocol(shape, 3, 2, bool(ckpt), True, 1, 2, passes)
    protocol_check.check(lines)
    per_step = [l for l in lines if l.startswith("1 ")]
    count = lambda op: sum(1 for l in per_step if f" {op} " in l)
    assert count("ADAM_ENQ") == L + 2
    assert count("ACCUM_ENQ") == (passes - 1) * (L + 2)
    assert count("D2H") == passes * (L + 2)
    assert count("WAIT_ADAM") == L + 2  # forward visits of the first pass only
    assert count("H2D") == passes * ((L + 2) + L)


def test_protocol_segment_order_hand_example(orc):
    """L = 7, interval 3: X_0, X_3, X_6 kept; segments [7], [4..6], [1..3]
    from the top, each rebuilding X_{s+1} .. X_{e-1} before its backward."""
    shape = configs.get("tiny", n_layers=7)
    lines = orc.protocol(shape, 1, 12, True, False, 3, 2)
    comp = [" ".join(l.split()[2:4]) for l in lines if l.split()[2] in ("FWD", "HEAD", "RECOMP", "BWD")]
    assert comp == ["FWD 0", "FWD 1", "FWD 2", "FWD 3", "FWD 4", "FWD 5", "FWD 6", "FWD 7", "HEAD 8",
                    "BWD 7", "RECOMP 4", "RECOMP 5", "BWD 6", "BWD 5", "BWD 4",
                    "RECOMP 1", "RECOMP 2", "BWD 3", "BWD 2", "BWD 1", "BWD 0"]
    saves = [int(l.split()[3]) for l in lines if " D2H_CKPT " in l]
    loads = [(int(l.split()[3]), int(l.split()[4])) for l in lines if " H2D_CKPT " in l]
    assert saves == [0, 3, 6]
    assert loads == [(7, 0), (4, 1), (1, 0)]  # (first layer of the segment, checkpoint slot)


@pytest.mark.parametrize("drop", ["W WAIT_BF", "C WAIT_WR", "G WAIT_BD", "H WAIT_STAGE", "H WAIT_ADAM",
                                  "C WAIT_XS", "W WAIT_XS", "H ACQ_SLAB"])
def test_protocol_checker_catches_missing_wait(orc, drop):
    shape = configs.get("tiny", n_layers=3)
    lines = orc.protocol(shape, 3, 2, True, True)
    bad = [l for l in lines if drop not in l]
    assert len(bad) < len(lines)
    with pytest.raises(AssertionError):
        protocol_check.check(bad)


def test_schedule_hand_example(orc):
    stall, k = orc.schedule([10, 20, 30], [0, 0, 5], [1.5, 1.0, 1.0], [0, 0, 2], 10.0, 5.0)
    assert np.allclose(stall, [1.0, 0.5, 2.0])
    assert k == 4


def _golden_rows(name):
    rows = []
    for line in open(os.path.join(os.path.dirname(__file__), "golden", name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


def test_schedule_transfer_times_match_pages(orc):
    """The schedule's transfer model against the per-layer transfer times the
    pages print (tests/golden/layer_transfer_times.txt): the first block has
    nothing to hide behind, so its predicted stall is its transfer time; a
    layer whose predecessor computes at least that long is fully hidden (the
    pages' condition for the pipeline), and one that computes less leaves the
    difference as stall."""
    rows = _golden_rows("layer_transfer_times.txt")
    assert len(rows) == 5
    for _src, _link, bw, mb, ms, dec in rows:
        bw, b, ms, dec = float(bw) * 1e9, float(mb) * 1e6, float(ms), int(dec)
        t = b / bw  # seconds
        stall, _ = orc.schedule([b, b], [0, 0], [t, 0], [0, 0], bw, bw)
        # the printed value is the transfer time rounded to `dec` decimals (in ms)
        assert abs(stall[0] * 1e3 - ms) <= 0.5 * 10.0 ** -dec + 1e-9, (_link, stall[0])
        assert stall[1] == pytest.approx(0.0, abs=1e-12)
        stall, _ = orc.schedule([b, b], [0, 0], [0.5 * t, 0], [0, 0], bw, bw)
        assert stall[1] == pytest.approx(0.5 * t, rel=1e-12)


def test_attention_rows_matches_full_oracle(orc):
    """The O(S hd)-per-row attention used at long context equals the full
    oracle's forward and backward on every row of a small case."""
    from oracle.attention_rows import attention_rows
    rng = np.random.default_rng(31)
    S, nh, nkv, hd = 150, 4, 2, 16
    qkv = rng.standard_normal((S, (nh + 2 * nkv) * hd))
    dout = rng.standard_normal((S, nh * hd))
    o_ref, lse_ref = orc.attention_fwd(qkv, 1, S, nh, nkv, hd)
    d_ref = orc.attention_bwd(qkv, o_ref, lse_ref, dout, 1, S, nh, nkv, hd)
    q, k, v = qkv[:, :nh * hd], qkv[:, nh * hd:(nh + nkv) * hd], qkv[:, (nh + nkv) * hd:]
    rows = np.arange(S)
    r = attention_rows(q, k, v, dout, nh, nkv, hd, rows, rows)
    assert np.allclose(r["o"], o_ref, rtol=1e-10, atol=1e-12)
    assert np.allclose(r["lse"], lse_ref, rtol=1e-10, atol=1e-12)
    assert np.allclose(r["dq"], d_ref[:, :nh * hd], rtol=1e-9, atol=1e-11)
    assert np.allclose(r["dk"], d_ref[:, nh * hd:(nh + nkv) * hd], rtol=1e-9, atol=1e-11)
    assert np.allclose(r["dv"], d_ref[:, (nh + nkv) * hd:], rtol=1e-9, atol=1e-11)
    # a subset of rows gives the same values as the full computation
    sub = attention_rows(q, k, v, dout, nh, nkv, hd, [0, 77, 149], [140, 149])
    assert np.allclose(sub["dq"], r["dq"][[0, 77, 149]], rtol=1e-12, atol=1e-13)
    assert np.allclose(sub["dk"], r["dk"][[140, 149]], rtol=1e-12, atol=1e-13)
    assert np.all(r["dq_mag"] >= np.abs(r["dq"]) - 1e-12) and np.all(r["dv_mag"] >= np.abs(r["dv"]) - 1e-12)
