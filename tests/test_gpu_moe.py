"""GPU parity of the routed mixture-of-experts path against the oracle.

The MoE layer (lilting.ch, MoE section: per token the router selects a few
experts and only those experts' weights are copied to the GPU) is checked
three ways:
* op level: mt_moe_ffn (router, top-k, expert-sorted grouped GEMMs, combine
  and the whole backward) against the oracle's layer on the same BF16
  inputs; the routing is an integer decision taken from FP32 logits on both
  sides, so each case first asserts that the oracle's smallest top-k margin
  is far above the FP32 summation error, then compares the selected experts
  exactly;
* whole step with routing that BF16 activations cannot flip: the embedding
  and router weights are set so that every token's top-k set is decided by
  a margin of several logit units (the oracle reports it, and the test
  asserts it), then the usual loss / gradient / teacher-forced Adam
  tolerances apply; half of the experts receive no token, which exercises
  streaming only the routed experts and Adam with a zero gradient.  (With
  unstructured weights a router fed BF16 activations and one fed FP32
  activations disagree on a few near-tied tokens per step, and a flipped
  token moves an expert's gradient by more than the tolerance: the
  decision itself is compared in the op-level test, on shared inputs);
* whole step with top_k = n_experts (no selection at all) at random init.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import host_memory_centric_gb300 as mt  # noqa: E402
from host_memory_centric_gb300 import configs, inputs, ops  # noqa: E402
from tests import protocol_check  # noqa: E402
from tests.test_gpu_step import oracle_shape, rel_l2, run_parity  # noqa: E402


@pytest.fixture(autouse=True)
def _no_kernel_errors():
    ops.kernel_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert ops.kernel_error(clear=True) == 0


def _bf(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("T,H,E,k,Fe,suppress,seed", [
    (300, 256, 8, 2, 384, 0, 3),        # ragged T, three 256-wide N tiles in W_gu
    (1000, 512, 16, 4, 128, 4, 11),     # 4 experts never chosen
    (64, 128, 8, 8, 64, 0, 5),          # every expert for every token
    (200, 128, 128, 8, 64, 0, 13),      # the largest expert count and top-k: 128 experts, 8 per token
    (3, 64, 16, 2, 64, 0, 17),          # three tokens: most experts unused, one partial tile each
])
def test_moe_ffn_matches_oracle(orc, T, H, E, k, Fe, suppress, seed):
    rng = np.random.default_rng(seed)
    yn = rng.standard_normal((T, H))
    if suppress:
        yn[:, 0] = 3.0
    x1 = rng.standard_normal((T, H))
    Wr = rng.standard_normal((E, H)) * (8.0 / math.sqrt(H))
    if suppress:
        Wr[E - suppress:, 0] = -40.0
    We = np.concatenate([rng.standard_normal((E, 2 * Fe * H)) / math.sqrt(H),
                         rng.standard_normal((E, H * Fe)) / math.sqrt(Fe)], axis=1)
    dout = rng.standard_normal((T, H))
    tens = [_bf(a).cuda() for a in (yn, x1, Wr, We, dout)]
    ref_in = [_f64(t) for t in tens]
    out, dyn, dWr, dWe, idx_o, gate_o, margin = orc.moe_layer(*ref_in, k, Fe)
    if k < E:
        assert margin > 1e-4, margin  # premise: no selection within FP32 rounding of a tie
    dev = torch.device("cuda")
    o_out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    o_dyn = torch.empty_like(o_out)
    o_dWr = torch.empty((E, H), dtype=torch.bfloat16, device=dev)
    o_dWe = torch.full((E, 3 * Fe * H), 7.0, dtype=torch.bfloat16, device=dev)
    o_idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    o_gate = torch.empty((T, k), dtype=torch.float32, device=dev)
    sc = torch.empty(ops.moe_scratch_bytes(T, H, E, k, Fe), dtype=torch.uint8, device=dev)
    ops.moe_ffn(*tens, k, Fe, o_out, o_dyn, o_dWr, o_dWe, o_idx, o_gate, sc)
    torch.cuda.synchronize()
    assert np.array_equal(o_idx.cpu().numpy(), idx_o)
    np.testing.assert_allclose(o_gate.cpu().numpy(), gate_o, rtol=2e-5, atol=1e-7)
    assert rel_l2(_f64(o_out), out) <= 1e-2
    assert rel_l2(_f64(o_dyn), dyn) <= 2e-2
    assert rel_l2(_f64(o_dWr), dWr) <= 2e-2
    got = _f64(o_dWe)
    routed = np.zeros(E, bool)
    routed[np.unique(idx_o)] = True
    assert not np.any(got[~routed])  # experts no token chose: zero gradient
    for e in np.flatnonzero(routed):
        assert rel_l2(got[e], dWe[e]) <= 2e-2, e
    if suppress:
        assert not routed[E - suppress:].any() and routed[:E - suppress].all()


def _structured_routing(c):
    """Store rewrite making every token's top-k set unambiguous: embedding
    column 1 is +1 for even and -1 for odd token ids (a zero-mean channel that
    dominates the normalised input of every layer), and router column 1 gives
    even tokens experts {0, 1} and odd tokens experts {2, 3} by about five
    logit units; experts 4..7 get no token.  The workloads using it train at
    lr 1e-4: Adam's first steps move every weight by about lr, and at 1e-3
    they reshape the 0.02-scale initial weights enough to erode the
    engineered margin within three steps."""
    import oracle

    def prep(m):
        lay = m.layout
        V, L = c["vocab"], c["n_layers"]
        th = m.read(0, mt.REGION_MASTER)
        eo, r, cc = lay[0]["tensors"][0]
        Em = th[eo:eo + r * cc].reshape(r, cc)
        Em[:, 1] = np.where(np.arange(V) % 2 == 0, 1.0, -1.0)
        m.write(0, mt.REGION_MASTER, th)
        m.write(0, mt.REGION_W, oracle.bf16_rne_fast(th))
        b = np.array([1.0, 0.9, -1.0, -0.9, 0.1, 0.0, -0.1, 0.05], np.float32)
        for j in range(1, L + 1):
            th = m.read(j, mt.REGION_MASTER)
            ro, E, H = lay[j]["tensors"][2]
            th[ro:ro + E * H].reshape(E, H)[:, 1] = b
            m.write(j, mt.REGION_MASTER, th)
            m.write(j, mt.REGION_W, oracle.bf16_rne_fast(th))
    return prep


def test_moe_step_parity_structured_routing(orc):
    c = configs.get("tiny_moe", lr=1e-4)
    report, log = run_parity(orc, c, 3, prepare=_structured_routing(c))
    for (step, loss, loss_ref, worst, margin) in report:
        assert margin > 3.0, (step, margin)
    assert protocol_check.mask_slabs(log) == protocol_check.mask_slabs(orc.protocol(oracle_shape(c), 3, 12, True, True))
    protocol_check.check(log)
    print("moe structured parity", report)


@pytest.mark.parametrize("rt", [dict(ckpt_interval=2, n_buffers=1), dict(ckpt_on_host=0, pin_store=1, n_grad_slabs=2)])
def test_moe_step_parity_recompute_and_placement(orc, rt):
    """The routed experts streamed with the shared weights in recompute and
    backward visits (interval 2, single buffer, just-in-time pack of the
    routed experts' rows) and with device checkpoints / pinned store."""
    c = configs.get("tiny_moe", lr=1e-4)
    report, log = run_parity(orc, c, 2, prepare=_structured_routing(c), **rt)
    assert all(r[4] > 2.0 for r in report)
    protocol_check.check(log)


def test_moe_step_parity_all_experts(orc):
    """top_k = n_experts: no routing decision; random init; all 8 experts of
    every token weighted by the softmax of all router logits."""
    c = configs.get("tiny_moe", top_k=8)
    report, _ = run_parity(orc, c, 2)
    assert all(math.isinf(r[4]) for r in report)


def test_moe_streams_only_routed_experts():
    """With half of the experts unused, the forward and backward copies and
    the gradient export move only the shared tensors and the used experts."""
    c = configs.get("tiny_moe", lr=1e-4)
    m = mt.Model(c, seed=1234, n_host_threads=4)
    _structured_routing(c)(m)
    lay = m.layout
    L = c["n_layers"]
    tok = inputs.tokens_for(c, 0)
    m.set_tokens(tok)
    s0 = m.stats()
    m.train_step(0)
    m.sync()
    s1 = m.stats()
    even = int((tok % 2 == 0).sum())
    for j in range(1, L + 1):  # parity decides: even tokens -> experts 0, 1; odd -> 2, 3
        assert m.expert_counts(j).tolist() == [even, even, tok.size - even, tok.size - even, 0, 0, 0, 0], j
    eo, E, row = lay[1]["tensors"][3]
    unused = 4 * row * 2  # bytes of experts 4..7 of one layer
    h2d = s1["h2d_bytes"] - s0["h2d_bytes"]
    d2h = s1["d2h_bytes"] - s0["d2h_bytes"]
    for j in range(1, L + 1):
        ge = m.read(j, mt.REGION_G)[eo:eo + E * row].reshape(E, row)
        assert not np.any(ge[4:]) and np.all(np.any(ge[:4] != 0, axis=1)), j
    m.close()
    ref = mt.Model(c, seed=1234, n_host_threads=4)  # random init: every expert gets tokens
    ref.set_tokens(tok)
    r0 = ref.stats()
    ref.train_step(0)
    ref.sync()
    r1 = ref.stats()
    for j in range(1, L + 1):
        ge = ref.read(j, mt.REGION_G)[eo:eo + E * row].reshape(E, row)
        assert np.all(np.any(ge != 0, axis=1)), j
    ref.close()
    # each decoder layer is copied in twice per step (forward, backward) and
    # exported once, each time without the four unused experts' rows
    dense_h2d = r1["h2d_bytes"] - r0["h2d_bytes"]
    dense_d2h = r1["d2h_bytes"] - r0["d2h_bytes"]
    assert dense_h2d - h2d == 2 * L * unused
    assert dense_d2h - d2h == L * unused


def test_moe_full_width_zero_head_properties():
    """The benchmark's MoE shape at full width (2 of its layers, 4 x 4096
    tokens): with a zero LM head the loss is ln V and every upstream gradient,
    router and experts included, is exactly zero; every expert gets tokens."""
    c = configs.get("moe", n_layers=2)
    V = c["vocab"]
    L = c["n_layers"]
    m = mt.Model(c, seed=1234)
    head = m.layout[L + 1]
    eo, r, cc = head["tensors"][1]
    w = m.read(L + 1, mt.REGION_W)
    w[eo:eo + r * cc] = 0
    m.write(L + 1, mt.REGION_W, w)
    m.set_tokens(inputs.tokens_for(c, 0))
    loss = m.train_step(0)
    m.sync()
    assert loss == pytest.approx(math.log(V), rel=2e-6)
    for j in range(L + 1):
        assert not np.any(m.read(j, mt.REGION_G)), j
    m.close()


def test_moe_full_width_one_layer_parity(orc):
    """The `moe` shape at full width (hidden 2880, 64 x 64 heads / 8 KV, 32
    experts of FFN 2880, top-4, vocabulary 201088), one decoder layer and one
    64-token sequence, against the oracle with the same unambiguous routing
    (a +-16 embedding sign channel and router column 1)."""
    c = configs.get("moe", n_layers=1, batch=1, seq=64, micro=1, lr=1e-4)
    E = c["n_experts"]

    def prep(m):
        import oracle
        lay = m.layout
        V = c["vocab"]
        th = m.read(0, mt.REGION_MASTER)
        eo, r, cc = lay[0]["tensors"][0]
        # +-16: at this width the attention output at init (about N(0, 1.4) per element for the
        # first positions) must not flip the sign channel
        th[eo:eo + r * cc].reshape(r, cc)[:, 1] = np.where(np.arange(V) % 2 == 0, 16.0, -16.0)
        m.write(0, mt.REGION_MASTER, th)
        m.write(0, mt.REGION_W, oracle.bf16_rne_fast(th))
        b = np.zeros(E, np.float32)
        b[:4], b[4:8] = [1.0, 0.9, 0.8, 0.7], [-1.0, -0.9, -0.8, -0.7]  # even -> 0..3, odd -> 4..7
        th = m.read(1, mt.REGION_MASTER)
        ro, EE, H = lay[1]["tensors"][2]
        th[ro:ro + EE * H].reshape(EE, H)[:, 1] = b
        m.write(1, mt.REGION_MASTER, th)
        m.write(1, mt.REGION_W, oracle.bf16_rne_fast(th))

    report, _ = run_parity(orc, c, 1, prepare=prep)
    assert report[0][4] > 1.0, report
