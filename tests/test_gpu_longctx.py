"""Attention parity at the long-context sizes (32K, 128K and 512K tokens, the
7.6B shape's 28 query heads / 4 KV heads of hd 128), where the full O(S^2)
oracle is out of reach: the library's forward and backward run on the whole
sequence and are compared on sampled rows with the oracle's exact
O(S hd)-per-row attention (oracle/attention_rows.py):

* o and LSE of 64 query rows per head (the first and last rows included);
* dq of the same rows, dk and dv of the last 64 key rows (they need every
  later query, which is at most 64 of them);
* two identities over the whole sequence, per kv head: sum_j dv_j equals the
  sum of dO over the group's heads and rows (every softmax row sums to 1), and
  sum_j dk_j = 0 (every dS row sums to 0).

Tolerances: the elementwise bounds of the op tests (BF16 output rounding plus
4 u times the magnitude of the summands, u = 2^-8); the identities allow
8 u times the root-sum-square of the terms, a bound on accumulated random
rounding, not a worst case.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from host_memory_centric_gb300 import ops  # noqa: E402
from oracle.attention_rows import attention_rows, rows_needed  # noqa: E402

NH, NKV, HD = 28, 4, 128
U = 2.0 ** -8


@pytest.fixture(autouse=True)
def _no_kernel_errors():
    ops.kernel_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert ops.kernel_error(clear=True) == 0


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.mark.parametrize("S", [32768, 131072, 524288])
def test_long_context_attention_sampled_rows(S):
    gen = torch.Generator(device="cuda").manual_seed(S)
    bf = torch.bfloat16
    ld = (NH + 2 * NKV) * HD
    qkv = (torch.randn(S, ld, generator=gen, device="cuda") * 0.5).to(bf)
    dout = torch.randn(S, NH * HD, generator=gen, device="cuda").to(bf)
    o = torch.empty(S, NH * HD, dtype=bf, device="cuda")
    lse = torch.empty(NH, S, dtype=torch.float32, device="cuda")
    ops.attention_fwd(qkv, 1, S, NH, NKV, HD, o, lse)
    dqkv = torch.full_like(qkv, float("nan"))
    scratch = torch.empty(ops.attention_bwd_scratch_bytes(1, S, NH, HD), dtype=torch.uint8, device="cuda")
    ops.attention_bwd(qkv, o, lse, dout, 1, S, NH, NKV, HD, dqkv, scratch)
    torch.cuda.synchronize()

    rng = np.random.default_rng(S + 1)
    q_rows = np.unique(np.concatenate([[0, 1, 127, 128, S // 2, S - 2, S - 1], rng.integers(0, S, 57)]))
    k_rows = np.arange(S - 64, S)
    idx = torch.as_tensor(rows_needed(q_rows, k_rows, S), device="cuda")
    qn = f64(qkv[idx, :NH * HD])  # only the query rows the reference reads
    dn = f64(dout[idx])
    k = f64(qkv[:, NH * HD:(NH + NKV) * HD])
    v = f64(qkv[:, (NH + NKV) * HD:])
    ref = attention_rows(qn, k, v, dn, NH, NKV, HD, q_rows, k_rows)

    qi = torch.as_tensor(q_rows, device="cuda")
    got_o = f64(o[qi])
    assert rel_l2(got_o, ref["o"]) <= 1e-2
    assert np.all(np.abs(got_o - ref["o"]) <= 1e-3 * np.abs(ref["o"]).max() + 2 ** -6 * np.abs(ref["o"]))
    got_lse = lse[:, qi].T.cpu().numpy().astype(np.float64)
    assert np.allclose(got_lse, ref["lse"], atol=2e-3)

    dq = f64(dqkv[qi, :NH * HD])
    assert rel_l2(dq, ref["dq"]) <= 2e-2
    assert np.all(np.abs(dq - ref["dq"]) <= 4 * U * ref["dq_mag"] + 2 ** -7 * np.abs(ref["dq"]) + 1e-6)
    ki = torch.as_tensor(k_rows, device="cuda")
    dk = f64(dqkv[ki, NH * HD:(NH + NKV) * HD])
    dv = f64(dqkv[ki, (NH + NKV) * HD:])
    for got, key in ((dk, "dk"), (dv, "dv")):
        assert rel_l2(got, ref[key]) <= 2e-2, key
        assert np.all(np.abs(got - ref[key]) <= 4 * U * ref[key + "_mag"] + 2 ** -7 * np.abs(ref[key]) + 1e-6), key

    # whole-sequence identities, per kv head and hd column
    dk_all = f64(dqkv[:, NH * HD:(NH + NKV) * HD]).reshape(S, NKV, HD)
    dv_all = f64(dqkv[:, (NH + NKV) * HD:]).reshape(S, NKV, HD)
    assert np.isfinite(dk_all).all() and np.isfinite(dv_all).all()
    do_all = dout.float().reshape(S, NKV, NH // NKV, HD).sum(dim=2).double().cpu().numpy()  # [S, NKV, HD]
    expect_v = do_all.sum(axis=0)
    tol_v = 8 * U * (np.sqrt((dv_all ** 2).sum(axis=0)) + np.sqrt((do_all ** 2).sum(axis=0)))
    assert np.all(np.abs(dv_all.sum(axis=0) - expect_v) <= tol_v)
    tol_k = 8 * U * np.sqrt((dk_all ** 2).sum(axis=0))
    assert np.all(np.abs(dk_all.sum(axis=0)) <= tol_k)
