"""GPU parity of each device op (through the C ABI) against the CPU oracle.

Inputs are BF16 values; the oracle computes in fp64 on the same values.
Shapes span several tiles and end in ragged tails.  Tolerances follow from
the arithmetic: outputs are rounded to BF16 (relative step 2^-8), sums are
FP32, so elementwise |gpu - ref| <= atol + 2^-6 |ref| and relative L2 error
<= 1e-2 (5e-3 for single roundings).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import host_memory_centric_gb300 as mt  # noqa: E402
from host_memory_centric_gb300 import ops  # noqa: E402


def bf(x, dev="cuda"):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(dev).contiguous()


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def close(gpu, ref, rel=1e-2, elem_rtol=2 ** -6, atol=None):
    """Relative L2 bound plus an elementwise bound |d| <= atol + elem_rtol |ref|;
    atol may be an array (the magnitude of the terms an element sums)."""
    if atol is None:
        atol = 1e-3 * (np.abs(ref).max() + 1e-30)
    assert rel_l2(gpu, ref) <= rel, rel_l2(gpu, ref)
    bad = np.abs(gpu - ref) > atol + elem_rtol * np.abs(ref)
    assert not bad.any(), (int(bad.sum()), float(np.abs(gpu - ref).max()))


@pytest.fixture(autouse=True)
def _no_kernel_errors():
    ops.kernel_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert ops.kernel_error(clear=True) == 0


def rnd(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


# ------------------------------------------------------------------ GEMM
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (128, 256, 64), (1000, 264, 1032)])
def test_gemm_majors(orc, a_mn, b_mn, M, N, K):
    A = rnd((M, K), 1); B = rnd((N, K), 2)
    # MN-major operands are stored [K][MN] with the row stride padded to 8
    # elements (16 bytes), as the tensor-memory-access unit requires
    pad = lambda n: (n + 7) // 8 * 8
    if a_mn:
        At = np.zeros((K, pad(M)), np.float32); At[:, :M] = A.T
        Ag, lda = bf(At), pad(M)
    else:
        Ag, lda = bf(A), K
    if b_mn:
        Bt = np.zeros((K, pad(N)), np.float32); Bt[:, :N] = B.T
        Bg, ldb = bf(Bt), pad(N)
    else:
        Bg, ldb = bf(B), K
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ops.gemm(Ag, Bg, M, N, K, a_mn=a_mn, b_mn=b_mn, lda=lda, ldb=ldb, D=D)
    ref = orc.linear_fwd(f64(bf(A)), f64(bf(B)))
    close(f64(D), ref, rel=5e-3)


def test_gemm_persistent_many_tiles_long_k(orc):
    M, N, K = 2304, 2560, 4096  # 18 x 10 tiles (> SM count after swizzle), 64 k-blocks
    A = rnd((M, K), 3, 0.5); B = rnd((N, K), 4, 0.5)
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ops.gemm(bf(A), bf(B), M, N, K, D=D)
    # oracle on sampled rows (each output row is an independent dot-product set)
    rows = np.random.default_rng(5).choice(M, 24, replace=False)
    Ab = f64(bf(A))[rows]; Bb = f64(bf(B))
    ref = orc.linear_fwd(Ab, Bb)
    close(f64(D)[rows], ref, rel=5e-3)


def test_gemm_residual_and_fp32_accumulate(orc):
    M, N, K = 200, 296, 136  # N ragged against the 256-wide tile, row stride 16-byte aligned
    A1, A2 = rnd((M, K), 6), rnd((M, K), 7)
    B = rnd((N, K), 8)
    R = rnd((M, N), 9)
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    acc = torch.empty(M, N, dtype=torch.float32, device="cuda")
    ops.gemm(bf(A1), bf(B), M, N, K, Dacc=acc, acc_mode=1)
    ops.gemm(bf(A2), bf(B), M, N, K, D=D, R=bf(R), Dacc=acc, acc_mode=2)
    ref = orc.linear_fwd(f64(bf(A1)), f64(bf(B))) + orc.linear_fwd(f64(bf(A2)), f64(bf(B)))
    close(acc.double().cpu().numpy(), ref, rel=1e-5, elem_rtol=1e-5, atol=1e-4)
    close(f64(D), ref + f64(bf(R)), rel=5e-3)


def test_gemm_dgrad_wgrad_forms(orc):
    T, N, K = 384, 264, 200
    dY = rnd((T, N), 10); W = rnd((N, K), 11); X = rnd((T, K), 12)
    dX = torch.empty(T, K, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
    # dX = dY W : A = dY K-major, B = W as [K'=N][N'=K] MN-major
    ops.gemm(bf(dY), bf(W), T, K, N, b_mn=True, ldb=K, D=dX)
    # dW = dY^T X : A = dY as [K'=T][M'=N] MN-major, B = X as [K'=T][N'=K] MN-major
    ops.gemm(bf(dY), bf(X), N, K, T, a_mn=True, lda=N, b_mn=True, ldb=K, D=dW)
    close(f64(dX), orc.linear_dgrad(f64(bf(dY)), f64(bf(W))), rel=5e-3)
    close(f64(dW), orc.linear_wgrad(f64(bf(dY)), f64(bf(X))), rel=5e-3)


def test_gemm_rejects_misaligned():
    A = torch.zeros(64, 20, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mt.MtError):
        ops.gemm(A, A, 64, 64, 20, lda=20, ldb=20, D=torch.empty(64, 64, dtype=torch.bfloat16, device="cuda"))


# ------------------------------------------------------------------ RMSNorm / RoPE / SwiGLU
# H picks the row kernels' forms (forward: vectors per lane 1, 4, 8, 12, 16
# and the generic re-reading form; backward: per-warp dgamma rows up to
# H = 2048, chunked column passes above); T spans ragged row blocks and, at
# 4099, more partial blocks than the dgamma reduction's eight slices.
@pytest.mark.parametrize("T,H,with_res", [(333, 520, True), (1, 8, True), (4099, 2048, True), (64, 2048, False),
                                          (257, 2880, False), (130, 3584, True), (70, 5120, True)])
def test_rmsnorm_fwd_bwd(orc, T, H, with_res):
    x = rnd((T, H), 13); g = 1 + 0.1 * rnd(H, 14); dy = rnd((T, H), 15); dres = rnd((T, H), 16)
    xg, gg = bf(x), bf(g)
    y = torch.empty_like(xg); r = torch.empty(T, dtype=torch.float32, device="cuda")
    ops.rmsnorm_fwd(xg, gg, 1e-6, y, r)
    yr, rr = orc.rmsnorm_fwd(f64(xg), f64(gg), 1e-6)
    close(f64(y), yr, rel=5e-3)
    assert np.allclose(r.cpu().numpy(), rr, rtol=1e-5)
    dx = torch.empty_like(xg); dgm = torch.empty(H, dtype=torch.bfloat16, device="cuda")
    scratch = torch.empty(ops.rmsnorm_bwd_scratch_bytes(T, H), dtype=torch.uint8, device="cuda")
    ops.rmsnorm_bwd(bf(dy), xg, gg, r, bf(dres) if with_res else None, dx, dgm, scratch)
    dxr, dgr = orc.rmsnorm_bwd(f64(bf(dy)), f64(xg), f64(gg), rr)
    close(f64(dx), dxr + (f64(bf(dres)) if with_res else 0.0), rel=5e-3)
    close(f64(dgm), dgr, rel=5e-3)
    # dgamma is reduced in a fixed order: a second run gives the same bits
    dx2 = torch.empty_like(xg); dgm2 = torch.empty_like(dgm)
    ops.rmsnorm_bwd(bf(dy), xg, gg, r, bf(dres) if with_res else None, dx2, dgm2, scratch)
    assert torch.equal(dgm, dgm2) and torch.equal(dx, dx2)


@pytest.mark.parametrize("hd", [64, 128])
def test_rope_fwd_inverse(orc, hd):
    n_seq, S, nh = 3, 77, 5
    x = rnd((n_seq * S, (nh + 2) * hd), 17)
    xg = bf(x)
    ref_in = f64(xg)
    cs = torch.as_tensor(ops.rope_table(S, hd, 1e6)).cuda()
    ops.rope(xg, nh, hd, S, cs)
    ref = orc.rope(ref_in, n_seq, S, nh, hd, 1e6)
    close(f64(xg), ref, rel=5e-3)
    ops.rope(xg, nh, hd, S, cs, inverse=True)
    # the round trip re-rounds rotated pairs: error scales with the pair norm
    r = ref_in.reshape(n_seq * S, nh + 2, 2, hd // 2)
    pair = np.broadcast_to(np.hypot(r[:, :, :1], r[:, :, 1:]), r.shape).reshape(ref_in.shape)
    close(f64(xg), ref_in, rel=1e-2, elem_rtol=0.0, atol=2 ** -6 * pair + 1e-6)


def test_swiglu(orc):
    T, F = 129, 264
    gu = rnd((T, 2 * F), 18, 2.0); dh = rnd((T, F), 19)
    gug = bf(gu)
    h = torch.empty(T, F, dtype=torch.bfloat16, device="cuda")
    ops.swiglu_fwd(gug, h)
    close(f64(h), orc.swiglu_fwd(f64(gug)), rel=5e-3)
    dgu = torch.empty_like(gug)
    ops.swiglu_bwd(gug, bf(dh), dgu)
    close(f64(dgu), orc.swiglu_bwd(f64(gug), f64(bf(dh))), rel=5e-3)


# ------------------------------------------------------------------ attention
@pytest.mark.parametrize("hd,nh,nkv,S,n_seq", [
    (64, 4, 4, 150, 2),    # MHA, ragged 128-tile, two sequences
    (128, 4, 2, 200, 1),   # ragged 64- and 128-sub-tiles
    (128, 8, 2, 64, 3),    # one sub-tile per sequence
    (128, 7, 1, 300, 1),   # seven query heads per kv head (the 7.6B grouping)
    (128, 2, 2, 33, 2),    # shorter than one sub-tile
    (64, 2, 1, 129, 1),    # one row past a tile
    (128, 4, 4, 512, 1),   # several full tiles on and off the diagonal
    # more work items than SMs: a persistent CTA runs several (query tile,
    # head, sequence) items one after another
    (64, 16, 4, 384, 4),   # 192 items of 1 to 3 key tiles
    (128, 40, 8, 100, 4),  # 160 single-tile items, groups of 5 (the 14.7B grouping)
])
def test_attention_fwd_bwd(orc, hd, nh, nkv, S, n_seq):
    T = n_seq * S
    qkv = rnd((T, (nh + 2 * nkv) * hd), 20)
    dout = rnd((T, nh * hd), 21)
    qg = bf(qkv)
    o = torch.empty(T, nh * hd, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(nh, T, dtype=torch.float32, device="cuda")
    ops.attention_fwd(qg, n_seq, S, nh, nkv, hd, o, lse)
    o_ref, lse_ref = orc.attention_fwd(f64(qg), n_seq, S, nh, nkv, hd)
    close(f64(o), o_ref, rel=1e-2)
    assert np.allclose(lse.cpu().numpy().T, lse_ref, atol=2e-3)
    dq = torch.full_like(qg, float("nan"))  # every element must be written
    scratch = torch.empty(ops.attention_bwd_scratch_bytes(n_seq, S, nh, hd), dtype=torch.uint8, device="cuda")
    dg = bf(dout)
    ops.attention_bwd(qg, o, lse, dg, n_seq, S, nh, nkv, hd, dq, scratch)
    d_ref = orc.attention_bwd(f64(qg), o_ref, lse_ref, f64(dg), n_seq, S, nh, nkv, hd)
    close(f64(dq), d_ref, rel=2e-2, elem_rtol=2 ** -7, atol=attn_bwd_error_scale(f64(qg), f64(dg), lse_ref,
                                                                                  n_seq, S, nh, nkv, hd))


def attn_bwd_error_scale(qkv, dout, lse, n_seq, S, nh, nkv, hd, c=4.0, u=2.0 ** -8):
    """Elementwise error allowance of the attention backward.  P and dS enter
    the tensor-core products as BF16, so each summand of dq_i = scale
    sum_j dS_ij k_j carries a relative error ~u: the allowance of an element is
    c u times the sum of its summands' magnitudes (bounded with max |k|, |q|,
    |dO|), not a multiple of the (possibly cancelled) result."""
    T = n_seq * S
    ld = (nh + 2 * nkv) * hd
    grp = nh // nkv
    scale = 1.0 / np.sqrt(hd)
    q = qkv[:, :nh * hd].reshape(n_seq, S, nh, hd)
    k = qkv[:, nh * hd:(nh + nkv) * hd].reshape(n_seq, S, nkv, hd)
    v = qkv[:, (nh + nkv) * hd:].reshape(n_seq, S, nkv, hd)
    do = dout.reshape(n_seq, S, nh, hd)
    out = np.zeros((n_seq, S, ld))
    mask = np.tril(np.ones((S, S), bool))
    for n in range(n_seq):
        for h in range(nh):
            g = h // grp
            s = q[n, :, h] @ k[n, :, g].T * scale
            p = np.where(mask, np.exp(s - lse[n * S:(n + 1) * S, h][:, None]), 0.0)
            dp = do[n, :, h] @ v[n, :, g].T
            D = (p * dp).sum(1, keepdims=True)
            w = p * (np.abs(dp) + np.abs(D))
            out[n, :, h * hd:(h + 1) * hd] += (c * u * scale * np.abs(k[n, :, g]).max() * w.sum(1))[:, None]
            kc = (nh + g) * hd
            out[n, :, kc:kc + hd] += (c * u * scale * np.abs(q[n, :, h]).max() * w.sum(0))[:, None]
            vc = (nh + nkv + g) * hd
            out[n, :, vc:vc + hd] += (c * u * np.abs(do[n, :, h]).max() * p.sum(0))[:, None]
    return out.reshape(T, ld) + 1e-6


# ------------------------------------------------------------------ embedding / CE
def test_embedding_fwd_bwd():
    V, H, T = 301, 264, 500
    E = rnd((V, H), 22)
    tok = np.random.default_rng(23).integers(0, V, T).astype(np.int32)
    Eg = bf(E)
    X = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    ops.embed_fwd(torch.as_tensor(tok).cuda(), Eg, X)
    assert torch.equal(X.cpu(), Eg.cpu()[torch.as_tensor(tok).long()])
    dX = rnd((T, H), 24)
    rs, rows = ops.token_csr(tok, V)
    dE = torch.full((V, H), 7.0, dtype=torch.bfloat16, device="cuda")
    ops.embed_bwd(torch.as_tensor(rs).cuda(), torch.as_tensor(rows).cuda(), bf(dX), V, dE)
    ref = np.zeros((V, H))
    np.add.at(ref, tok, f64(bf(dX)))
    close(f64(dE), ref, rel=5e-3)


# V = 1000: one 8-logit group per thread at most; 32000: several groups per
# thread and a ragged last round; 1001: the scalar path.  ramp: logits rising
# along the row, so the running max moves at almost every group.
@pytest.mark.parametrize("n_seq,S,V,ramp", [(3, 50, 1000, False), (2, 20, 32000, False), (2, 20, 32000, True),
                                            (2, 30, 1001, False)])
def test_cross_entropy(orc, n_seq, S, V, ramp):
    T = n_seq * S
    z = rnd((T, V), 25, 2.0)
    if ramp:
        z = z + np.linspace(-12.0, 12.0, V, dtype=np.float32)
    tok = np.random.default_rng(26).integers(0, V, T).astype(np.int32)
    tgt = np.array([tok[t + 1] if (t % S) < S - 1 else -1 for t in range(T)], dtype=np.int32)
    zg = bf(z)
    zin = f64(zg)
    norm = n_seq * (S - 1)
    rl = torch.empty(T, dtype=torch.float32, device="cuda")
    ops.cross_entropy(zg, torch.as_tensor(tgt).cuda(), 1.0 / norm, rl)
    loss_ref, dl_ref = orc.cross_entropy(zin, tok, n_seq, S, norm)
    assert float(rl.sum()) / norm == pytest.approx(loss_ref, rel=1e-4)
    close(f64(zg), dl_ref, rel=1e-2, atol=1e-3 * np.abs(dl_ref).max())


def test_gemm_pair_in_one_launch(orc):
    """wgrad (both operands MN-major) and dgrad of one projection in one launch."""
    T, N, K = 320, 264, 200
    dY = rnd((T, N), 30); X = rnd((T, K), 31); W = rnd((N, K), 32)
    dYg, Xg, Wg = bf(dY), bf(X), bf(W)
    dW = torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
    dX = torch.empty(T, K, dtype=torch.bfloat16, device="cuda")
    ops.gemm2([dict(A=dYg, B=Xg, M=N, N=K, K=T, a_mn=1, b_mn=1, lda=N, ldb=K, D=dW),
               dict(A=dYg, B=Wg, M=T, N=K, K=N, b_mn=1, ldb=K, D=dX)])
    close(f64(dW), orc.linear_wgrad(f64(dYg), f64(Xg)), rel=5e-3)
    close(f64(dX), orc.linear_dgrad(f64(dYg), f64(Wg)), rel=5e-3)
