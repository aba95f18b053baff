"""The CTA-pair GEMM (mt_gemm_mode 1): two SMs of one cluster compute one
256 x 256 output tile with cta_group::2 MMAs, each holding half of A's rows
and half of B's rows in its shared memory and its 128 rows of the
accumulator in its tensor memory.

It is checked against the oracle in every operand layout on shapes that end
in ragged tails (rows, columns and K), in the epilogue forms the training
step uses, in the two-GEMM launch, and against the one-CTA tiling, which
accumulates the same K blocks in the same order and must agree bit for bit;
both tile orders of the pair (tiles drawn from a per-launch counter, and
every n-th tile) are run.  Many successive launches reuse the counters, which
the last draw of each launch resets.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from host_memory_centric_gb300 import configs, inputs, ops  # noqa: E402
import host_memory_centric_gb300 as mt  # noqa: E402
from tests.test_gpu_ops import bf, close, f64, rnd  # noqa: E402


@pytest.fixture(autouse=True)
def _no_kernel_errors():
    ops.kernel_error(clear=True)
    yield
    torch.cuda.synchronize()
    assert ops.kernel_error(clear=True) == 0


@pytest.fixture
def pair_mode():
    prev = ops.gemm_mode(1)
    yield
    ops.gemm_mode(prev)


def all_modes(fn, modes=(0, 1, 2)):
    """fn() under the one-CTA tiling (mode 0), CTA pairs drawing tiles from a
    counter (1), CTA pairs in static order (2) and, where asked, counter order
    without the 512-wide tiles of long-K launches (3)."""
    prev = ops.gemm_mode(-1)
    out = []
    try:
        for mode in modes:
            ops.gemm_mode(mode)
            out.append(fn())
    finally:
        ops.gemm_mode(prev)
    return out


def test_mode_switch_reads_and_sets():
    prev = ops.gemm_mode(-1)
    assert prev in (0, 1)
    assert ops.gemm_mode(1) == prev
    assert ops.gemm_mode(2) == 1
    assert ops.gemm_mode(3) == 2
    assert ops.gemm_mode(7) == 3  # ignored
    assert ops.gemm_mode(prev) == 3
    assert ops.gemm_mode(-1) == prev


def test_single_pair_tile(orc, pair_mode):
    """One 256 x 256 tile, one K block: the smallest case of the pair."""
    M = N = 256
    K = 64
    A = rnd((M, K), 1); B = rnd((N, K), 2)
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ops.gemm(bf(A), bf(B), M, N, K, D=D)
    close(f64(D), orc.linear_fwd(f64(bf(A)), f64(bf(B))), rel=5e-3)


def _majors_case(a_mn, b_mn, M, N, K, seed):
    A = rnd((M, K), seed); B = rnd((N, K), seed + 1)
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

    def run():
        D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        ops.gemm(Ag, Bg, M, N, K, a_mn=a_mn, b_mn=b_mn, lda=lda, ldb=ldb, D=D)
        torch.cuda.synchronize()
        return D

    return A, B, run


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (300, 520, 200), (128, 136, 64), (1000, 264, 1032),
                                   (520, 1800, 328)])
def test_pair_majors_against_oracle_and_one_cta(orc, a_mn, b_mn, M, N, K):
    """M = 128 and 300 leave the odd CTA of a pair with no rows or a few;
    N = 136 and 264 leave it no columns of B or a few."""
    A, B, run = _majors_case(a_mn, b_mn, M, N, K, 3 * M + N)
    one, two, static = all_modes(run)
    close(f64(two), orc.linear_fwd(f64(bf(A)), f64(bf(B))), rel=5e-3)
    assert torch.equal(one, two) and torch.equal(one, static)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_wide_tiles_at_long_k(orc, a_mn, b_mn):
    """K >= 8192 and N >= 512: the pair launches use 256 x 512 tiles with one
    512-column accumulator (modes 1 and 2; mode 3 keeps 256 x 256).  N = 1320
    leaves the last wide tile with its first half inside and 40 columns of
    its second; M = 300 and K = 8200 are ragged too."""
    M, N, K = 300, 1320, 8200
    A, B, run = _majors_case(a_mn, b_mn, M, N, K, 77 + 2 * a_mn + b_mn)
    one, two, static, narrow = all_modes(run, (0, 1, 2, 3))
    assert torch.equal(one, two) and torch.equal(one, static) and torch.equal(one, narrow)
    rows = np.random.default_rng(9).choice(M, 32, replace=False)
    close(f64(two)[rows], orc.linear_fwd(f64(bf(A))[rows], f64(bf(B))), rel=5e-3)


def test_wide_wgrad_dgrad_in_one_launch(orc):
    """Both GEMMs of the launch have K >= 8192 (T and N), so it runs wide."""
    T, N, K = 8200, 8256, 600
    dY = rnd((T, N), 40, 0.5); X = rnd((T, K), 41, 0.5); W = rnd((N, K), 42, 0.5)
    dYg, Xg, Wg = bf(dY), bf(X), bf(W)

    def run():
        dW = torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
        dX = torch.empty(T, K, dtype=torch.bfloat16, device="cuda")
        ops.gemm2([dict(A=dYg, B=Xg, M=N, N=K, K=T, a_mn=1, b_mn=1, lda=N, ldb=K, D=dW),
                   dict(A=dYg, B=Wg, M=T, N=K, K=N, b_mn=1, ldb=K, D=dX)])
        torch.cuda.synchronize()
        return dW, dX

    (dW1, dX1), (dW2, dX2), (dW3, dX3) = all_modes(run, (0, 1, 3))
    assert torch.equal(dW1, dW2) and torch.equal(dX1, dX2)
    assert torch.equal(dW1, dW3) and torch.equal(dX1, dX3)
    rng = np.random.default_rng(10)
    rw, rx = rng.choice(N, 16, replace=False), rng.choice(T, 16, replace=False)
    dY64, X64, W64 = f64(dYg), f64(Xg), f64(Wg)
    close(f64(dW2)[rw], orc.linear_fwd(np.ascontiguousarray(dY64[:, rw].T), np.ascontiguousarray(X64.T)), rel=5e-3)
    close(f64(dX2)[rx], orc.linear_fwd(dY64[rx], np.ascontiguousarray(W64.T)), rel=5e-3)


def test_counter_reuse_over_many_launches(orc, pair_mode):
    """More launches than there are tile counters (1024): every launch finds
    its counter at zero, so every output tile is computed each time."""
    M, N, K = 520, 776, 64  # 3 x 4 pair tiles
    A = rnd((M, K), 11); B = rnd((N, K), 12)
    Ag, Bg = bf(A), bf(B)
    ref = orc.linear_fwd(f64(Ag), f64(Bg))
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    first = None
    for i in range(1100):
        D.fill_(float("nan"))
        ops.gemm(Ag, Bg, M, N, K, D=D)
        if i in (0, 1023, 1024, 1099):
            torch.cuda.synchronize()
            assert not torch.isnan(D).any(), i
            if first is None:
                first = D.clone()
                close(f64(D), ref, rel=5e-3)
            assert torch.equal(D, first), i


def test_pair_many_tiles_long_k(orc):
    """More pair tiles than resident pairs and 64 K blocks (the persistent
    loop wraps the stage ring many times); sampled rows against the oracle."""
    M, N, K = 4352, 2816, 4096  # 17 x 11 pair tiles
    A = rnd((M, K), 5, 0.5); B = rnd((N, K), 6, 0.5)
    Ag, Bg = bf(A), bf(B)

    def run():
        D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        ops.gemm(Ag, Bg, M, N, K, D=D)
        torch.cuda.synchronize()
        return D

    one, two, static = all_modes(run)
    assert torch.equal(one, two) and torch.equal(one, static)
    rows = np.random.default_rng(7).choice(M, 24, replace=False)
    close(f64(two)[rows], orc.linear_fwd(f64(Ag)[rows], f64(Bg)), rel=5e-3)


def test_pair_residual_and_fp32_accumulate(orc, pair_mode):
    M, N, K = 300, 296, 136
    A1, A2, B, R = rnd((M, K), 6), rnd((M, K), 7), rnd((N, K), 8), rnd((M, N), 9)
    D = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    acc = torch.empty(M, N, dtype=torch.float32, device="cuda")
    ops.gemm(bf(A1), bf(B), M, N, K, Dacc=acc, acc_mode=1)
    ops.gemm(bf(A2), bf(B), M, N, K, D=D, R=bf(R), Dacc=acc, acc_mode=2)
    ref = orc.linear_fwd(f64(bf(A1)), f64(bf(B))) + orc.linear_fwd(f64(bf(A2)), f64(bf(B)))
    close(acc.double().cpu().numpy(), ref, rel=1e-5, elem_rtol=1e-5, atol=1e-4)
    close(f64(D), ref + f64(bf(R)), rel=5e-3)


def test_pair_wgrad_dgrad_in_one_launch(orc):
    T, N, K = 320, 264, 200
    dY = rnd((T, N), 30); X = rnd((T, K), 31); W = rnd((N, K), 32)
    dYg, Xg, Wg = bf(dY), bf(X), bf(W)

    def run():
        dW = torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
        dX = torch.empty(T, K, dtype=torch.bfloat16, device="cuda")
        ops.gemm2([dict(A=dYg, B=Xg, M=N, N=K, K=T, a_mn=1, b_mn=1, lda=N, ldb=K, D=dW),
                   dict(A=dYg, B=Wg, M=T, N=K, K=N, b_mn=1, ldb=K, D=dX)])
        torch.cuda.synchronize()
        return dW, dX

    (dW1, dX1), (dW2, dX2), (dW3, dX3) = all_modes(run)
    close(f64(dW2), orc.linear_wgrad(f64(dYg), f64(Xg)), rel=5e-3)
    close(f64(dX2), orc.linear_dgrad(f64(dYg), f64(Wg)), rel=5e-3)
    assert torch.equal(dW1, dW2) and torch.equal(dX1, dX2)
    assert torch.equal(dW1, dW3) and torch.equal(dX1, dX3)


def test_training_step_identical_under_pairs():
    """A whole training step (dense GEMMs of every visit) gives the same loss
    and the same updated parameters bit for bit under either tiling."""
    c = configs.get("tiny", n_layers=2)
    tok = inputs.tokens_for(c, 0)

    def run():
        m = mt.Model(c, seed=11)
        m.set_tokens(tok)
        loss = m.train_step(0)
        m.sync()
        w = [m.read(j, mt.REGION_MASTER) for j in range(len(m.layout))]
        m.close()
        return loss, w

    (l1, w1), (l2, w2), (l3, w3) = all_modes(run)
    assert l1 == l2 == l3
    for a, b, c3 in zip(w1, w2, w3):
        assert np.array_equal(a, b) and np.array_equal(a, c3)
