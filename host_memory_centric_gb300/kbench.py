"""Kernel micro-benchmark: one libmt device op at a chosen shape, timed with
CUDA events on the launching stream after warm-up (inputs larger than L2
unless the shape is small).

python -m host_memory_centric_gb300.kbench gemm --M 8192 --N 11264 --K 2048 [--a-mn] [--b-mn] [--gemm-mode 1]
python -m host_memory_centric_gb300.kbench attn_fwd --S 2048 --nseq 4 --nh 16 --nkv 4 --hd 128
python -m host_memory_centric_gb300.kbench attn_bwd --S 2048 --nseq 4 --nh 16 --nkv 4 --hd 128
python -m host_memory_centric_gb300.kbench rmsnorm_bwd --T 8192 --H 2048
python -m host_memory_centric_gb300.kbench cross_entropy --T 8192 --V 32000
python -m host_memory_centric_gb300.kbench moe_ffn --T 16384 --H 2880 --E 32 --k 4 --Fe 2880
python -m host_memory_centric_gb300.kbench layer_gemms --config 7.6b
"""
from __future__ import annotations

import argparse
import json

import torch

from . import ops


def timeit(fn, iters, warmup):
    for _ in range(warmup):
        fn()
    s = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(s)
    for _ in range(iters):
        fn()
    b.record(s)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("op")
    ap.add_argument("--M", type=int, default=8192)
    ap.add_argument("--N", type=int, default=11264)
    ap.add_argument("--K", type=int, default=2048)
    ap.add_argument("--a-mn", action="store_true")
    ap.add_argument("--b-mn", action="store_true")
    ap.add_argument("--S", type=int, default=2048)
    ap.add_argument("--nseq", type=int, default=4)
    ap.add_argument("--nh", type=int, default=16)
    ap.add_argument("--nkv", type=int, default=4)
    ap.add_argument("--hd", type=int, default=128)
    ap.add_argument("--T", type=int, default=8192)
    ap.add_argument("--H", type=int, default=2048)
    ap.add_argument("--V", type=int, default=32000)
    ap.add_argument("--E", type=int, default=32)
    ap.add_argument("--k", type=int, default=4)
    ap.add_argument("--Fe", type=int, default=2880)
    ap.add_argument("--config", default="7.6b")
    ap.add_argument("--no-head", action="store_true", help="layer_gemms: leave out the LM-head forms")
    ap.add_argument("--gemm-mode", type=int, default=-1,
                    help="dense GEMM tiling: 0 one CTA per 128 x 256 tile; CTA pairs per 256 x 256 tile "
                         "(256 x 512 at long K), 1 drawing tiles from a counter, 2 every n-th tile, "
                         "3 as 1 without the 512-wide tiles")
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    a = ap.parse_args()
    torch.manual_seed(0)
    bf = torch.bfloat16
    dev = "cuda"
    if a.gemm_mode >= 0:
        ops.gemm_mode(a.gemm_mode)
    res = {"op": a.op, "gemm_mode": ops.gemm_mode(-1)}
    if a.op == "gemm":
        A = (torch.randn(a.K, a.M) if a.a_mn else torch.randn(a.M, a.K)).to(bf).to(dev)
        B = (torch.randn(a.K, a.N) if a.b_mn else torch.randn(a.N, a.K)).to(bf).to(dev)
        D = torch.empty(a.M, a.N, dtype=bf, device=dev)
        ms = timeit(lambda: ops.gemm(A, B, a.M, a.N, a.K, a_mn=a.a_mn, b_mn=a.b_mn, D=D), a.iters, a.warmup)
        res.update(shape=[a.M, a.N, a.K], a_mn=a.a_mn, b_mn=a.b_mn, ms=ms, tflops=2 * a.M * a.N * a.K / ms / 1e9)
        ref_ms = timeit(lambda: torch.matmul(A.T if a.a_mn else A, B if a.b_mn else B.T, out=D), a.iters, a.warmup)
        res.update(torch_matmul_ms=ref_ms, torch_matmul_tflops=2 * a.M * a.N * a.K / ref_ms / 1e9)
    elif a.op == "gemm_pair":
        # the 1.2B backward pair of the gate/up projection: dW = dY^T X (both MN-major) and dX = dY W
        T, N, K = a.M, a.N, a.K
        dY = torch.randn(T, N).to(bf).to(dev)
        X = torch.randn(T, K).to(bf).to(dev)
        W = torch.randn(N, K).to(bf).to(dev)
        dW = torch.empty(N, K, dtype=bf, device=dev)
        dX = torch.empty(T, K, dtype=bf, device=dev)
        sw = dict(A=dY, B=X, M=N, N=K, K=T, a_mn=1, b_mn=1, lda=N, ldb=K, D=dW)
        sd = dict(A=dY, B=W, M=T, N=K, K=N, b_mn=1, ldb=K, D=dX)
        fl = 2 * 2 * T * N * K
        ms_pair = timeit(lambda: ops.gemm2([sw, sd]), a.iters, a.warmup)
        ms_w = timeit(lambda: ops.gemm(dY, X, N, K, T, a_mn=True, b_mn=True, lda=N, ldb=K, D=dW), a.iters, a.warmup)
        ms_d = timeit(lambda: ops.gemm(dY, W, T, K, N, b_mn=True, ldb=K, D=dX), a.iters, a.warmup)
        res.update(shape=[T, N, K], pair_ms=ms_pair, pair_tflops=fl / ms_pair / 1e9, wgrad_ms=ms_w, dgrad_ms=ms_d,
                   separate_tflops=fl / (ms_w + ms_d) / 1e9)
    elif a.op in ("attn_fwd", "attn_bwd"):
        T = a.nseq * a.S
        qkv = (torch.randn(T, (a.nh + 2 * a.nkv) * a.hd) * 0.5).to(bf).to(dev)
        o = torch.empty(T, a.nh * a.hd, dtype=bf, device=dev)
        lse = torch.empty(a.nh, T, dtype=torch.float32, device=dev)
        fl = 4.0 * a.nseq * a.nh * a.hd * a.S * a.S / 2
        ops.attention_fwd(qkv, a.nseq, a.S, a.nh, a.nkv, a.hd, o, lse)
        if a.op == "attn_fwd":
            ms = timeit(lambda: ops.attention_fwd(qkv, a.nseq, a.S, a.nh, a.nkv, a.hd, o, lse), a.iters, a.warmup)
        else:
            fl *= 2.5
            do = torch.randn(T, a.nh * a.hd).to(bf).to(dev)
            dq = torch.empty_like(qkv)
            sc = torch.empty(ops.attention_bwd_scratch_bytes(a.nseq, a.S, a.nh, a.hd), dtype=torch.uint8,
                             device=dev)
            ms = timeit(lambda: ops.attention_bwd(qkv, o, lse, do, a.nseq, a.S, a.nh, a.nkv, a.hd, dq, sc),
                        a.iters, a.warmup)
        res.update(shape=dict(S=a.S, nseq=a.nseq, nh=a.nh, nkv=a.nkv, hd=a.hd), ms=ms, tflops=fl / ms / 1e9)
    elif a.op in ("rmsnorm_fwd", "rmsnorm_bwd"):
        x = torch.randn(a.T, a.H).to(bf).to(dev)
        g = torch.ones(a.H, dtype=bf, device=dev)
        y = torch.empty_like(x)
        r = torch.empty(a.T, dtype=torch.float32, device=dev)
        ops.rmsnorm_fwd(x, g, 1e-6, y, r)
        if a.op == "rmsnorm_fwd":
            ms = timeit(lambda: ops.rmsnorm_fwd(x, g, 1e-6, y, r), a.iters, a.warmup)
            by = 4.0 * a.T * a.H
        else:
            dx = torch.empty_like(x)
            dg = torch.empty(a.H, dtype=bf, device=dev)
            sc = torch.empty(ops.rmsnorm_bwd_scratch_bytes(a.T, a.H), dtype=torch.uint8, device=dev)
            ms = timeit(lambda: ops.rmsnorm_bwd(y, x, g, r, y, dx, dg, sc), a.iters, a.warmup)
            by = 8.0 * a.T * a.H
        res.update(shape=[a.T, a.H], ms=ms, gbs=by / ms / 1e6)
    elif a.op == "cross_entropy":
        # --T rows of --V logits, every row with a target; the kernel rewrites the logits in place
        # with dlogits, so each timed launch runs on the previous launch's output (same work)
        V = a.V
        z = torch.randn(a.T, V).to(bf).to(dev)
        tgt = torch.randint(0, V, (a.T,), dtype=torch.int32, device=dev)
        rl = torch.empty(a.T, dtype=torch.float32, device=dev)
        ms = timeit(lambda: ops.cross_entropy(z, tgt, 1.0 / a.T, rl), a.iters, a.warmup)
        by = 4.0 * a.T * V
        res.update(shape=[a.T, V], ms=ms, gbs=by / ms / 1e6)
    elif a.op == "moe_ffn":
        # one MoE feed-forward, forward and backward (router, routing, grouped expert GEMMs, combine);
        # includes one host synchronisation for the per-expert counts
        T, H, E, k, Fe = a.T, a.H, a.E, a.k, a.Fe
        yn = torch.randn(T, H).to(bf).to(dev)
        x1 = torch.randn(T, H).to(bf).to(dev)
        Wr = (torch.randn(E, H) / H ** 0.5).to(bf).to(dev)
        We = torch.cat([torch.randn(E, 2 * Fe * H) / H ** 0.5, torch.randn(E, H * Fe) / Fe ** 0.5], 1).to(bf).to(dev)
        dout = torch.randn(T, H).to(bf).to(dev)
        out, dyn = torch.empty_like(yn), torch.empty_like(yn)
        dWr, dWe = torch.empty_like(Wr), torch.empty_like(We)
        idx = torch.empty(T, k, dtype=torch.int32, device=dev)
        gate = torch.empty(T, k, dtype=torch.float32, device=dev)
        sc = torch.empty(ops.moe_scratch_bytes(T, H, E, k, Fe), dtype=torch.uint8, device=dev)
        run = lambda: ops.moe_ffn(yn, x1, Wr, We, dout, k, Fe, out, dyn, dWr, dWe, idx, gate, sc)
        ms = timeit(run, a.iters, a.warmup)
        fl = 2.0 * T * k * 3 * H * Fe * 3 + 2.0 * T * E * H * 3  # experts fwd + dgrad + wgrad, router x3
        res.update(shape=dict(T=T, H=H, E=E, k=k, Fe=Fe), ms=ms, tflops=fl / ms / 1e9)
    elif a.op == "layer_gemms":
        # the GEMM launches of one decoder layer's forward and backward visits
        # and of the LM head, in the forms and order the runtime issues them:
        # forward qkv, o (+residual), gate/up, down (+residual); the backward's
        # recompute of qkv, o, gate/up; then one launch per projection pairing
        # its weight and input gradients (down, gate/up, o, qkv); the head's
        # logits and its pair.  Each form is timed; launches per step = L per
        # layer form, 1 per head form.
        from . import configs
        c = configs.get(a.config)
        T = c["micro"] * c["batch"] * c["seq"]
        H, F, V = c["hidden"], c["ffn"], c["vocab"]
        nqkv, nhd = (c["n_heads"] + 2 * c["n_kv_heads"]) * c["head_dim"], c["n_heads"] * c["head_dim"]
        r = lambda *sh: (torch.randn(*sh) * 0.05).to(bf).to(dev)
        X = r(T, max(H, nhd, F))
        Wq, Wo, Wgu, Wd = r(nqkv, H), r(H, nhd), r(2 * F, H), r(H, F)
        Yq, Yo, Ygu, Yd = (torch.empty(T, n, dtype=bf, device=dev) for n in (nqkv, H, 2 * F, H))
        dWq, dWo, dWgu, dWd = (torch.empty_like(w) for w in (Wq, Wo, Wgu, Wd))
        dXa = torch.empty(T, max(H, F), dtype=bf, device=dev)

        def fprop(Xin, W, N, K, Y, R=None):
            return lambda: ops.gemm(Xin, W, T, N, K, lda=X.shape[1], D=Y, R=R)

        def pair(dY, Xin, W, N, K, dW):  # dW = dY^T X, dX = dY W
            sw = dict(A=dY, B=Xin, M=N, N=K, K=T, a_mn=1, b_mn=1, lda=N, ldb=Xin.shape[1], D=dW)
            sd = dict(A=dY, B=W, M=T, N=K, K=N, b_mn=1, ldb=K, D=dXa, ldd=dXa.shape[1])
            return lambda: ops.gemm2([sw, sd])

        forms = [("fwd_qkv", fprop(X, Wq, nqkv, H, Yq), 2 * T * nqkv * H, 2),
                 ("fwd_o", fprop(X, Wo, H, nhd, Yo, Yo), 2 * T * H * nhd, 2),
                 ("fwd_gu", fprop(X, Wgu, 2 * F, H, Ygu), 2 * T * 2 * F * H, 2),
                 ("fwd_down", fprop(X, Wd, H, F, Yd, Yd), 2 * T * H * F, 1),
                 ("bwd_down", pair(Yd, X, Wd, H, F, dWd), 4 * T * H * F, 1),
                 ("bwd_gu", pair(Ygu, X, Wgu, 2 * F, H, dWgu), 4 * T * 2 * F * H, 1),
                 ("bwd_o", pair(Yo, X, Wo, H, nhd, dWo), 4 * T * H * nhd, 1),
                 ("bwd_qkv", pair(Yq, X, Wq, nqkv, H, dWq), 4 * T * nqkv * H, 1)]
        if not a.no_head:
            Wh = r(V, H)
            Lg = torch.empty(T, V, dtype=bf, device=dev)
            dWh = torch.empty_like(Wh)
            forms += [("head_fwd", lambda: ops.gemm(X, Wh, T, V, H, lda=X.shape[1], D=Lg), 2 * T * V * H, 0),
                      ("head_pair", pair(Lg, X, Wh, V, H, dWh), 4 * T * V * H, 0)]
        out = {}
        per_layer = c["n_layers"]
        tot_fl = tot_ms = 0.0
        launches = 0
        for name, fn, fl, nl in forms:
            ms = timeit(fn, a.iters, a.warmup)
            cnt = per_layer * nl if nl else 1
            out[name] = {"ms": ms, "tflops": fl / ms / 1e9, "launches_per_step": cnt}
            tot_fl += fl * cnt
            tot_ms += ms * cnt
            launches += cnt
        res.update(config=a.config, T=T, forms=out, step_gemm_ms=tot_ms, step_gemm_tflops=tot_fl / tot_ms / 1e9,
                   launches_per_step=launches)
    else:
        raise SystemExit("unknown op " + a.op)
    print(json.dumps(res))


if __name__ == "__main__":
    main()
