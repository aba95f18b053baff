"""Per-op device entry points of libmt on torch tensors (marshalling only).

Each function passes device pointers and the current torch stream to the
matching ``mt_*`` call of ``include/mt.h``; all arithmetic runs in the
library's sm_103a kernels.
"""
from __future__ import annotations

import ctypes as C

import numpy as np


def _L():
    from . import lib
    return lib()


def _chk(s):
    from . import MtError
    if s != 0:
        raise MtError(s, "device op failed")


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def _p(t):
    return None if t is None else t.data_ptr()


def gemm(A, B, M, N, K, *, a_mn=False, b_mn=False, lda=None, ldb=None, D=None, ldd=None, R=None, ldr=None,
         Dacc=None, ldacc=None, acc_mode=0):
    lda = lda if lda is not None else (M if a_mn else K)
    ldb = ldb if ldb is not None else (N if b_mn else K)
    ldd = ldd if ldd is not None else N
    ldr = ldr if ldr is not None else N
    ldacc = ldacc if ldacc is not None else N
    _chk(_L().mt_gemm(_p(A), lda, int(a_mn), _p(B), ldb, int(b_mn), M, N, K, _p(D), ldd, _p(R), ldr,
                      _p(Dacc), ldacc, acc_mode, _stream()))


def gemm_mode(mode=-1) -> int:
    """Dense GEMM tiling: 0 one CTA per 128 x 256 tile; 1 CTA pairs per
    256 x 256 tile (256 x 512 when every GEMM of the launch has K >= 8192 and
    N >= 512) drawing tiles from a counter, 2 the same taking every n-th
    tile, 3 as 1 without the 512-wide tiles; -1 only reads.  Returns the
    previous mode."""
    return int(_L().mt_gemm_mode(int(mode)))


def gemm2(specs):
    """Two GEMMs in one launch; specs = two dicts with A, B, M, N, K, D and
    optional a_mn, b_mn, lda, ldb, ldd (defaults as in gemm)."""
    arr = lambda ct, vals: (ct * 2)(*vals)
    A, B, D, lda, ldb, ldd, amn, bmn, M, N, K = ([] for _ in range(11))
    for s in specs:
        a_mn, b_mn = int(s.get("a_mn", 0)), int(s.get("b_mn", 0))
        A.append(s["A"].data_ptr()); B.append(s["B"].data_ptr()); D.append(s["D"].data_ptr())
        M.append(s["M"]); N.append(s["N"]); K.append(s["K"]); amn.append(a_mn); bmn.append(b_mn)
        lda.append(s.get("lda", s["M"] if a_mn else s["K"])); ldb.append(s.get("ldb", s["N"] if b_mn else s["K"]))
        ldd.append(s.get("ldd", s["N"]))
    _chk(_L().mt_gemm2(arr(C.c_void_p, A), arr(C.c_int64, lda), arr(C.c_int32, amn), arr(C.c_void_p, B),
                       arr(C.c_int64, ldb), arr(C.c_int32, bmn), arr(C.c_int32, M), arr(C.c_int32, N),
                       arr(C.c_int32, K), arr(C.c_void_p, D), arr(C.c_int64, ldd), _stream()))


def rmsnorm_fwd(x, gamma, eps, y, rstd):
    T, H = x.shape
    _chk(_L().mt_rmsnorm_fwd(_p(x), _p(gamma), T, H, eps, _p(y), _p(rstd), _stream()))


def rmsnorm_bwd_scratch_bytes(T, H):
    return int(_L().mt_rmsnorm_bwd_scratch_bytes(T, H))


def rmsnorm_bwd(dy, x, gamma, rstd, dres, dx, dgamma, scratch):
    T, H = x.shape
    _chk(_L().mt_rmsnorm_bwd(_p(dy), _p(x), _p(gamma), _p(rstd), _p(dres), T, H, _p(dx), _p(dgamma),
                             _p(scratch), scratch.numel() * scratch.element_size(), _stream()))


def rope_table(S, hd, base) -> np.ndarray:
    out = np.empty(S * hd, dtype=np.float32)
    _chk(_L().mt_rope_table(S, hd, base, out.ctypes.data_as(C.POINTER(C.c_float))))
    return out


def rope(x, n_heads, hd, S, cs, inverse=False):
    T, ld = x.shape
    _chk(_L().mt_rope(_p(x), T, ld, n_heads, hd, S, _p(cs), int(inverse), _stream()))


def attention_fwd(qkv, n_seq, S, nh, nkv, hd, o, lse):
    _chk(_L().mt_attention_fwd(_p(qkv), n_seq, S, nh, nkv, hd, _p(o), _p(lse), _stream()))


def attention_bwd_scratch_bytes(n_seq, S, nh, hd):
    return int(_L().mt_attention_bwd_scratch_bytes(n_seq, S, nh, hd))


def attention_bwd(qkv, o, lse, dout, n_seq, S, nh, nkv, hd, dqkv, scratch):
    _chk(_L().mt_attention_bwd(_p(qkv), _p(o), _p(lse), _p(dout), n_seq, S, nh, nkv, hd, _p(dqkv), _p(scratch),
                               scratch.numel() * scratch.element_size(), _stream()))


def swiglu_fwd(gu, h):
    T, F2 = gu.shape
    _chk(_L().mt_swiglu_fwd(_p(gu), T, F2 // 2, _p(h), _stream()))


def swiglu_bwd(gu, dh, dgu):
    T, F2 = gu.shape
    _chk(_L().mt_swiglu_bwd(_p(gu), _p(dh), T, F2 // 2, _p(dgu), _stream()))


def embed_fwd(tok, E, X):
    V, H = E.shape
    _chk(_L().mt_embed_fwd(_p(tok), _p(E), tok.numel(), H, V, _p(X), _stream()))


def token_csr(tok: np.ndarray, V: int):
    tok = np.ascontiguousarray(tok, dtype=np.int32).ravel()
    rs = np.empty(V + 1, dtype=np.int32)
    rows = np.empty(tok.size, dtype=np.int32)
    P = C.POINTER(C.c_int32)
    _chk(_L().mt_token_csr(tok.ctypes.data_as(P), tok.size, V, rs.ctypes.data_as(P), rows.ctypes.data_as(P)))
    return rs, rows


def embed_bwd(row_start, rows, dX, V, dE):
    H = dX.shape[1]
    _chk(_L().mt_embed_bwd(_p(row_start), _p(rows), _p(dX), V, H, _p(dE), _stream()))


def cross_entropy(logits, target, inv_norm, row_loss):
    rows, V = logits.shape
    _chk(_L().mt_cross_entropy(_p(logits), _p(target), rows, V, inv_norm, _p(row_loss), _stream()))


def moe_scratch_bytes(T, H, E, k, Fe):
    return int(_L().mt_moe_scratch_bytes(T, H, E, k, Fe))


def moe_ffn(yn, x1, Wr, We, dout, k, Fe, out, dyn, dWr, dWe, idx, gate, scratch):
    """Routed MoE feed-forward forward + backward (mt_moe_ffn)."""
    T, H = yn.shape
    E = Wr.shape[0]
    _chk(_L().mt_moe_ffn(_p(yn), _p(x1), _p(Wr), _p(We), _p(dout), T, H, E, k, Fe, _p(out), _p(dyn), _p(dWr),
                         _p(dWe), _p(idx), _p(gate), _p(scratch), scratch.numel() * scratch.element_size(),
                         _stream()))


def kernel_error(clear=True) -> int:
    c = C.c_int32()
    _chk(_L().mt_kernel_error(C.byref(c), int(clear)))
    return int(c.value)
