"""ctypes wrapper of the reference oracle (TEST INFRASTRUCTURE ONLY).

The oracle (``oracle.cpp``) is a plain, slow CPU statement of one step of the
layer-streamed training method; see its header for what it computes and which
page sections each part follows.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  It shares
no code with the GPU library and never imports it.

Functions here only marshal arguments: every number is computed in C++.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile liboracle.so with the host C++ compiler (no CUDA involved)."""
    src = os.path.join(_HERE, "oracle.cpp")
    hdr = os.path.join(_HERE, "oracle.h")
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= max(os.path.getmtime(src), os.path.getmtime(hdr))):
        return _SO
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-fopenmp-simd",
           "-o", _SO + ".tmp", src]
    subprocess.run(cmd, check=True)
    os.replace(_SO + ".tmp", _SO)
    return _SO


class Cfg(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("hidden", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn", C.c_int32),
                ("vocab", C.c_int32), ("batch", C.c_int32), ("seq", C.c_int32),
                ("micro", C.c_int32), ("rope_base", C.c_double), ("rms_eps", C.c_double),
                ("init_std", C.c_double), ("n_experts", C.c_int32), ("top_k", C.c_int32),
                ("expert_ffn", C.c_int32)]


def make_cfg(shape: dict) -> Cfg:
    return Cfg(shape["n_layers"], shape["hidden"], shape["n_heads"], shape["n_kv_heads"],
               shape["head_dim"], shape["ffn"], shape["vocab"], shape["batch"], shape["seq"],
               shape["micro"], shape.get("rope_base", 10000.0), shape.get("rms_eps", 1e-6),
               shape.get("init_std", 0.02), shape.get("n_experts", 0), shape.get("top_k", 0),
               shape.get("expert_ffn", 0))


_lib = None
_P = C.POINTER


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_SO)
        d, f, i64, i32, u64, u16 = C.c_double, C.c_float, C.c_int64, C.c_int32, C.c_uint64, C.c_uint16
        pc = _P(Cfg)
        sig = {
            "or_n_blocks": (i64, [pc]),
            "or_layout_block": (i64, [pc, i32, _P(i64), i64]),
            "or_param_count": (i64, [pc]),
            "or_store_bytes": (i64, [pc]),
            "or_splitmix64": (u64, [u64, u64]),
            "or_normal": (d, [u64, u64]),
            "or_init_block": (i32, [pc, u64, i32, _P(f)]),
            "or_bf16_rne": (u16, [f]),
            "or_bf16_to_f32": (f, [u16]),
            "or_rmsnorm_fwd_d": (None, [_P(d), _P(d), i64, i64, d, _P(d), _P(d)]),
            "or_rmsnorm_bwd_d": (None, [_P(d), _P(d), _P(d), _P(d), i64, i64, _P(d), _P(d)]),
            "or_linear_fwd_d": (None, [_P(d), _P(d), i64, i64, i64, _P(d)]),
            "or_linear_dgrad_d": (None, [_P(d), _P(d), i64, i64, i64, _P(d)]),
            "or_linear_wgrad_d": (None, [_P(d), _P(d), i64, i64, i64, _P(d)]),
            "or_rope_d": (None, [_P(d), i64, i64, i64, i64, i64, d, i32]),
            "or_attention_fwd_d": (None, [_P(d), i64, i64, i64, i64, i64, _P(d), _P(d)]),
            "or_attention_bwd_d": (None, [_P(d), _P(d), _P(d), _P(d), i64, i64, i64, i64, i64, _P(d)]),
            "or_swiglu_fwd_d": (None, [_P(d), i64, i64, _P(d)]),
            "or_swiglu_bwd_d": (None, [_P(d), _P(d), i64, i64, _P(d)]),
            "or_cross_entropy_d": (d, [_P(d), _P(i32), i64, i64, i64, d, _P(d)]),
            "or_step_fwd_bwd_f": (d, [pc, _P(_P(f)), _P(i32), _P(_P(f))]),
            "or_step_fwd_bwd_d": (d, [pc, _P(_P(d)), _P(i32), _P(_P(d))]),
            "or_forward_hidden_f": (d, [pc, _P(_P(f)), _P(i32), i32, _P(f)]),
            "or_adam": (None, [i64, _P(u16), _P(f), _P(f), _P(f), _P(u16), i32, f, f, f, f, f]),
            "or_protocol": (i64, [pc, i32, i32, i32, i32, i32, i32, i32, C.c_char_p, i64]),
            "or_adam_f32": (None, [i64, _P(f), _P(u16), _P(f), _P(f), _P(f), _P(u16), i32, f, f, f, f, f]),
            "or_schedule": (i32, [i32, _P(d), _P(d), _P(d), _P(d), d, d, _P(d)]),
            "or_last_route_margin": (d, []),
            "or_moe_layer_d": (d, [i64, i64, i64, i64, i64] + [_P(d)] * 9 + [_P(i32), _P(d)]),
            "or_moe_layer_f": (d, [i64, i64, i64, i64, i64] + [_P(f)] * 9 + [_P(i32), _P(f)]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(a: np.ndarray, ct):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(_P(ct))


def _d(a):
    return _ptr(a, C.c_double)


# ---------------------------------------------------------------- layout / init
def layout(shape: dict) -> list[dict]:
    """Per block: tensors (elem offset, rows, cols), region offsets, sizes."""
    c = make_cfg(shape)
    out = []
    for j in range(lib().or_n_blocks(C.byref(c))):
        buf = np.zeros(64, dtype=np.int64)
        n = lib().or_layout_block(C.byref(c), j, _ptr(buf, C.c_int64), 64)
        assert n > 0
        nt = int(buf[0])
        out.append(dict(
            n_tensors=nt, n_real=int(buf[1]), n_pad=int(buf[2]),
            off_W=int(buf[3]), off_G=int(buf[4]), off_master=int(buf[5]), off_m=int(buf[6]),
            off_v=int(buf[7]), bytes=int(buf[8]), store_off=int(buf[9]),
            tensors=[(int(buf[10 + 3 * t]), int(buf[11 + 3 * t]), int(buf[12 + 3 * t]))
                     for t in range(nt)]))
    return out


def param_count(shape: dict) -> int:
    return int(lib().or_param_count(C.byref(make_cfg(shape))))


def store_bytes(shape: dict) -> int:
    return int(lib().or_store_bytes(C.byref(make_cfg(shape))))


def splitmix64(seed: int, i: int) -> int:
    return int(lib().or_splitmix64(seed, i))


def normal(key: int, e: int) -> float:
    return float(lib().or_normal(key, e))


def init_block(shape: dict, seed: int, j: int) -> np.ndarray:
    lay = layout(shape)[j]
    out = np.empty(lay["n_pad"], dtype=np.float32)
    assert lib().or_init_block(C.byref(make_cfg(shape)), seed, j, _ptr(out, C.c_float)) == 0
    return out


def bf16_rne(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    fn = lib().or_bf16_rne
    return np.array([fn(float(v)) for v in x], dtype=np.uint16)


def bf16_rne_fast(x: np.ndarray) -> np.ndarray:
    """Vectorised restatement used only to build large oracle inputs; the
    scalar C++ routine above is the definition and a test checks they agree."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = ((u & 0x7F800000) == 0x7F800000) & ((u & 0x007FFFFF) != 0)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r.reshape(np.shape(x))


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- per-op (fp64)
def rmsnorm_fwd(x, g, eps=1e-6):
    x = np.ascontiguousarray(x, np.float64); g = np.ascontiguousarray(g, np.float64)
    T, H = x.shape
    y = np.empty_like(x); r = np.empty(T)
    lib().or_rmsnorm_fwd_d(_d(x), _d(g), T, H, eps, _d(y), _d(r))
    return y, r


def rmsnorm_bwd(dy, x, g, rstd):
    dy, x, g, rstd = (np.ascontiguousarray(a, np.float64) for a in (dy, x, g, rstd))
    T, H = x.shape
    dx = np.empty_like(x); dg = np.zeros(H)
    lib().or_rmsnorm_bwd_d(_d(dy), _d(x), _d(g), _d(rstd), T, H, _d(dx), _d(dg))
    return dx, dg


def linear_fwd(X, W):
    X = np.ascontiguousarray(X, np.float64); W = np.ascontiguousarray(W, np.float64)
    T, K = X.shape; N = W.shape[0]
    Y = np.empty((T, N))
    lib().or_linear_fwd_d(_d(X), _d(W), T, N, K, _d(Y))
    return Y


def linear_dgrad(dY, W):
    dY = np.ascontiguousarray(dY, np.float64); W = np.ascontiguousarray(W, np.float64)
    T, N = dY.shape; K = W.shape[1]
    dX = np.empty((T, K))
    lib().or_linear_dgrad_d(_d(dY), _d(W), T, N, K, _d(dX))
    return dX


def linear_wgrad(dY, X):
    dY = np.ascontiguousarray(dY, np.float64); X = np.ascontiguousarray(X, np.float64)
    T, N = dY.shape; K = X.shape[1]
    dW = np.empty((N, K))
    lib().or_linear_wgrad_d(_d(dY), _d(X), T, N, K, _d(dW))
    return dW


def rope(x, n_seq, S, n_heads, hd, base, inverse=False):
    x = np.array(x, np.float64, order="C", copy=True)
    lib().or_rope_d(_d(x), n_seq, S, x.shape[1], n_heads, hd, base, int(inverse))
    return x


def attention_fwd(qkv, n_seq, S, nh, nkv, hd):
    qkv = np.ascontiguousarray(qkv, np.float64)
    T = n_seq * S
    o = np.empty((T, nh * hd)); lse = np.empty((T, nh))
    lib().or_attention_fwd_d(_d(qkv), n_seq, S, nh, nkv, hd, _d(o), _d(lse))
    return o, lse


def attention_bwd(qkv, o, lse, dout, n_seq, S, nh, nkv, hd):
    qkv, o, lse, dout = (np.ascontiguousarray(a, np.float64) for a in (qkv, o, lse, dout))
    dqkv = np.empty_like(qkv)
    lib().or_attention_bwd_d(_d(qkv), _d(o), _d(lse), _d(dout), n_seq, S, nh, nkv, hd, _d(dqkv))
    return dqkv


def swiglu_fwd(gu):
    gu = np.ascontiguousarray(gu, np.float64)
    T, F2 = gu.shape
    h = np.empty((T, F2 // 2))
    lib().or_swiglu_fwd_d(_d(gu), T, F2 // 2, _d(h))
    return h


def swiglu_bwd(gu, dh):
    gu = np.ascontiguousarray(gu, np.float64); dh = np.ascontiguousarray(dh, np.float64)
    T, F2 = gu.shape
    dgu = np.empty_like(gu)
    lib().or_swiglu_bwd_d(_d(gu), _d(dh), T, F2 // 2, _d(dgu))
    return dgu


def cross_entropy(logits, tok, n_seq, S, norm):
    logits = np.ascontiguousarray(logits, np.float64)
    tok = np.ascontiguousarray(tok, np.int32)
    V = logits.shape[1]
    dl = np.empty_like(logits)
    loss = lib().or_cross_entropy_d(_d(logits), _ptr(tok, C.c_int32), n_seq, S, V, norm, _d(dl))
    return loss, dl


def moe_layer(yn, x1, Wr, We, dout, k, Fe, dtype=np.float64):
    """The MoE feed-forward of one layer and its backward (see or_moe_layer_d).
    Returns out, dyn, dWr, dWe, idx [T, k], gate [T, k], smallest margin."""
    ct = C.c_double if dtype == np.float64 else C.c_float
    yn, x1, Wr, We, dout = (np.ascontiguousarray(a, dtype) for a in (yn, x1, Wr, We, dout))
    T, H = yn.shape
    E = Wr.shape[0]
    out = np.empty((T, H), dtype); dyn = np.empty((T, H), dtype)
    dWr = np.empty_like(Wr); dWe = np.empty_like(We)
    idx = np.empty((T, k), np.int32); gate = np.empty((T, k), dtype)
    fn = lib().or_moe_layer_d if dtype == np.float64 else lib().or_moe_layer_f
    p = lambda a: _ptr(a, ct)
    mg = fn(T, H, E, k, Fe, p(yn), p(x1), p(Wr), p(We), p(dout), p(out), p(dyn), p(dWr), p(dWe),
            _ptr(idx, C.c_int32), p(gate))
    return out, dyn, dWr, dWe, idx, gate, float(mg)


def last_route_margin() -> float:
    """Smallest routing margin of the last whole-step / forward call."""
    return float(lib().or_last_route_margin())


# ---------------------------------------------------------------- whole step
def step_fwd_bwd(shape: dict, W: list, tok: np.ndarray, dtype=np.float32):
    """Loss and per-block gradients (layout order) from per-block weights."""
    c = make_cfg(shape)
    ct = C.c_float if dtype == np.float32 else C.c_double
    W = [np.ascontiguousarray(w, dtype=dtype) for w in W]
    lay = layout(shape)
    G = [np.zeros(b["n_pad"], dtype=dtype) for b in lay]
    Wp = (_P(ct) * len(W))(*[_ptr(w, ct) for w in W])
    Gp = (_P(ct) * len(G))(*[_ptr(g, ct) for g in G])
    tok = np.ascontiguousarray(tok, dtype=np.int32)
    fn = lib().or_step_fwd_bwd_f if dtype == np.float32 else lib().or_step_fwd_bwd_d
    loss = fn(C.byref(c), Wp, _ptr(tok, C.c_int32), Gp)
    return float(loss), G


def forward_hidden(shape: dict, W: list, tok: np.ndarray, j: int) -> np.ndarray:
    c = make_cfg(shape)
    W = [np.ascontiguousarray(w, dtype=np.float32) for w in W]
    Wp = (_P(C.c_float) * len(W))(*[_ptr(w, C.c_float) for w in W])
    tok = np.ascontiguousarray(tok, dtype=np.int32)
    T = shape["micro"] * shape["batch"] * shape["seq"]
    out = np.empty((T, shape["hidden"]), dtype=np.float32)
    lib().or_forward_hidden_f(C.byref(c), Wp, _ptr(tok, C.c_int32), j, _ptr(out, C.c_float))
    return out


def adam(g_bf16, master, m, v, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0):
    """In-place Adam on (master, m, v); returns the new BF16 weights."""
    g = np.ascontiguousarray(g_bf16, np.uint16)
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    w = np.empty(g.size, dtype=np.uint16)
    lib().or_adam(g.size, _ptr(g, C.c_uint16), _ptr(master, C.c_float), _ptr(m, C.c_float),
                  _ptr(v, C.c_float), _ptr(w, C.c_uint16), step, lr, beta1, beta2, eps, wd)
    return w


def adam_f32(g32, master, m, v, step, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0):
    """In-place Adam on (master, m, v) with an FP32 gradient; returns the new BF16 weights."""
    g = np.ascontiguousarray(g32, np.float32)
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    w = np.empty(g.size, dtype=np.uint16)
    lib().or_adam_f32(g.size, _ptr(g, C.c_float), None, _ptr(master, C.c_float), _ptr(m, C.c_float),
                      _ptr(v, C.c_float), _ptr(w, C.c_uint16), step, lr, beta1, beta2, eps, wd)
    return w


def protocol(shape: dict, n_steps: int, n_slabs: int, ckpt_on_host: bool, jit_pack: bool,
             ckpt_interval: int = 1, n_buffers: int = 2, n_passes: int = 1) -> list[str]:
    c = make_cfg(shape)
    args = (n_steps, n_slabs, int(ckpt_on_host), int(jit_pack), int(ckpt_interval), int(n_buffers), int(n_passes))
    need = -lib().or_protocol(C.byref(c), *args, None, 0)
    assert need > 0, "invalid protocol arguments"
    buf = C.create_string_buffer(int(need) + 1)
    n = lib().or_protocol(C.byref(c), *args, buf, need + 1)
    assert n >= 0
    return buf.value.decode().splitlines()


def schedule(b, d, c, a, bw_h2d, bw_d2h):
    b, d, c, a = (np.ascontiguousarray(x, np.float64) for x in (b, d, c, a))
    stall = np.empty(len(b))
    k = lib().or_schedule(len(b), _d(b), _d(d), _d(c), _d(a), bw_h2d, bw_d2h, _d(stall))
    return stall, int(k)
