"""CPU tests of libmt's host side against the oracle (no GPU needed).

The library and the oracle are independent implementations; here they must
agree bit-exactly on the flat layout, the seeded initial weights, the event
protocol and the schedule, and to FP32 rounding on host Adam.
"""
import ctypes as C
import os
import re

import numpy as np
import pytest

import host_memory_centric_gb300 as mt
from host_memory_centric_gb300 import configs
from tests import protocol_check

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
F32_002 = float(np.float32(0.02))  # mt_config carries init_std as float


def shape_for_oracle(c):
    return dict(c, init_std=F32_002, rope_base=float(np.float32(c["rope_base"])))


def test_library_exports_every_declared_symbol():
    hdr = open(os.path.join(ROOT, "include", "mt.h")).read()
    names = sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(mt_\w+)\s*\(", hdr, flags=re.M)))
    assert len(names) > 40
    L = mt.lib()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


@pytest.mark.parametrize("name", list(configs.CONFIGS))
def test_layout_bit_exact(orc, name):
    c = configs.get(name)
    assert mt.layout(mt.make_config(c)) == orc.layout(c)
    cfg = mt.make_config(c)
    assert mt.lib().mt_param_count(C.byref(cfg)) == orc.param_count(c)
    assert mt.lib().mt_store_bytes(C.byref(cfg)) == orc.store_bytes(c)


def _lib_init(c, j):
    cfg = mt.make_config(c, seed=77)
    n = mt.layout(cfg)[j]["n_pad"]
    out = np.empty(n, dtype=np.float32)
    assert mt.lib().mt_host_init_block(C.byref(cfg), j, out.ctypes.data_as(C.POINTER(C.c_float))) == 0
    return out


@pytest.mark.parametrize("j", [0, 1, 2, 3])
def test_init_bit_exact_tiny(orc, j):
    c = configs.get("tiny")
    a = _lib_init(c, j)
    b = orc.init_block(shape_for_oracle(c), 77, j)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_init_bit_exact_full_width_decoder_block(orc):
    c = configs.get("1.2b", n_layers=1)
    a = _lib_init(c, 1)
    b = orc.init_block(shape_for_oracle(c), 77, 1)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_host_adam_matches_oracle(orc):
    rng = np.random.default_rng(0)
    n = 300_000
    g = orc.bf16_rne_fast((rng.standard_normal(n) * 1e-3).astype(np.float32))
    th = (0.02 * rng.standard_normal(n)).astype(np.float32)
    m = (1e-4 * rng.standard_normal(n)).astype(np.float32)
    v = (1e-7 * rng.random(n)).astype(np.float32)
    a = [x.copy() for x in (th, m, v)]
    b = [x.copy() for x in (th, m, v)]
    wa = np.empty(n, np.uint16)
    P = lambda x, t: x.ctypes.data_as(C.POINTER(t))
    for t in (1, 2, 7):
        assert mt.lib().mt_host_adam(n, P(g, C.c_uint16), P(a[0], C.c_float), P(a[1], C.c_float),
                                     P(a[2], C.c_float), P(wa, C.c_uint16), t, 1e-3, 0.9, 0.999, 1e-8, 0.0,
                                     4) == 0
        wb = orc.adam(g, b[0], b[1], b[2], t)
    for x, y in zip(a, b):
        assert np.linalg.norm(x - y) <= 1e-6 * np.linalg.norm(y)
    assert np.mean(wa == wb) > 0.999


def test_host_adam_zero_gradient_matches_oracle(orc):
    """The unrouted-expert path (no gradient transferred, g = 0): after a step
    with a gradient, further zero-gradient steps still move the master by
    its momentum, exactly as the oracle's Adam fed zeros."""
    rng = np.random.default_rng(1)
    n = 100_000
    g = orc.bf16_rne_fast((rng.standard_normal(n) * 1e-3).astype(np.float32))
    zero = np.zeros(n, np.uint16)
    th = (0.02 * rng.standard_normal(n)).astype(np.float32)
    a = [th.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)]
    b = [x.copy() for x in a]
    w = np.empty(n, np.uint16)
    P = lambda x, t: x.ctypes.data_as(C.POINTER(t))
    for t, grad in ((1, g), (2, None), (3, None)):
        gp = P(grad, C.c_uint16) if grad is not None else None
        assert mt.lib().mt_host_adam(n, gp, P(a[0], C.c_float), P(a[1], C.c_float), P(a[2], C.c_float),
                                     P(w, C.c_uint16), t, 1e-3, 0.9, 0.999, 1e-8, 0.0, 2) == 0
        wb = orc.adam(grad if grad is not None else zero, b[0], b[1], b[2], t)
    for x, y in zip(a, b):
        assert np.linalg.norm(x - y) <= 1e-6 * np.linalg.norm(y)
    assert np.mean(w == wb) > 0.999
    assert np.linalg.norm(a[0] - th) > 0  # momentum kept moving the weights


def _plan(c, steps, **rt):
    cfg = mt.make_config(c, **rt)
    need = -mt.lib().mt_plan_protocol(C.byref(cfg), steps, None, 0)
    buf = C.create_string_buffer(int(need) + 1)
    n = mt.lib().mt_plan_protocol(C.byref(cfg), steps, buf, need + 1)
    assert n > 0
    return buf.value.decode().splitlines()


@pytest.mark.parametrize("ckpt", [0, 1])
@pytest.mark.parametrize("pin", [0, 1])
@pytest.mark.parametrize("slabs", [1, 3, 12])
def test_protocol_plan_bit_exact(orc, ckpt, pin, slabs):
    c = configs.get("tiny", n_layers=3)
    lines = _plan(c, 3, ckpt_on_host=ckpt, pin_store=pin, n_grad_slabs=slabs)
    assert protocol_check.mask_slabs(lines) == protocol_check.mask_slabs(orc.protocol(c, 3, slabs, bool(ckpt), not pin))
    protocol_check.check(lines)


@pytest.mark.parametrize("ci,nbuf,ckpt", [(2, 2, 1), (3, 1, 0), (5, 2, 0), (1, 1, 1)])
def test_protocol_plan_segments_bit_exact(orc, ci, nbuf, ckpt):
    c = configs.get("tiny", n_layers=5)
    lines = _plan(c, 2, ckpt_on_host=ckpt, pin_store=0, n_grad_slabs=3, ckpt_interval=ci, n_buffers=nbuf)
    ref = orc.protocol(c, 2, 3, bool(ckpt), True, ci, nbuf)
    assert protocol_check.mask_slabs(lines) == protocol_check.mask_slabs(ref)
    protocol_check.check(lines)


@pytest.mark.parametrize("micro,ckpt", [(2, 1), (3, 0)])
def test_protocol_plan_host_accumulation_bit_exact(orc, micro, ckpt):
    c = configs.get("tiny", n_layers=3, micro=micro)
    lines = _plan(c, 2, ckpt_on_host=ckpt, pin_store=0, n_grad_slabs=3, host_grad_accum=1)
    ref = orc.protocol(c, 2, 3, bool(ckpt), True, 1, 2, micro)
    assert protocol_check.mask_slabs(lines) == protocol_check.mask_slabs(ref)
    protocol_check.check(lines)


def test_host_accumulation_shrinks_device_region():
    """With one pass per micro-batch the device holds one micro-batch's
    activations."""
    L = mt.lib()
    c = configs.get("1.2b", micro=4)
    n = {}
    for acc in (0, 1):
        cfg = mt.make_config(c, host_grad_accum=acc)
        b = C.c_size_t()
        assert L.mt_query_device_bytes(C.byref(cfg), C.byref(b)) == 0
        n[acc] = b.value
    assert n[1] < 0.5 * n[0]


@pytest.mark.parametrize("L,ci", [(2, 1), (5, 2), (7, 3), (4, 4)])
def test_visit_plan_matches_oracle(orc, L, ci):
    c = configs.get("tiny", n_layers=L)
    plan = mt.visit_plan(mt.make_config(c, ckpt_interval=ci))
    names = {"FWD": 0, "HEAD": 1, "RECOMP": 2, "BWD": 3}
    ref = [(names[l.split()[2]], int(l.split()[3])) for l in orc.protocol(c, 1, 12, True, False, ci, 2)
           if l.split()[2] in names]
    assert plan == ref


def test_device_checkpoints_scale_with_segments():
    """Device-resident checkpoints: one slot per segment plus c - 1 recompute
    slots, so a larger interval needs less device memory."""
    L = mt.lib()
    c = configs.get("1.2b")
    act = c["batch"] * c["seq"] * c["hidden"] * 2
    size = {}
    for ci in (1, 2, 5):
        cfg = mt.make_config(c, ckpt_on_host=0, ckpt_interval=ci)
        n = C.c_size_t()
        assert L.mt_query_device_bytes(C.byref(cfg), C.byref(n)) == 0
        size[ci] = n.value
    nl = c["n_layers"]
    assert size[1] - size[2] == pytest.approx((nl - (-(-nl // 2)) - 1) * act, abs=4096 * nl)
    assert size[5] < size[2] < size[1]  # slots: 22, 12, 5 + 4


@pytest.mark.parametrize("name", ["1.2b", "7.6b", "14.7b"])
def test_protocol_plan_full_depth(orc, name):
    c = configs.get(name)
    assert protocol_check.mask_slabs(_plan(c, 2)) == protocol_check.mask_slabs(orc.protocol(c, 2, 12, True, True))


def test_schedule_matches_oracle(orc):
    rng = np.random.default_rng(3)
    for _ in range(20):
        n = int(rng.integers(3, 60))
        b, d, cc, a = (rng.random(n) * s for s in (1e9, 1e9, 0.02, 0.05))
        d[rng.random(n) < 0.5] = 0.0
        st_o, k_o = orc.schedule(b, d, cc, a, 2e11, 1.9e11)
        st_l = np.empty(n)
        P = lambda x: np.ascontiguousarray(x, np.float64).ctypes.data_as(C.POINTER(C.c_double))
        k_l = mt.lib().mt_schedule(n, P(b), P(d), P(cc), P(a), 2e11, 1.9e11, P(st_l))
        assert k_l == k_o
        assert np.allclose(st_l, st_o, rtol=1e-12, atol=1e-15)


def test_token_csr():
    rng = np.random.default_rng(4)
    tok = rng.integers(0, 50, 1000).astype(np.int32)
    rs, rows = mt.ops.token_csr(tok, 50)
    assert rs[0] == 0 and rs[-1] == tok.size
    for v in range(50):
        assert list(rows[rs[v]:rs[v + 1]]) == list(np.nonzero(tok == v)[0])


def test_rope_table():
    t = mt.ops.rope_table(37, 16, 1e4).reshape(37, 8, 2)
    p = np.arange(37)[:, None]
    ang = p * 1e4 ** (-2 * np.arange(8) / 16.0)
    assert np.allclose(t[..., 0], np.cos(ang), atol=1e-7) and np.allclose(t[..., 1], np.sin(ang), atol=1e-7)


def test_bad_arguments_rejected_without_gpu():
    L = mt.lib()
    cfg = mt.make_config(configs.get("tiny"))
    nbytes = C.c_size_t()
    assert L.mt_query_device_bytes(C.byref(cfg), C.byref(nbytes)) == 0 and nbytes.value > 0
    bad = mt.make_config(configs.get("tiny"), n_kv_heads=3)
    assert L.mt_query_device_bytes(C.byref(bad), C.byref(nbytes)) == -1
    for kw in (dict(ckpt_interval=0), dict(ckpt_interval=3), dict(n_buffers=0), dict(n_buffers=3),
               dict(host_grad_accum=2)):
        bad = mt.make_config(configs.get("tiny"), **kw)  # tiny has 2 layers
        assert L.mt_query_device_bytes(C.byref(bad), C.byref(nbytes)) == -1, kw
    ok = mt.make_config(configs.get("tiny"), ckpt_interval=2, n_buffers=1)
    assert L.mt_query_device_bytes(C.byref(ok), C.byref(nbytes)) == 0
    h = C.c_void_p()
    assert L.mt_init_model(C.byref(cfg), mt.DevRegion(None, 0), mt.Streams(None, None, None), C.byref(h)) == -1
    assert L.mt_train_step(None, 0, None) == -1


def test_empty_inputs_launch_nothing_and_succeed():
    """Zero rows (T = 0, rows = 0, V = 0) are no-ops: the device calls return
    MT_OK before any CUDA call, so they succeed here without a GPU (pointers
    must still be non-null)."""
    L = mt.lib()
    buf = np.zeros(4096, np.float32)
    p = buf.ctypes.data_as(C.c_void_p)
    H = 256
    sc = L.mt_rmsnorm_bwd_scratch_bytes(0, H)
    assert sc >= H * 4  # one partial row even for no rows
    assert L.mt_rmsnorm_fwd(p, p, 0, H, 1e-6, p, p, None) == 0
    assert L.mt_rmsnorm_bwd(p, p, p, p, None, 0, H, p, p, p, sc, None) == 0
    assert L.mt_rope(p, 0, 512, 4, 64, 16, p, 0, None) == 0
    assert L.mt_swiglu_fwd(p, 0, 64, p, None) == 0
    assert L.mt_swiglu_bwd(p, p, 0, 64, p, None) == 0
    assert L.mt_embed_fwd(p, p, 0, H, 100, p, None) == 0
    assert L.mt_embed_bwd(p, p, p, 0, H, p, None) == 0
    assert L.mt_cross_entropy(p, p, 0, 1000, 1.0, p, None) == 0
    # null pointers are still rejected, empty or not
    assert L.mt_rmsnorm_fwd(None, p, 0, H, 1e-6, p, p, None) == -1
    assert L.mt_cross_entropy(p, None, 0, 1000, 1.0, p, None) == -1


def test_device_footprint_independent_of_depth():
    """With host checkpoints the carved device region does not grow with depth."""
    L = mt.lib()
    sizes = []
    for depth in (12, 24, 48):
        cfg = mt.make_config(configs.get("14.7b", n_layers=depth))
        n = C.c_size_t()
        assert L.mt_query_device_bytes(C.byref(cfg), C.byref(n)) == 0
        sizes.append(n.value)
    assert sizes[0] == sizes[1] == sizes[2]
    dev = []
    for depth in (12, 24):
        cfg = mt.make_config(configs.get("14.7b", n_layers=depth), ckpt_on_host=0)
        n = C.c_size_t()
        L.mt_query_device_bytes(C.byref(cfg), C.byref(n))
        dev.append(n.value)
    assert dev[1] > dev[0]


def test_worker_pool_has_no_data_race(tmp_path):
    """The host worker pool under ThreadSanitizer: concurrent parallel_for
    calls from two threads must report no data race (a worker that touched a
    caller's completion latch after the caller returned once crashed the
    library intermittently)."""
    import shutil
    import subprocess
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no g++")
    here = os.path.dirname(os.path.abspath(__file__))
    src = os.path.join(os.path.dirname(here), "host_memory_centric_gb300", "csrc")
    inc = os.path.join(os.path.dirname(here), "include")
    exe = str(tmp_path / "pool_stress")
    cmd = [cxx, "-std=c++17", "-O1", "-g", "-fsanitize=thread", "-I" + src, "-I" + inc,
           "-I" + os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include"),
           os.path.join(here, "pool_stress.cpp"), os.path.join(src, "mt_host.cpp"), "-o", exe, "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("ThreadSanitizer build unavailable: " + r.stderr[-200:])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, TSAN_OPTIONS="halt_on_error=1 exitcode=66"))
    assert "ThreadSanitizer" not in r.stderr, r.stderr[-2000:]
    assert r.returncode == 0 and r.stdout.startswith("ok"), (r.returncode, r.stdout, r.stderr[-500:])


# ------------------------------------------------------------------ routed MoE
def test_init_bit_exact_moe_block(orc):
    c = configs.get("tiny_moe")
    for j in (1, 2):
        a = _lib_init(c, j)
        b = orc.init_block(shape_for_oracle(c), 77, j)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("pin,ckpt,ci,nbuf", [(0, 1, 1, 2), (1, 1, 1, 2), (0, 0, 2, 2), (1, 0, 1, 1), (0, 1, 3, 1)])
def test_protocol_plan_moe_bit_exact(orc, pin, ckpt, ci, nbuf):
    """MoE forward visits: Route-Ready, the host's wait, the routed experts'
    copy and Experts-Ready sit where the simulator puts them."""
    c = configs.get("tiny_moe", n_layers=3)
    lines = _plan(c, 3, ckpt_on_host=ckpt, pin_store=pin, n_grad_slabs=2, ckpt_interval=ci, n_buffers=nbuf)
    ref = orc.protocol(c, 3, 2, bool(ckpt), not pin, ci, nbuf)
    assert protocol_check.mask_slabs(lines) == protocol_check.mask_slabs(ref)
    protocol_check.check(lines)
    assert sum(" H2D_EXP " in l for l in lines) == 3 * 3


def test_bad_moe_configs_rejected():
    L = mt.lib()
    n = C.c_size_t()
    for kw in (dict(n_experts=12), dict(n_experts=136), dict(top_k=0), dict(top_k=9), dict(expert_ffn=100),
               dict(hidden=320, n_heads=5), dict(host_grad_accum=1)):
        bad = mt.make_config(configs.get("tiny_moe", **{k: v for k, v in kw.items() if k != "host_grad_accum"}),
                             **({"host_grad_accum": 1} if "host_grad_accum" in kw else {}))
        assert L.mt_query_device_bytes(C.byref(bad), C.byref(n)) == -1, kw
    ok = mt.make_config(configs.get("tiny_moe"))
    assert L.mt_query_device_bytes(C.byref(ok), C.byref(n)) == 0
    assert L.mt_moe_scratch_bytes(256, 256, 8, 2, 256) > 0


def test_gemm_mode_switch_is_host_state():
    """mt_gemm_mode only reads and sets the process's dense-GEMM tiling (no
    device call): it returns the mode in force before the call, takes 0-3 and
    ignores anything else."""
    L = mt.lib()
    L.mt_gemm_mode.restype = C.c_int32
    L.mt_gemm_mode.argtypes = [C.c_int32]
    prev = L.mt_gemm_mode(-1)
    assert prev in (0, 1, 2, 3)
    try:
        for m in (0, 1, 2, 3):
            L.mt_gemm_mode(m)
            assert L.mt_gemm_mode(-1) == m
        assert L.mt_gemm_mode(4) == 3  # out of range: nothing changes
        assert L.mt_gemm_mode(-7) == 3
        assert L.mt_gemm_mode(1) == 3
    finally:
        L.mt_gemm_mode(prev)
