"""Layer-streamed, host-memory-centric training step on one GB300 (sm_103a).

Thin ctypes binding of ``libmt.so`` (C ABI in ``include/mt.h``): argument
marshalling only.  Every step of the training path runs in the library's
native code and CUDA kernels; PyTorch is used here only to allocate the device
region and the three CUDA streams.  Importing works without a GPU; the model
and the device ops need one and raise if the native library cannot be built
or loaded.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import configs  # noqa: F401
from .build import OUT as _SO_PATH
from .build import build as _build

__all__ = ["lib", "Model", "make_config", "MtConfig", "ops", "REGION_W", "REGION_G",
           "REGION_MASTER", "REGION_M", "REGION_V"]

REGION_W, REGION_G, REGION_MASTER, REGION_M, REGION_V, REGION_GACC = range(6)
STATUS = {0: "MT_OK", -1: "MT_ERR_ARG", -2: "MT_ERR_STATE", -3: "MT_ERR_HOST_OOM", -4: "MT_ERR_CUDA",
          -5: "MT_ERR_TIMEOUT", -6: "MT_ERR_INTERNAL", -7: "MT_ERR_DEVICE_OOM"}
MAX_TENSORS = 8


class MtError(RuntimeError):
    def __init__(self, status: int, msg: str = ""):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class MtConfig(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("hidden", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn", C.c_int32),
                ("vocab", C.c_int32), ("rope_base", C.c_float), ("rms_eps", C.c_float),
                ("init_std", C.c_float), ("batch", C.c_int32), ("seq", C.c_int32),
                ("micro_batches", C.c_int32), ("ckpt_interval", C.c_int32),
                ("ckpt_on_host", C.c_int32), ("n_grad_slabs", C.c_int32),
                ("n_host_threads", C.c_int32), ("lr", C.c_float), ("beta1", C.c_float),
                ("beta2", C.c_float), ("adam_eps", C.c_float), ("weight_decay", C.c_float),
                ("seed", C.c_uint64), ("timeout_ms", C.c_uint32), ("pin_store", C.c_int32),
                ("head_chunk", C.c_int32), ("log_protocol", C.c_int32), ("keep_host_grad", C.c_int32),
                ("n_buffers", C.c_int32), ("host_grad_accum", C.c_int32), ("n_experts", C.c_int32),
                ("top_k", C.c_int32), ("expert_ffn", C.c_int32), ("debug_guards", C.c_int32)]


class DevRegion(C.Structure):
    _fields_ = [("base", C.c_void_p), ("bytes", C.c_size_t)]


class Streams(C.Structure):
    _fields_ = [("compute", C.c_void_p), ("weight", C.c_void_p), ("grad", C.c_void_p)]


class LayerView(C.Structure):
    _fields_ = [("w", C.c_void_p * MAX_TENSORS), ("g", C.c_void_p * MAX_TENSORS),
                ("n_tensors", C.c_int32), ("block", C.c_int32), ("buf", C.c_int32)]


class SchedIn(C.Structure):
    _fields_ = [("n_visits", C.c_int32), ("kind", C.POINTER(C.c_int32)), ("block", C.POINTER(C.c_int32)),
                ("b", C.POINTER(C.c_double)), ("p", C.POINTER(C.c_double)), ("d", C.POINTER(C.c_double)),
                ("c", C.POINTER(C.c_double)), ("a", C.POINTER(C.c_double)), ("n_buffers", C.c_int32),
                ("bw_h2d", C.c_double), ("bw_d2h", C.c_double), ("pack_rate", C.c_double),
                ("adam_rate", C.c_double), ("adam_bytes", C.c_double), ("host_bw", C.c_double)]


class SchedPlan(C.Structure):
    _fields_ = [("K", C.c_int32), ("measured", C.c_int32), ("period_ms", C.c_double), ("stall_ms", C.c_double),
                ("adam_busy_ms", C.c_double), ("slab_wait_ms", C.c_double), ("pack_ms", C.c_double),
                ("adam_gelem_s", C.c_double), ("bw_h2d_gbs", C.c_double), ("bw_d2h_gbs", C.c_double),
                ("pack_gbs", C.c_double), ("adam_gelem_s_idle", C.c_double), ("host_gbs", C.c_double)]


class Stats(C.Structure):
    _fields_ = [("steps_done", C.c_int64), ("h2d_bytes", C.c_int64), ("d2h_bytes", C.c_int64),
                ("device_bytes_used", C.c_int64), ("last_step_ms", C.c_double),
                ("adam_ms_total", C.c_double), ("pack_ms_total", C.c_double),
                ("host_store_bytes", C.c_int64), ("pinned_bytes", C.c_int64)]


_lib = None
_P = C.POINTER
_v = C.c_void_p


def lib():
    """Loads libmt.so (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    _build()
    L = C.CDLL(_SO_PATH)
    i32, i64, f32, f64, u16, sz = C.c_int32, C.c_int64, C.c_float, C.c_double, C.c_uint16, C.c_size_t
    pc = _P(MtConfig)
    sig = {
        "mt_default_config": (i32, [pc]),
        "mt_query_device_bytes": (i32, [pc, _P(sz)]),
        "mt_init_model": (i32, [pc, DevRegion, Streams, _P(_v)]),
        "mt_set_tokens": (i32, [_v, _P(i32)]),
        "mt_stream_in": (i32, [_v, i32, i32]),
        "mt_bind": (i32, [_v, i32, i32, _P(LayerView)]),
        "mt_step_forward": (i32, [_v, _P(LayerView)]),
        "mt_step_backward": (i32, [_v, _P(LayerView)]),
        "mt_stream_out": (i32, [_v, i32, i32, _P(i32)]),
        "mt_adam_host": (i32, [_v, i32, i32, i32]),
        "mt_train_step": (i32, [_v, i32, _P(f32)]),
        "mt_sync": (i32, [_v]),
        "mt_read_host": (i32, [_v, i32, i32, _v, sz]),
        "mt_write_host": (i32, [_v, i32, i32, _v, sz]),
        "mt_get_stats": (i32, [_v, _P(Stats)]),
        "mt_protocol_log": (i64, [_v, C.c_char_p, i64]),
        "mt_last_error": (C.c_char_p, [_v]),
        "mt_destroy": (None, [_v]),
        "mt_layout_block": (i64, [pc, i32, _P(i64), i64]),
        "mt_param_count": (i64, [pc]),
        "mt_store_bytes": (i64, [pc]),
        "mt_host_init_block": (i32, [pc, i32, _P(f32)]),
        "mt_host_adam": (i32, [i64, _P(u16), _P(f32), _P(f32), _P(f32), _P(u16), i32, f32, f32, f32,
                               f32, f32, i32]),
        "mt_plan_protocol": (i64, [pc, i32, C.c_char_p, i64]),
        "mt_visit_plan": (i32, [pc, _P(i32), _P(i32), i32]),
        "mt_schedule": (i32, [i32, _P(f64), _P(f64), _P(f64), _P(f64), f64, f64, _P(f64)]),
        "mt_schedule_simulate": (i32, [_P(SchedIn), i32, _P(SchedPlan), _P(f64)]),
        "mt_schedule_plan": (i32, [_P(SchedIn), i32, _P(SchedPlan)]),
        "mt_get_schedule": (i32, [_v, i32, _P(SchedPlan)]),
        "mt_token_csr": (i32, [_P(i32), i64, i32, _P(i32), _P(i32)]),
        "mt_host_bandwidth": (i32, [sz, i32, _P(f64), _P(f64)]),
        "mt_rope_table": (i32, [i32, i32, f64, _P(f32)]),
        "mt_timing": (i32, [_v, i32]),
        "mt_timing_read": (i32, [_v, i32, _P(i64), _P(f64), _P(f64), _P(f64)]),
        "mt_timing_visits": (i32, [_v, _P(f64), i32, _P(i32)]),
        "mt_trace": (i32, [_v, i32]),
        "mt_save": (i32, [_v, C.c_char_p]),
        "mt_load": (i32, [_v, C.c_char_p]),
        "mt_trace_json": (i64, [_v, C.c_char_p, i64]),
        "mt_gemm": (i32, [_v, i64, i32, _v, i64, i32, i32, i32, i32, _v, i64, _v, i64, _v, i64, i32, _v]),
        "mt_gemm_mode": (i32, [i32]),
        "mt_gemm2": (i32, [_P(_v), _P(i64), _P(i32), _P(_v), _P(i64), _P(i32), _P(i32), _P(i32), _P(i32),
                            _P(_v), _P(i64), _v]),
        "mt_rmsnorm_fwd": (i32, [_v, _v, i64, i32, f32, _v, _v, _v]),
        "mt_rmsnorm_bwd": (i32, [_v, _v, _v, _v, _v, i64, i32, _v, _v, _v, sz, _v]),
        "mt_rmsnorm_bwd_scratch_bytes": (sz, [i64, i32]),
        "mt_rope": (i32, [_v, i64, i64, i32, i32, i32, _v, i32, _v]),
        "mt_attention_fwd": (i32, [_v, i32, i32, i32, i32, i32, _v, _v, _v]),
        "mt_attention_bwd": (i32, [_v, _v, _v, _v, i32, i32, i32, i32, i32, _v, _v, sz, _v]),
        "mt_attention_bwd_scratch_bytes": (sz, [i32, i32, i32, i32]),
        "mt_swiglu_fwd": (i32, [_v, i64, i32, _v, _v]),
        "mt_swiglu_bwd": (i32, [_v, _v, i64, i32, _v, _v]),
        "mt_embed_fwd": (i32, [_v, _v, i64, i32, i32, _v, _v]),
        "mt_embed_bwd": (i32, [_v, _v, _v, i32, i32, _v, _v]),
        "mt_cross_entropy": (i32, [_v, _v, i64, i32, f32, _v, _v]),
        "mt_kernel_error": (i32, [_P(i32), i32]),
        "mt_fault_inject": (i32, [i32, i32]),
        "mt_moe_scratch_bytes": (sz, [i64, i32, i32, i32, i32]),
        "mt_expert_counts": (i32, [_v, i32, _P(i32), i32]),
        "mt_debug_poke_guard": (i32, [_v, i32, _P(i32)]),
        "mt_moe_ffn": (i32, [_v, _v, _v, _v, _v, i64, i32, i32, i32, i32, _v, _v, _v, _v, _v, _v, _v, sz, _v]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def check(status: int, model=None):
    if status != 0:
        msg = lib().mt_last_error(model).decode() if model is not None else ""
        raise MtError(status, msg)


def make_config(shape: dict, **rt) -> MtConfig:
    """mt_config from a shape dict (see configs.py) plus runtime overrides."""
    c = MtConfig()
    check(lib().mt_default_config(C.byref(c)))
    for k in ("n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "batch", "seq"):
        setattr(c, k, int(shape[k]))
    c.micro_batches = int(shape.get("micro", shape.get("micro_batches", 1)))
    for k in ("n_experts", "top_k", "expert_ffn"):
        setattr(c, k, int(shape.get(k, 0)))
    for k in ("rope_base", "rms_eps", "init_std", "lr", "beta1", "beta2", "adam_eps", "weight_decay"):
        if k in shape:
            setattr(c, k, float(shape[k]))
    for k, v in rt.items():
        setattr(c, k, v)
    return c


def _ptr(a: np.ndarray, ct):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(_P(ct))


def visit_plan(cfg: MtConfig) -> list[tuple[int, int]]:
    """(kind, block) of every visit of one step; kind 0 forward, 1 head,
    2 recompute (driven with step_forward), 3 block backward."""
    n = lib().mt_visit_plan(C.byref(cfg), None, None, 0)
    if n < 0:
        raise MtError(-1, "invalid config")
    k = (C.c_int32 * n)()
    b = (C.c_int32 * n)()
    lib().mt_visit_plan(C.byref(cfg), k, b, n)
    return list(zip(k, b))


def sched_in(kind, block, b, p, d, c, a, n_buffers=2, bw_h2d=2e11, bw_d2h=2e11, pack_rate=1.2e11,
             adam_rate=8.5e9, adam_bytes=28.0, host_bw=0.0):
    """An mt_sched_in over numpy arrays (kept alive on the returned object)."""
    arrs = [np.ascontiguousarray(kind, np.int32), np.ascontiguousarray(block, np.int32)]
    arrs += [np.ascontiguousarray(x, np.float64) for x in (b, p, d, c, a)]
    s = SchedIn(len(arrs[0]), *(_ptr(x, C.c_int32) for x in arrs[:2]), *(_ptr(x, C.c_double) for x in arrs[2:]),
                n_buffers, bw_h2d, bw_d2h, pack_rate, adam_rate, adam_bytes, host_bw)
    s._keep = arrs
    return s


def schedule_simulate(si: SchedIn, K: int) -> tuple[dict, np.ndarray]:
    """mt_schedule_simulate: the predicted steady-state step and per-visit stalls."""
    p = SchedPlan()
    stall = np.zeros(si.n_visits)
    check(lib().mt_schedule_simulate(C.byref(si), K, C.byref(p), _ptr(stall, C.c_double)))
    return {k: getattr(p, k) for k, _ in SchedPlan._fields_}, stall


def schedule_plan(si: SchedIn, k_max: int) -> dict:
    """mt_schedule_plan: the slab count chosen by the simulation."""
    p = SchedPlan()
    check(lib().mt_schedule_plan(C.byref(si), k_max, C.byref(p)))
    return {k: getattr(p, k) for k, _ in SchedPlan._fields_}


def host_bandwidth(nbytes: int = 1 << 30, threads: int = 0) -> dict:
    """Host memory copy bandwidth (GB/s, read + write) and Adam rate."""
    if threads <= 0:
        threads = os.cpu_count() or 1
    a, b = C.c_double(), C.c_double()
    check(lib().mt_host_bandwidth(nbytes, threads, C.byref(a), C.byref(b)))
    return {"copy_gbs": a.value, "adam_gelem_s": b.value, "threads": threads}


def layout(cfg: MtConfig) -> list[dict]:
    out = []
    for j in range(cfg.n_layers + 2):
        buf = np.zeros(64, dtype=np.int64)
        n = lib().mt_layout_block(C.byref(cfg), j, _ptr(buf, C.c_int64), 64)
        if n < 0:
            raise MtError(-1, "bad config")
        nt = int(buf[0])
        out.append(dict(n_tensors=nt, n_real=int(buf[1]), n_pad=int(buf[2]),
                        off_W=int(buf[3]), off_G=int(buf[4]), off_master=int(buf[5]),
                        off_m=int(buf[6]), off_v=int(buf[7]), bytes=int(buf[8]),
                        store_off=int(buf[9]),
                        tensors=[(int(buf[10 + 3 * t]), int(buf[11 + 3 * t]), int(buf[12 + 3 * t]))
                                 for t in range(nt)]))
    return out


class Model:
    """One model: host flat store + device region + three streams."""

    def __init__(self, shape: dict, **rt):
        import torch
        if not torch.cuda.is_available():
            raise RuntimeError("host_memory_centric_gb300.Model needs a CUDA GPU")
        self.shape = dict(shape)
        self.cfg = make_config(shape, **rt)
        L = lib()
        nbytes = C.c_size_t()
        check(L.mt_query_device_bytes(C.byref(self.cfg), C.byref(nbytes)))
        self.device_bytes = int(nbytes.value)
        self.dev = torch.empty(self.device_bytes, dtype=torch.uint8, device="cuda")
        self.streams = [torch.cuda.Stream() for _ in range(3)]
        h = _v()
        st = Streams(self.streams[0].cuda_stream, self.streams[1].cuda_stream, self.streams[2].cuda_stream)
        check(L.mt_init_model(C.byref(self.cfg), DevRegion(self.dev.data_ptr(), self.device_bytes), st,
                              C.byref(h)))
        self.h = h
        self.layout = layout(self.cfg)
        self.T = self.cfg.micro_batches * self.cfg.batch * self.cfg.seq

    # -- training
    def set_tokens(self, tok: np.ndarray):
        tok = np.ascontiguousarray(tok, dtype=np.int32)
        assert tok.size == self.T
        check(lib().mt_set_tokens(self.h, _ptr(tok, C.c_int32)), self.h)

    def train_step(self, step: int, want_loss: bool = True) -> float | None:
        loss = C.c_float()
        check(lib().mt_train_step(self.h, step, C.byref(loss) if want_loss else None), self.h)
        return float(loss.value) if want_loss else None

    def sync(self):
        check(lib().mt_sync(self.h), self.h)

    # -- the pages' primitives, one by one
    def stream_in(self, block, buf):
        check(lib().mt_stream_in(self.h, block, buf), self.h)

    def bind(self, block, buf) -> LayerView:
        v = LayerView()
        check(lib().mt_bind(self.h, block, buf, C.byref(v)), self.h)
        return v

    def step_forward(self, view):
        check(lib().mt_step_forward(self.h, C.byref(view)), self.h)

    def step_backward(self, view):
        check(lib().mt_step_backward(self.h, C.byref(view)), self.h)

    def stream_out(self, block, buf) -> int:
        k = C.c_int32()
        check(lib().mt_stream_out(self.h, block, buf, C.byref(k)), self.h)
        return int(k.value)

    def adam_host(self, block, slab, adam_step):
        check(lib().mt_adam_host(self.h, block, slab, adam_step), self.h)

    # -- host store access (after sync)
    def read(self, block: int, region: int) -> np.ndarray:
        n = self.layout[block]["n_pad"]
        dt = np.uint16 if region < 2 else np.float32
        out = np.empty(n, dtype=dt)
        check(lib().mt_read_host(self.h, block, region, out.ctypes.data, out.nbytes), self.h)
        return out

    def write(self, block: int, region: int, arr: np.ndarray):
        dt = np.uint16 if region < 2 else np.float32
        arr = np.ascontiguousarray(arr, dtype=dt)
        check(lib().mt_write_host(self.h, block, region, arr.ctypes.data, arr.nbytes), self.h)

    def expert_counts(self, block: int) -> np.ndarray:
        """Tokens routed to each expert in block's last forward (MoE models)."""
        n = int(self.cfg.n_experts)
        out = np.zeros(max(n, 1), dtype=np.int32)
        check(lib().mt_expert_counts(self.h, block, _ptr(out, C.c_int32), n), self.h)
        return out

    def stats(self) -> dict:
        s = Stats()
        check(lib().mt_get_stats(self.h, C.byref(s)), self.h)
        return {k: getattr(s, k) for k, _ in Stats._fields_}

    def protocol_log(self) -> list[str]:
        need = -lib().mt_protocol_log(self.h, None, 0)
        buf = C.create_string_buffer(int(need) + 1)
        lib().mt_protocol_log(self.h, buf, need + 1)
        return buf.value.decode().splitlines()

    def timing(self, on: bool):
        check(lib().mt_timing(self.h, int(on)), self.h)

    def timing_read(self, kind: int) -> dict:
        n = C.c_int64(); ms = C.c_double(); fl = C.c_double(); by = C.c_double()
        check(lib().mt_timing_read(self.h, kind, C.byref(n), C.byref(ms), C.byref(fl), C.byref(by)), self.h)
        return dict(launches=n.value, ms=ms.value, flops=fl.value, bytes=by.value)

    def save(self, path: str):
        """Write the host store and the step count (mt_save)."""
        check(lib().mt_save(self.h, os.fsencode(path)), self.h)

    def load(self, path: str):
        """Resume from a file written by save() for a model of this shape."""
        check(lib().mt_load(self.h, os.fsencode(path)), self.h)

    def trace(self, on: bool):
        """Start (clearing it) or stop the stream timeline (mt_trace)."""
        check(lib().mt_trace(self.h, int(on)), self.h)

    def trace_events(self) -> list[dict]:
        """The recorded timeline as Chrome trace events (ts / dur in us)."""
        import json
        need = -lib().mt_trace_json(self.h, None, 0)
        if need <= 0:
            return []
        buf = C.create_string_buffer(int(need) + 1)
        n = lib().mt_trace_json(self.h, buf, need + 1)
        return json.loads(buf.value.decode())["traceEvents"] if n > 0 else []

    def timing_visits(self) -> np.ndarray:
        """Mean compute time (ms) of each visit of the step over the timed steps."""
        n = C.c_int32()
        check(lib().mt_timing_visits(self.h, None, 0, C.byref(n)), self.h)
        out = np.zeros(n.value, dtype=np.float64)
        check(lib().mt_timing_visits(self.h, _ptr(out, C.c_double), n.value, C.byref(n)), self.h)
        return out

    def schedule(self, which: int = 0) -> dict | None:
        """The static schedule the model runs with (mt_get_schedule): 0 the
        plan made at init, 1 the plan on the first step's measured compute
        times (None until that step has completed)."""
        p = SchedPlan()
        st = lib().mt_get_schedule(self.h, which, C.byref(p))
        if st == -2:
            return None
        check(st, self.h)
        return {k: getattr(p, k) for k, _ in SchedPlan._fields_}

    def last_error(self) -> str:
        return lib().mt_last_error(self.h).decode()

    def close(self):
        if getattr(self, "h", None):
            lib().mt_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


from . import ops  # noqa: E402,F401
