"""Benchmark of the layer-streamed training step on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

Prints one JSON line (rank 0).  A step is one mt_train_step: every block
streamed in, run forward, recomputed and run backward, its gradients streamed
out and Adam applied on the host.  `value` is tokens/s with the step's tokens
already resident on the device; `e2e` adds, every step, the upload of that
step's tokens from pinned host memory and the read-back of the loss.  Host
state (weights, gradients, master, moments) lives in host RAM by design, so
every step streams it in both cases.

Multi-GPU: one independent replica per GPU (the path has no exchange step),
weak scaling; value = all ranks' tokens / max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "training tokens/sec (1 GB300, host-resident state); % of step roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "fallback": True}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["fallback"] = False
        return d
    return dict(FALLBACK_PEAKS)


def model_numbers(c, ckpt_interval=1):
    """Parameter count P, tensor FLOPs the method executes per step (forward,
    block recompute, backward; causal attention; head once; with a checkpoint
    interval c > 1 also the segment forwards rebuilt in the backward, L - nseg
    extra layer forwards), and the pages' 6NT + 12 L B S^2 H convention."""
    L, H, nh, nkv, hd, F, V = (c[k] for k in ("n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "ffn",
                                              "vocab"))
    B, S, M = c["batch"], c["seq"], c["micro"]
    t = B * S
    E = c.get("n_experts", 0)
    attn = H * (nh + 2 * nkv) * hd + nh * hd * H
    if E:  # routed experts: a token runs the router and top_k experts (P_mm = active matrix params)
        k, Fe = c["top_k"], c["expert_ffn"]
        P_mm = attn + E * H + k * 3 * H * Fe
        P = L * (attn + E * H + E * 3 * H * Fe + 2 * H) + 2 * V * H + H
    else:
        P_mm = attn + 3 * H * F
        P = L * (P_mm + 2 * H) + 2 * V * H + H
    F_exec = M * (L * (8 * t * P_mm + 9 * B * nh * hd * S * S) + 6 * t * H * V)
    n_recomp = L - -(-L // ckpt_interval)
    F_exec += M * n_recomp * (2 * t * P_mm + 2 * B * nh * hd * S * S)
    # 6 N T with N the parameters a token uses (all of them for a dense model)
    N_active = L * (P_mm + 2 * H) + 2 * V * H + H
    F_pages = 6 * N_active * M * t + 12 * L * B * M * S * S * H
    return P, F_exec, F_pages


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(r[1]) for r in self.rows if len(r) > 8 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) > 8 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in self.rows if len(r) > 8 for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def link_bandwidth(torch, nbytes=1 << 30, reps=10):
    """Pinned cudaMemcpyAsync of 1 GiB per direction (best of reps) and both at once."""
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dev2 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h2 = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    out = {}
    for name in ("h2d", "d2h", "both"):
        best = 1e9
        for _ in range(reps):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            if name in ("h2d", "both"):
                with torch.cuda.stream(s1):
                    dev.copy_(h, non_blocking=True)
            if name in ("d2h", "both"):
                with torch.cuda.stream(s2):
                    h2.copy_(dev2, non_blocking=True)
            torch.cuda.current_stream().wait_stream(s1)
            torch.cuda.current_stream().wait_stream(s2)
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b) / 1e3)
        out[name] = (2 if name == "both" else 1) * nbytes / best
    del dev, dev2, h, h2
    return out


class CpuBaseline:
    """The oracle (single-threaded per op) timed on slices of the workload and
    extrapolated per component to the full step:
    * slice: embedding + 1 full-width decoder layer + head at s tokens, fwd+bwd;
    * the same with 2 layers: the difference is one layer's token-linear cost;
    * attention forward + backward of all heads of one sequence at S_a tokens:
      its cost, scaled by (S / S_a)^2, is the layer's quadratic term.
    full step = L * (T * layer_per_token + B*M * attn(S_a) * (S/S_a)^2)
                + T * head_and_embedding_per_token."""

    def __init__(self, cfg_name, over=None):
        import oracle
        from host_memory_centric_gb300 import configs
        oracle.build()
        self.oracle = oracle
        self.c = configs.get(cfg_name, **(over or {}))
        c = self.c
        self.s = 8 if c["vocab"] > 10000 else min(c["seq"], 64)
        self.sa = min(c["seq"], 256)
        self.W = None

    def _slice(self, layers):
        import numpy as np_
        from host_memory_centric_gb300 import inputs
        c = self.c
        sh = dict(c, n_layers=layers, batch=1, micro=1, seq=self.s, init_std=float(np.float32(0.02)),
                  rms_eps=float(np.float32(1e-6)))
        W = [self.oracle.init_block(sh, 1234, j) for j in range(layers + 2)]
        tok = inputs.tokens(1234, 0, 1, 1, self.s, c["vocab"])
        t0 = time.perf_counter()
        self.oracle.step_fwd_bwd(sh, W, tok, np_.float32)
        return time.perf_counter() - t0

    def _attention(self):
        c = self.c
        nh, nkv, hd, S = c["n_heads"], c["n_kv_heads"], c["head_dim"], self.sa
        rng = np.random.default_rng(0)
        qkv = rng.standard_normal((S, (nh + 2 * nkv) * hd))
        dout = rng.standard_normal((S, nh * hd))
        t0 = time.perf_counter()
        o, lse = self.oracle.attention_fwd(qkv, 1, S, nh, nkv, hd)
        self.oracle.attention_bwd(qkv, o, lse, dout, 1, S, nh, nkv, hd)
        return time.perf_counter() - t0

    def calibrate(self):
        """The per-layer and attention terms (run once; part of the warm-up)."""
        t1 = self._slice(1)
        t2 = self._slice(2)
        self.layer_tok = max(t2 - t1, 1e-9) / self.s
        self.attn = self._attention()
        return t1 + t2 + self.attn

    def sample(self):
        """One timed slice (embedding + 1 layer + head); returns (seconds,
        extrapolated full-step seconds)."""
        c = self.c
        t1 = self._slice(1)
        head_tok = max(t1 / self.s - self.layer_tok, 0.0)
        T = c["micro"] * c["batch"] * c["seq"]
        per_layer = T * self.layer_tok + c["batch"] * c["micro"] * self.attn * (c["seq"] / self.sa) ** 2
        return t1, c["n_layers"] * per_layer + T * head_tok

    def describe(self, n, t_sample):
        return (f"oracle, one thread per op: slices of the workload timed and extrapolated per component to the "
                f"full step -- embedding + 1 full-width layer + head at {self.s} tokens ({n} run(s), "
                f"{t_sample:.2f} s each), the same with 2 layers for the per-layer cost, and attention fwd+bwd "
                f"of all heads at {self.sa} tokens scaled by (S/{self.sa})^2 (extrapolated)")


def tiny_full_steps(n=3):
    """The oracle on whole steps of the tiny config (measured, not extrapolated)."""
    import oracle
    from host_memory_centric_gb300 import configs, inputs
    c = configs.get("tiny")
    sh = dict(c, init_std=float(np.float32(0.02)), rms_eps=float(np.float32(1e-6)))
    W = [oracle.init_block(sh, 1234, j) for j in range(c["n_layers"] + 2)]
    ts = []
    for k in range(n):
        tok = inputs.tokens_for(c, k)
        t0 = time.perf_counter()
        oracle.step_fwd_bwd(sh, W, tok, np.float32)
        ts.append(time.perf_counter() - t0)
    return configs.tokens_per_step(c) / statistics.median(ts)


def cpu_sample(cfg_name, over=None):
    """cpu_baseline of the bench line: calibration + 3 slice samples
    (about 30 s at the 7.6B shape) and whole tiny steps."""
    cb = CpuBaseline(cfg_name, over)
    t_cal = cb.calibrate()
    res = [cb.sample() for _ in range(3)]
    t_s = statistics.median(r[0] for r in res)
    full = statistics.median(r[1] for r in res)
    T = cb.c["micro"] * cb.c["batch"] * cb.c["seq"]
    return {"value": T / full, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": cb.describe(len(res), t_s), "extrapolated": True, "full_step_s_extrapolated": full,
            "tiny_full_step_tokens_s": tiny_full_steps(), "seconds": t_cal + sum(r[0] for r in res)}


def schedule_report(m, vis_ms, t_step):
    """The static schedule the library runs with (mt_get_schedule): its plan
    at init (compute estimated from FLOPs) and after the first step (compute
    measured), each with its predicted step time and compute-stream stall,
    beside the stall measured here: the timed step minus the compute of its
    visits (per-visit CUDA events of the timed steps)."""
    p0, p1 = m.schedule(0), m.schedule(1)
    keep = ("K", "measured", "period_ms", "stall_ms", "adam_busy_ms", "slab_wait_ms", "pack_ms", "adam_gelem_s")
    out = {"init": {k: p0[k] for k in keep}, "after_first_step": ({k: p1[k] for k in keep} if p1 else None),
           "probes": {k: p0[k] for k in ("bw_h2d_gbs", "bw_d2h_gbs", "pack_gbs", "adam_gelem_s_idle", "host_gbs")}}
    if len(vis_ms) and np.all(vis_ms > 0):
        out["measured"] = {"step_ms": t_step * 1e3, "compute_ms": float(vis_ms.sum()),
                           "stall_ms": float(t_step * 1e3 - vis_ms.sum())}
    out["note"] = ("K set by the plan at init; predicted = the pipeline model (link, chunked pack, compute, "
                   "export into K slabs, host Adam sharing the measured host-memory bandwidth with DMA and the pack)")
    return out


def _union(iv):
    """Total length of the union of intervals [(t0, t1), ...]."""
    tot, end = 0.0, None
    for a, b in sorted(iv):
        if end is None or a > end:
            tot += b - a
            end = b
        elif b > end:
            tot += b - end
            end = b
    return tot


def _overlap(x, y):
    """Length of union(x) intersected with union(y)."""
    return _union(x) + _union(y) - _union(x + y)


def switch_gaps(ev):
    """Buffer-switch latency on the compute stream: for each pair of
    consecutive visits whose second visit's weights were already resident
    (its block's latest H2D copy ended before the first visit's compute
    ended), the idle time between the two compute spans -- the cost of
    switching buffers and binding the next layer (one page sets a target
    under 100 us).  Such a gap can also hold a wait for a checkpoint slot or
    a gradient slab; those show up in the tail.  Times in us."""
    comp = sorted((e for e in ev if e.get("tid") == "compute stream"), key=lambda e: e["ts"])
    h2d = sorted((e for e in ev if e.get("tid") == "weight stream" and e["name"].split()[0] == "H2D"),
                 key=lambda e: e["ts"])
    gaps = []
    for a, b in zip(comp, comp[1:]):
        blk = b.get("args", {}).get("block")
        ready = [h for h in h2d if h.get("args", {}).get("block") == blk and h["ts"] < b["ts"]]
        if ready and ready[-1]["ts"] + ready[-1]["dur"] <= a["ts"] + a["dur"]:
            gaps.append(max(0.0, b["ts"] - (a["ts"] + a["dur"])))
    if not gaps:
        return None
    g = np.sort(np.array(gaps))
    return {"pairs": int(len(g)), "median_us": float(np.median(g)), "p90_us": float(np.percentile(g, 90)),
            "max_us": float(g[-1]), "over_100us": int((g > 100.0).sum())}


def timeline(m, toks, step, path=""):
    """Two steps traced in the steady state (recording starts without draining
    the pipeline, after an untraced step) and one period analysed: from the
    start of the first traced step's first compute to the start of the
    second's.  Busy fractions of the weight, compute and gradient streams and
    of host Adam within it, the share of weight-copy time overlapped by
    compute (the pages' overlap ratio) and the buffer-switch latency."""
    m.set_tokens(toks[0])
    m.train_step(step, want_loss=False)
    m.trace(True)
    for k in (1, 2):
        m.set_tokens(toks[k])
        m.train_step(step + k, want_loss=False)
    m.sync()
    ev = m.trace_events()
    m.trace(False)
    if path:
        with open(path, "w") as f:
            json.dump({"traceEvents": ev}, f)
    comp0 = sorted((e for e in ev if e["tid"] == "compute stream" and e["args"].get("block") == 0
                    and e["name"].startswith("FWD")), key=lambda e: e["ts"])
    if len(comp0) < 2:
        return None
    t0, t1 = comp0[0]["ts"] / 1e3, comp0[1]["ts"] / 1e3
    span = t1 - t0
    clip = lambda a, b: (max(a, t0), min(b, t1))
    by = {}
    for e in ev:
        a, b = clip(e["ts"] / 1e3, (e["ts"] + e["dur"]) / 1e3)
        if b > a:
            by.setdefault(e["tid"], []).append((a, b))
    busy = {k: _union(v) / span for k, v in by.items()}
    w, c = by.get("weight stream", []), by.get("compute stream", [])
    try:
        sw = switch_gaps(ev)
    except Exception as e:  # a statistic of the trace must not cost the benchmark line
        sw = {"error": repr(e)}
    return {"period_ms": span, "busy_frac": busy,
            "weight_copy_overlapped_by_compute": _overlap(w, c) / max(_union(w), 1e-9),
            "buffer_switch": sw, "events": len(ev), "file": path or None,
            "window": "steady state: start of one step's first compute to the next step's"}


def cpu_model() -> str:
    """CPU model of this host (lscpu's model name, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def mem_available_bytes() -> int:
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def host_bytes_needed(c: dict, slabs: int, ckpt_on_host: int, ckpt_interval: int = 1, host_accum: int = 0) -> int:
    """Host RAM one replica allocates: the flat store, the pinned gradient
    slabs (largest block's gradient region each) and the checkpoints."""
    import ctypes
    import host_memory_centric_gb300 as mt
    cfg = mt.make_config(c)
    store = mt.lib().mt_store_bytes(ctypes.byref(cfg))
    wb = max(2 * b["n_pad"] for b in mt.layout(cfg))
    nseg = -(-c["n_layers"] // ckpt_interval)
    micro_per_pass = 1 if host_accum else c["micro"]
    ckpt = nseg * micro_per_pass * c["batch"] * c["seq"] * c["hidden"] * 2 if ckpt_on_host else 0
    acc = 2 * sum(b["n_pad"] for b in mt.layout(cfg)) * 2 if host_accum else 0  # FP32 accumulator
    return int(store + slabs * wb + 2 * wb + ckpt + acc)


def all_max(x: float, dist=None, device="cpu") -> float:
    """Maximum of x over the ranks of the process group (x itself without one)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(t_step_local: float, tokens_per_step: int, world: int, dist=None, device="cpu"):
    """Whole-job throughput of independent replicas: every rank trains its own
    copy on its own tokens, so value = world x tokens / (slowest rank's step)."""
    t = all_max(t_step_local, dist, device)
    return world * tokens_per_step / t, t


def workload_desc(name, c):
    mlp = (f"{c['n_experts']} routed SwiGLU experts of FFN {c['expert_ffn']}, top-{c['top_k']} (only routed "
           f"experts streamed)" if c.get("n_experts") else f"FFN {c['ffn']}")
    return (f"{name}-shaped decoder: {c['n_layers']} layers, hidden {c['hidden']}, {c['n_heads']}x{c['head_dim']} "
            f"heads ({c['n_kv_heads']} KV), {mlp}, vocab {c['vocab']}, batch {c['batch']} x seq "
            f"{c['seq']} x {c['micro']} micro-batches; host-resident BF16/FP32 state, host Adam")


def run_reference(args):
    """The oracle on the host cores, for the same workload, metric and unit.
    Warm-up: the calibration runs of CpuBaseline (the per-layer and attention
    terms) and W untimed slices.  Each of the K timed steps is one slice
    (embedding + one full-width layer + head at a few tokens); ms_per_step is
    the measured time of those slices, and value the full workload's tokens/s
    extrapolated from them (labelled)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    t_start = time.time()
    cb = CpuBaseline(args.config, _overrides(args))
    cb.calibrate()
    for _ in range(args.warmup):
        cb.sample()
    res = [cb.sample() for _ in range(args.steps)]
    t_sample = statistics.mean(r[0] for r in res)
    full = statistics.median(r[1] for r in res)
    c = cb.c
    T = c["micro"] * c["batch"] * c["seq"]
    v = T / full
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_sample,
            "ms_per_step_is": "measured time of one timed slice (the step's unit of work here)",
            "full_step_ms_extrapolated": 1e3 * full, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": workload_desc(args.config, c), "model": args.config,
                       "global_batch": c["batch"] * c["micro"], "seq_len": c["seq"], "parallelism": "none (CPU)"},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": cb.describe(len(res), t_sample), "extrapolated": True},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.time() - t_start}
    print(json.dumps(line), flush=True)


def _overrides(args):
    over = {"n_layers": args.layers} if args.layers > 0 else {}
    for kv in args.set:
        key, _, val = kv.partition("=")
        over[key] = float(val) if "." in val or "e" in val.lower() else int(val)
    return over


# DRAM bytes (read + write) per GEMM launch, from one ncu capture of the
# GEMM forms of one decoder layer of the default workload (the 7.6B-shaped
# decoder at 16384 tokens per visit, launched by `kbench layer_gemms`;
# metrics dram__bytes_read.sum and dram__bytes_write.sum, each form weighted
# by its launches per step: 308 of the step's 310 GEMM launches, the LM
# head's two not captured).  Valid only for the kernel source it was taken
# from: any change to the GEMM kernel reports null.
GEMM_TRAFFIC = {"source_sha256_16": "a80f201da4b6d1a5", "config": "7.6b", "bytes_per_launch": 2.2463e9}


def gemm_traffic_per_launch(name, c, args):
    import hashlib
    root = os.path.join(os.path.dirname(os.path.abspath(__file__)), "host_memory_centric_gb300", "csrc")
    h = hashlib.sha256()
    with open(os.path.join(root, "k_gemm.cu"), "rb") as fh:
        h.update(fh.read())
    default_shape = (name == GEMM_TRAFFIC["config"] and not args.set and not args.layers and args.ckpt_interval == 1
                     and args.buffers == 2 and not args.host_accum)
    if h.hexdigest()[:16] != GEMM_TRAFFIC["source_sha256_16"] or not default_shape:
        return None
    return GEMM_TRAFFIC["bytes_per_launch"]


def host_triad(torch, n=1 << 28):
    """STREAM triad a = b + s c over 1 GiB float32 arrays on torch's CPU
    threads (one per online core): GB/s counting 12 bytes per element."""
    thr = os.cpu_count() or 1
    old = torch.get_num_threads()
    torch.set_num_threads(thr)
    a = torch.empty(n, dtype=torch.float32)
    b = torch.ones(n, dtype=torch.float32)
    c = torch.ones(n, dtype=torch.float32)
    best = 1e9
    for _ in range(4):
        t0 = time.perf_counter()
        torch.add(b, c, alpha=3.0, out=a)
        best = min(best, time.perf_counter() - t0)
    torch.set_num_threads(old)
    del a, b, c
    return {"triad_GBs": 12 * n / best / 1e9, "threads": thr, "cores": os.cpu_count()}


def device_used(torch):
    free, total = torch.cuda.mem_get_info()
    return total - free


def side_run(mt, torch, inputs, c, steps, warmup, pin_store, seed=7):
    """A short run of another shape (the 14.7B width at reduced depth):
    tokens/s over `steps` steps after `warmup`, the device region carved, the
    peak device memory in use above the level before the model existed, and
    the host state."""
    torch.cuda.synchronize()
    base = device_used(torch)
    m = mt.Model(c, seed=seed, pin_store=pin_store, keep_host_grad=0)
    peak = device_used(torch) - base
    step = 0
    for _ in range(warmup):
        m.set_tokens(inputs.tokens_for(c, step))
        m.train_step(step, want_loss=False)
        step += 1
        peak = max(peak, device_used(torch) - base)
    m.sync()
    w0 = time.perf_counter()
    for _ in range(steps):
        m.set_tokens(inputs.tokens_for(c, step))
        m.train_step(step, want_loss=False)
        step += 1
        peak = max(peak, device_used(torch) - base)
    m.sync()
    dt = (time.perf_counter() - w0) / max(steps, 1)
    st = m.stats()
    T = c["micro"] * c["batch"] * c["seq"]
    out = {"n_layers": c["n_layers"], "tokens_per_s": T / dt if steps else None, "ms_per_step": dt * 1e3 if steps else None,
           "device_region_GB": m.device_bytes / 1e9, "device_peak_used_GB": peak / 1e9,
           "host_store_GB": st["host_store_bytes"] / 1e9, "pinned_GB": st["pinned_bytes"] / 1e9,
           "params": int(sum(b["n_real"] for b in m.layout))}
    m.close()
    del m
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="7.6b")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--pin-store", type=int, default=0,
                    help="0: just-in-time pack into pinned staging (the method); 1: register the whole store")
    ap.add_argument("--threads", type=int, default=0)
    ap.add_argument("--slabs", type=int, default=0, help="gradient slabs K (0: chosen by the static schedule)")
    ap.add_argument("--keep-host-grad", type=int, default=0)
    ap.add_argument("--ckpt-on-host", type=int, default=1)
    ap.add_argument("--ckpt-interval", type=int, default=1, help="layers per recompute segment")
    ap.add_argument("--buffers", type=int, default=2, help="device weight buffers (1: single-buffer ablation)")
    ap.add_argument("--layers", type=int, default=0, help="decoder depth override (depth sweeps; 0 = the config's)")
    ap.add_argument("--trace", default="", help="write the steady-state stream timeline (Chrome trace JSON)")
    ap.add_argument("--host-accum", type=int, default=0,
                    help="1: one pass per micro-batch, gradients summed in FP32 on the host")
    ap.add_argument("--set", action="append", default=[], metavar="KEY=VALUE",
                    help="override a shape field of the config (e.g. hidden=4096); repeatable")
    ap.add_argument("--timeout", type=float, default=0,
                    help="limit of every bounded host wait, seconds (0: four times the step's tensor work at "
                         "400 TFLOP/s, at least 60 s)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--wide-layers", type=int, default=24,
                    help="after the main run: the 14.7B-shaped decoder at this depth (its full 48 layers need "
                         "more host RAM than one GB300's share) and the footprint at half of it; 0: skip")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import host_memory_centric_gb300 as mt
    from host_memory_centric_gb300 import configs, inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    def barrier():
        if dist:
            dist.barrier()
        torch.cuda.synchronize()

    c = configs.get(args.config, **_overrides(args))
    T = c["micro"] * c["batch"] * c["seq"]
    P, F_exec, F_pages = model_numbers(c, args.ckpt_interval)
    # every replica on this host holds its own host state: refuse to start
    # rather than exhaust host RAM
    local_world = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    need = local_world * host_bytes_needed(c, args.slabs or 16, args.ckpt_on_host, args.ckpt_interval,
                                           args.host_accum)
    avail = mem_available_bytes()
    if avail and need > 0.85 * avail:
        msg = (f"{local_world} replica(s) of the {args.config} workload need {need / 1e9:.1f} GB of host RAM; "
               f"{avail / 1e9:.1f} GB available")
        if rank == 0:
            print(json.dumps({"metric": METRIC, "error": msg, "n_gpus": world}), flush=True)
        sys.exit(2)
    pk = peaks()
    bw = link_bandwidth(torch)
    hbw = mt.host_bandwidth(1 << 30)
    triad = host_triad(torch)

    t_init = time.time()
    # every host wait of the library is bounded; a long-context step is minutes of GPU work
    timeout_s = args.timeout if args.timeout > 0 else max(60.0, 4.0 * F_exec / 4e14)
    dev_base = device_used(torch)
    m = mt.Model(c, seed=1234, pin_store=args.pin_store, n_host_threads=args.threads, n_grad_slabs=args.slabs,
                 timeout_ms=int(min(timeout_s * 1e3, 4.0e9)),
                 keep_host_grad=args.keep_host_grad, ckpt_on_host=args.ckpt_on_host,
                 ckpt_interval=args.ckpt_interval, n_buffers=args.buffers, host_grad_accum=args.host_accum)
    init_s = time.time() - t_init
    toks = [inputs.tokens_for(c, s) for s in range(args.warmup + 2 * args.steps + 4)]
    step = 0
    dev_peak = device_used(torch) - dev_base
    for w in range(args.warmup):
        m.set_tokens(toks[step])
        m.train_step(step)
        step += 1
        dev_peak = max(dev_peak, device_used(torch) - dev_base)
    m.sync()

    # ---------------- device-resident tokens: the kernel-side number
    m.set_tokens(toks[step])
    m.sync()
    cs = m.streams[0]  # the compute stream the library launches on
    barrier()
    m.timing(True)
    st0 = m.stats()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(cs)
        w0 = time.perf_counter()
        losses = []
        for k in range(args.steps):
            losses.append(m.train_step(step, want_loss=(k == args.steps - 1)))
            step += 1
        m.sync()
        ev1.record(cs)
        torch.cuda.synchronize()
        wall = time.perf_counter() - w0
    barrier()
    dev_peak = max(dev_peak, device_used(torch) - dev_base)
    dev_s = ev0.elapsed_time(ev1) / 1e3
    kern = {name: m.timing_read(i) for i, name in enumerate(("gemm", "attn_fwd", "attn_bwd", "other"))}
    vis_ms = m.timing_visits()
    m.timing(False)
    st1 = m.stats()
    value, t_step = aggregate(max(dev_s, wall) / args.steps, T, world, dist, "cuda")

    # ---------------- end to end: tokens uploaded and loss read back every step
    e2e = None
    if not args.no_e2e:
        barrier()
        sh0 = m.stats()
        w0 = time.perf_counter()
        ev0.record(cs)
        for k in range(args.steps):
            m.set_tokens(toks[step])
            m.train_step(step, want_loss=True)
            step += 1
        m.sync()
        ev1.record(cs)
        torch.cuda.synchronize()
        e2e_v, e2e_s = aggregate(max(time.perf_counter() - w0, ev0.elapsed_time(ev1) / 1e3) / args.steps, T,
                                 world, dist, "cuda")
        sh1 = m.stats()
        e2e = {"value": e2e_v, "unit": "tokens/s",
               "h2d_bytes_per_step": int((sh1["h2d_bytes"] - sh0["h2d_bytes"]) / args.steps),
               "d2h_bytes_per_step": int((sh1["d2h_bytes"] - sh0["d2h_bytes"]) / args.steps)}

    if rank != 0:
        m.close()
        if dist:
            dist.destroy_process_group()
        return

    g = kern["gemm"]
    traffic = gemm_traffic_per_launch(args.config, c, args)
    # the GEMMs run inside a seconds-long step: the sustained peak unless the
    # clocks stayed at their maximum with no power cap, then the burst peak
    ck = clk.summary()
    burst = (ck.get("sm_mhz") is not None and ck.get("sm_max_mhz") and ck["sm_mhz"] >= 0.99 * ck["sm_max_mhz"]
             and "sw_power_cap" not in ck.get("reasons", []))
    peak_key = "bf16_tflops" if burst else "bf16_tflops_sustained"
    peak_t = pk.get(peak_key, 1700.0)
    achieved = g["flops"] / (g["ms"] / 1e3) / 1e12 if g["ms"] > 0 else None
    burst_t = pk.get("bf16_tflops", 1900.0)
    roof = {"bound": "tensor", "kernel": "gemm_pair_kernel / gemm_kernel (tcgen05 BF16 GEMM, all projections)",
            "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s",
            "frac": (achieved / peak_t) if achieved else None, "traffic": traffic,
            "frac_of_burst": (achieved / burst_t) if achieved else None,
            "peak_source": peak_key + " of " + ("fallback" if pk.get("fallback") else "measured"),
            "launches": g["launches"], "avg_launch_ms": g["ms"] / max(1, g["launches"]),
            "flops_per_launch": g["flops"] / max(1, g["launches"])}
    t_compute = F_exec / (pk.get("bf16_tflops_sustained", 1700.0) * 1e12)
    t_link = max(2 * P / bw["h2d"], 2 * P / bw["d2h"])
    t_roof = max(t_compute, t_link)
    kernels = {}
    for name, k in kern.items():
        if k["launches"]:
            kernels[name] = {"launches": k["launches"], "ms_per_step": k["ms"] / args.steps,
                             "TFLOP/s": (k["flops"] / (k["ms"] / 1e3) / 1e12) if k["flops"] else None,
                             "GB/s": (k["bytes"] / (k["ms"] / 1e3) / 1e9) if k["bytes"] else None}
    launches = sum(k["launches"] for k in kern.values())
    # host memory traffic per step: Adam reads slab (2 B) + master, m, v (12 B), writes master, m, v
    # (12 B) + W (2 B) [+ G (2 B) when unpacking]; every DMA reads or writes host memory once; the
    # just-in-time pack reads the store and writes staging (2 x the bytes it packs)
    n_pad = sum(b["n_pad"] for b in m.layout)
    adam_b = n_pad * (28 + 2 * args.keep_host_grad)
    dma_b = (st1["h2d_bytes"] - st0["h2d_bytes"] + st1["d2h_bytes"] - st0["d2h_bytes"]) / args.steps
    pack_b = 0.0
    if not args.pin_store:
        plan = mt.visit_plan(m.cfg)
        pack_b = 2.0 * sum(2 * m.layout[j]["n_pad"] for k, j in plan if not (k == 3 and j == 0))
    host_b = adam_b + dma_b + pack_b
    t_host = host_b / (triad["triad_GBs"] * 1e9)
    host = {"adam_ms_per_step": (st1["adam_ms_total"] - st0["adam_ms_total"]) / args.steps,
            "pack_ms_per_step": (st1["pack_ms_total"] - st0["pack_ms_total"]) / args.steps,
            "h2d_GB_per_step": (st1["h2d_bytes"] - st0["h2d_bytes"]) / args.steps / 1e9,
            "d2h_GB_per_step": (st1["d2h_bytes"] - st0["d2h_bytes"]) / args.steps / 1e9,
            "device_bytes": m.device_bytes, "device_peak_used_GB": dev_peak / 1e9,
            "host_store_GB": st1["host_store_bytes"] / 1e9, "pinned_GB": st1["pinned_bytes"] / 1e9,
            "init_s": init_s, "nproc": os.cpu_count(), "cpu_model": cpu_model(), "last_loss": losses[-1]}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded uniform token ids, N(0,0.02) weights)",
        "config": {"workload": workload_desc(args.config, c), "model": args.config,
                   "global_batch": world * c["batch"] * c["micro"], "seq_len": c["seq"],
                   "tokens_per_step": T, "parallelism": f"replicas x{world} (no exchange step)",
                   "pin_store": args.pin_store, "n_grad_slabs": m.schedule(0)["K"] if not args.slabs else args.slabs,
                   "keep_host_grad": args.keep_host_grad, "ckpt_on_host": args.ckpt_on_host,
                   "ckpt_interval": args.ckpt_interval, "n_buffers": args.buffers,
                   "host_grad_accum": args.host_accum,
                   "l2": "inputs larger than L2 (every step streams "
                   f"{2 * P / 1e9:.2f} GB of weights in and out)"},
        "step_roofline": {"frac": t_roof / t_step, "t_roof_ms": t_roof * 1e3, "t_step_ms": t_step * 1e3,
                          "bound": "tensor" if t_compute >= t_link else "host link",
                          "F_exec_pflop": F_exec / 1e15, "peak_tflops": pk.get("bf16_tflops_sustained", 1700.0),
                          "link_h2d_GBs": bw["h2d"] / 1e9, "link_d2h_GBs": bw["d2h"] / 1e9,
                          "link_both_GBs": bw["both"] / 1e9, "params": P,
                          "pages_tflops_convention": F_pages / t_step / 1e12,
                          "model_tflops_executed": F_exec / t_step / 1e12},
        "host_dram_bound": {"triad_GBs": triad["triad_GBs"], "triad_threads": triad["threads"],
                            "host_copy_GBs": hbw["copy_gbs"], "host_adam_Gelem_s": hbw["adam_gelem_s"],
                            "threads": hbw["threads"], "bytes_per_step_GB": host_b / 1e9,
                            "bytes_per_param": host_b / P, "adam_GB": adam_b / 1e9, "dma_GB": dma_b / 1e9,
                            "pack_GB": pack_b / 1e9, "t_host_ms": t_host * 1e3, "frac": t_host / t_step,
                            "note": "host memory traffic of Adam, DMA and the pack over the measured STREAM triad "
                                    "bandwidth; not part of the step roofline"},
        "roofline": roof,
        "kernels": kernels,
        "cpu_baseline": None,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": ck,
        "host": host,
    }
    line["schedule"] = schedule_report(m, vis_ms, t_step)
    line["timeline"] = timeline(m, toks[step:step + 3], step, args.trace)
    step += 3
    if c.get("n_experts"):
        # routed experts of the last forward: how many experts each layer's
        # stream-ins copied, and the load of the busiest expert over the mean
        cnt = np.stack([m.expert_counts(j) for j in range(1, c["n_layers"] + 1)])
        line["moe"] = {"n_experts": c["n_experts"], "top_k": c["top_k"],
                       "routed_experts_per_layer": [int(x) for x in (cnt > 0).sum(axis=1)],
                       "routed_frac": float((cnt > 0).mean()),
                       "max_over_mean_load": float((cnt.max(axis=1) / cnt.mean(axis=1)).mean())}
    m.close()
    del m
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    # ---------------- the 14.7B width at reduced depth, and the footprint over depth
    if args.wide_layers > 0 and world == 1 and not args.layers and not args.set:
        wide = {}
        try:
            for d, (st, wu) in ((args.wide_layers, (3, 2)), (args.wide_layers // 2, (0, 2))):
                cw = configs.get("14.7b", n_layers=d)
                if host_bytes_needed(cw, 16, 1) > 0.85 * mem_available_bytes():
                    wide[str(d)] = {"skipped": "host RAM"}
                    continue
                wide[str(d)] = side_run(mt, torch, inputs, cw, st, wu, args.pin_store)
            r = wide.get(str(args.wide_layers), {})
            if r.get("tokens_per_s"):
                Pw, Fw, _ = model_numbers(configs.get("14.7b", n_layers=args.wide_layers))
                r["step_roofline_frac"] = max(Fw / (pk.get("bf16_tflops_sustained", 1700.0) * 1e12),
                                              2 * Pw / bw["h2d"], 2 * Pw / bw["d2h"]) / (r["ms_per_step"] / 1e3)
        except Exception as e:  # a side measurement must not cost the benchmark line
            wide["error"] = repr(e)
        line["width_14p7b"] = {"runs": wide, "note": "14.7B-shaped decoder (hidden 5120, 40/8 heads, FFN 13824, "
                               "vocab 152064, 4 x 4096 tokens) at reduced depth: host-state of all 48 layers (236 GB) "
                               "exceeds this host; tokens/s over 3 steps after 2, footprint = device memory in use"}
        line["footprint"] = {"by_depth_14p7b_width": {d: {k: v for k, v in r.items() if k.startswith(("device", "n_"))}
                                                      for d, r in wide.items() if isinstance(r, dict)},
                             "main_run_GB": {"device_region": line["host"]["device_bytes"] / 1e9,
                                             "device_peak_used": dev_peak / 1e9}}
    if not args.no_cpu and world == 1:
        try:
            line["cpu_baseline"] = cpu_sample(args.config, _overrides(args))
        except Exception as e:  # the oracle is a reported baseline only
            line["cpu_baseline"] = {"value": None, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                    "sample": f"failed: {e}"}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
