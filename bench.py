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


def cpu_sample(cfg_name, budget_s=20.0):
    """Times the oracle (single-threaded) on a depth-1, full-width slice of
    the workload with one short sequence and applies its FLOP rate to the
    full workload's FLOPs (an extrapolation, labelled as such)."""
    import oracle
    from host_memory_centric_gb300 import configs, inputs
    c = configs.get(cfg_name)
    seq = 32 if c["vocab"] > 10000 else min(c["seq"], 128)
    s = dict(c, n_layers=1, batch=1, micro=1, seq=seq, init_std=float(np.float32(0.02)))
    oracle.build()
    W = []
    for j in range(3):
        W.append(oracle.init_block(s, 1234, j))
    tok = inputs.tokens(1234, 0, 1, 1, seq, c["vocab"])
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.step_fwd_bwd(s, W, tok, np.float32)
        n += 1
        if time.perf_counter() - t0 > budget_s / 2 or n >= 3:
            break
    dt = (time.perf_counter() - t0) / n
    _, F_sample, _ = model_numbers(dict(s, micro=1))
    _, F_full, _ = model_numbers(c)
    T_full = c["micro"] * c["batch"] * c["seq"]
    flops_rate = F_sample / dt
    tok_s = flops_rate * T_full / F_full
    return {"value": tok_s, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"oracle fwd+bwd of a 1-layer, full-width slice, 1 x {seq} tokens, {n} run(s) of "
                      f"{dt:.2f} s; its FLOP rate ({flops_rate / 1e9:.2f} GFLOP/s) applied to the full "
                      f"workload's {F_full / 1e15:.4f} PFLOP per step (extrapolated)",
            "seconds": dt * n}


def static_schedule(m, vis_ms, bw, hbw, slabs):
    """The static prefetch schedule (mt_schedule) evaluated on this run's
    measurements: per visit the H2D bytes of its block, the exported gradient
    bytes, the measured compute time of the visit and the host Adam time of
    its block at the measured Adam rate; the measured link bandwidths.  It
    predicts the compute stream's stalls and the slab pool the exports need
    (the host Adam bound is outside its model)."""
    import ctypes
    import host_memory_centric_gb300 as mt
    plan = mt.visit_plan(m.cfg)
    lay = m.layout
    n = len(plan)
    if len(vis_ms) != n or not np.all(vis_ms > 0):
        return None
    D = ctypes.POINTER(ctypes.c_double)
    b = np.array([0.0 if (k == 3 and j == 0) else 2.0 * lay[j]["n_pad"] for k, j in plan])
    d = np.array([2.0 * lay[j]["n_pad"] if k in (1, 3) else 0.0 for k, j in plan])
    a = np.array([lay[j]["n_pad"] / (hbw["adam_gelem_s"] * 1e9) if k in (1, 3) else 0.0 for k, j in plan])
    cv = np.ascontiguousarray(vis_ms / 1e3)
    stall = np.zeros(n)
    p = lambda x: x.ctypes.data_as(D)
    need = mt.lib().mt_schedule(n, p(b), p(d), p(cv), p(a), bw["h2d"], bw["d2h"], p(stall))
    return {"visits": n, "compute_ms_per_step": float(cv.sum() * 1e3),
            "predicted_stall_ms_per_step": float(stall.sum() * 1e3),
            "predicted_gpu_timeline_ms": float((cv + stall).sum() * 1e3),
            "worst_visit_stall_ms": float(stall.max() * 1e3), "slabs_needed": int(need), "slabs_used": slabs,
            "note": "mt_schedule on measured per-visit compute, block bytes, link bandwidth and Adam rate; "
                    "host Adam throughput is not in its model"}


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


def timeline(m, tok, step, path=""):
    """One extra step (outside the timed region) with the stream timeline
    on: busy fractions of the weight, compute and gradient streams and of
    host Adam over the step's span (first copy to last Adam job), and how
    much of the weight stream's copying overlaps compute (the pages' overlap
    ratio)."""
    m.set_tokens(tok)
    m.trace(True)
    m.train_step(step, want_loss=False)
    m.sync()
    ev = m.trace_events()
    m.trace(False)
    if path:
        with open(path, "w") as f:
            json.dump({"traceEvents": ev}, f)
    by = {}
    for e in ev:
        by.setdefault(e["tid"], []).append((e["ts"] / 1e3, (e["ts"] + e["dur"]) / 1e3))
    allv = [iv for v in by.values() for iv in v]
    if not allv:
        return None
    t0, t1 = min(a for a, _ in allv), max(b for _, b in allv)  # first copy .. last Adam
    span = t1 - t0
    busy = {k: _union(v) / span for k, v in by.items()}
    w, c = by.get("weight stream", []), by.get("compute stream", [])
    try:
        sw = switch_gaps(ev)
    except Exception as e:  # a statistic of the trace must not cost the benchmark line
        sw = {"error": repr(e)}
    return {"span_ms": span, "busy_frac": busy,
            "weight_copy_overlapped_by_compute": _overlap(w, c) / max(_union(w), 1e-9),
            "buffer_switch": sw, "events": len(ev), "file": path or None}


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
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from host_memory_centric_gb300 import configs
    c = configs.get(args.config)
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state
    vals = []
    t0 = time.time()
    per_step = max(5.0, 60.0 / max(1, args.steps))
    for _ in range(args.steps):
        r = cpu_sample(args.config, budget_s=per_step)
        vals.append(r["value"])
    v = statistics.median(vals)
    T = c["micro"] * c["batch"] * c["seq"]
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * T / v, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": workload_desc(args.config, c), "model": args.config,
                       "global_batch": c["batch"] * c["micro"], "seq_len": c["seq"], "parallelism": "none (CPU)"},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": r["sample"]},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.time() - t0}
    print(json.dumps(line), flush=True)


# DRAM bytes (read + write) per GEMM launch from one ncu capture of the
# default 1.2B-shaped step (metrics dram__bytes_read.sum, dram__bytes_write.sum
# over the 244 GEMM launches of one step; profiles/gemm_tcgen05_*.md).  Valid
# only for the kernel source it was taken from: any change to the GEMM kernel
# reports null.
GEMM_TRAFFIC = {"source_sha256_16": "d673657982fa8dcb", "config": "1.2b", "bytes_per_launch": 270.65e6}


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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="1.2b")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--pin-store", type=int, default=1)
    ap.add_argument("--threads", type=int, default=0)
    ap.add_argument("--slabs", type=int, default=12)
    ap.add_argument("--keep-host-grad", type=int, default=1)
    ap.add_argument("--ckpt-on-host", type=int, default=1)
    ap.add_argument("--ckpt-interval", type=int, default=1, help="layers per recompute segment")
    ap.add_argument("--buffers", type=int, default=2, help="device weight buffers (1: single-buffer ablation)")
    ap.add_argument("--layers", type=int, default=0, help="decoder depth override (depth sweeps; 0 = the config's)")
    ap.add_argument("--trace", default="", help="write the stream timeline of one extra step (Chrome trace JSON)")
    ap.add_argument("--host-accum", type=int, default=0,
                    help="1: one pass per micro-batch, gradients summed in FP32 on the host")
    ap.add_argument("--set", action="append", default=[], metavar="KEY=VALUE",
                    help="override a shape field of the config (e.g. hidden=4096); repeatable")
    ap.add_argument("--timeout", type=float, default=0,
                    help="limit of every bounded host wait, seconds (0: four times the step's tensor work at "
                         "400 TFLOP/s, at least 60 s)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-e2e", action="store_true")
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

    over = {"n_layers": args.layers} if args.layers > 0 else {}
    for kv in args.set:
        key, _, val = kv.partition("=")
        over[key] = float(val) if "." in val or "e" in val.lower() else int(val)
    c = configs.get(args.config, **over)
    T = c["micro"] * c["batch"] * c["seq"]
    P, F_exec, F_pages = model_numbers(c, args.ckpt_interval)
    # every replica on this host holds its own host state: refuse to start
    # rather than exhaust host RAM
    local_world = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    need = local_world * host_bytes_needed(c, args.slabs, args.ckpt_on_host, args.ckpt_interval, args.host_accum)
    avail = mem_available_bytes()
    if avail and need > 0.85 * avail:
        msg = (f"{local_world} replica(s) of the {args.config} workload need {need / 1e9:.1f} GB of host RAM; "
               f"{avail / 1e9:.1f} GB available")
        if rank == 0:
            print(json.dumps({"metric": METRIC, "error": msg, "n_gpus": world}), flush=True)
        sys.exit(2)
    pk = peaks()
    bw = link_bandwidth(torch)

    t_init = time.time()
    hbw = mt.host_bandwidth(1 << 30)
    # every host wait of the library is bounded; a long-context step is minutes of GPU work
    timeout_s = args.timeout if args.timeout > 0 else max(60.0, 4.0 * F_exec / 4e14)
    m = mt.Model(c, seed=1234, pin_store=args.pin_store, n_host_threads=args.threads, n_grad_slabs=args.slabs,
                 timeout_ms=int(min(timeout_s * 1e3, 4.0e9)),
                 keep_host_grad=args.keep_host_grad, ckpt_on_host=args.ckpt_on_host,
                 ckpt_interval=args.ckpt_interval, n_buffers=args.buffers, host_grad_accum=args.host_accum)
    init_s = time.time() - t_init
    toks = [inputs.tokens_for(c, s) for s in range(args.warmup + 2 * args.steps + 1)]
    step = 0
    for w in range(args.warmup):
        m.set_tokens(toks[step])
        m.train_step(step)
        step += 1
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
    peak_t = pk.get("bf16_tflops_sustained", 1700.0)
    achieved = g["flops"] / (g["ms"] / 1e3) / 1e12 if g["ms"] > 0 else None
    roof = {"bound": "tensor", "kernel": "gemm_kernel (tcgen05 BF16 GEMM, all projections)",
            "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s",
            "frac": (achieved / peak_t) if achieved else None, "traffic": traffic,
            "peak_source": "bf16_tflops_sustained of " + ("fallback" if pk.get("fallback") else "measured"),
            "launches": g["launches"], "avg_launch_ms": g["ms"] / max(1, g["launches"]),
            "flops_per_launch": g["flops"] / max(1, g["launches"])}
    t_compute = F_exec / (peak_t * 1e12)
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
    # (12 B) + W (2 B) [+ G (2 B) when unpacking], and every DMA reads or writes host memory once
    n_pad = sum(b["n_pad"] for b in m.layout)
    adam_b = n_pad * (28 + 2 * args.keep_host_grad)
    dma_b = (st1["h2d_bytes"] - st0["h2d_bytes"] + st1["d2h_bytes"] - st0["d2h_bytes"]) / args.steps
    t_host = (adam_b + dma_b) / (hbw["copy_gbs"] * 1e9)
    cpu = None
    if not args.no_cpu and world == 1:
        try:
            cpu = cpu_sample(args.config)
        except Exception as e:  # the oracle is a reported baseline only
            cpu = {"value": None, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": f"failed: {e}"}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded uniform token ids, N(0,0.02) weights)",
        "config": {"workload": workload_desc(args.config, c), "model": args.config,
                   "global_batch": world * c["batch"] * c["micro"], "seq_len": c["seq"],
                   "tokens_per_step": T, "parallelism": f"replicas x{world} (no exchange step)",
                   "pin_store": args.pin_store, "n_grad_slabs": args.slabs, "keep_host_grad": args.keep_host_grad,
                   "ckpt_on_host": args.ckpt_on_host, "ckpt_interval": args.ckpt_interval,
                   "n_buffers": args.buffers, "host_grad_accum": args.host_accum,
                   "l2": "inputs larger than L2 (every step streams "
                   f"{2 * P / 1e9:.2f} GB of weights in and out)"},
        "step_roofline": {"frac": t_roof / t_step, "t_roof_ms": t_roof * 1e3, "t_step_ms": t_step * 1e3,
                          "bound": "tensor" if t_compute >= t_link else "host link",
                          "F_exec_pflop": F_exec / 1e15, "peak_tflops": peak_t,
                          "link_h2d_GBs": bw["h2d"] / 1e9, "link_d2h_GBs": bw["d2h"] / 1e9,
                          "link_both_GBs": bw["both"] / 1e9, "params": P,
                          "pages_tflops_convention": F_pages / t_step / 1e12,
                          "model_tflops_executed": F_exec / t_step / 1e12},
        "host_dram_bound": {"host_copy_GBs": hbw["copy_gbs"], "host_adam_Gelem_s": hbw["adam_gelem_s"],
                            "threads": hbw["threads"], "bytes_per_step_GB": (adam_b + dma_b) / 1e9,
                            "t_host_ms": t_host * 1e3, "frac": t_host / t_step,
                            "note": "host DRAM traffic of Adam + DMA over the measured 16-thread copy bandwidth; "
                                    "not part of the step roofline"},
        "roofline": roof,
        "kernels": kernels,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "host": {"adam_ms_per_step": (st1["adam_ms_total"] - st0["adam_ms_total"]) / args.steps,
                 "pack_ms_per_step": (st1["pack_ms_total"] - st0["pack_ms_total"]) / args.steps,
                 "h2d_GB_per_step": (st1["h2d_bytes"] - st0["h2d_bytes"]) / args.steps / 1e9,
                 "d2h_GB_per_step": (st1["d2h_bytes"] - st0["d2h_bytes"]) / args.steps / 1e9,
                 "device_bytes": m.device_bytes, "host_store_GB": st1["host_store_bytes"] / 1e9,
                 "pinned_GB": st1["pinned_bytes"] / 1e9, "init_s": init_s, "nproc": os.cpu_count(),
                 "cpu_model": cpu_model(),
                 "last_loss": losses[-1]},
    }
    line["schedule"] = static_schedule(m, vis_ms, bw, hbw, args.slabs)
    line["timeline"] = timeline(m, toks[step % len(toks)], step, args.trace)
    if c.get("n_experts"):
        # routed experts of the last forward: how many experts each layer's
        # stream-ins copied, and the load of the busiest expert over the mean
        cnt = np.stack([m.expert_counts(j) for j in range(1, c["n_layers"] + 1)])
        line["moe"] = {"n_experts": c["n_experts"], "top_k": c["top_k"],
                       "routed_experts_per_layer": [int(x) for x in (cnt > 0).sum(axis=1)],
                       "routed_frac": float((cnt > 0).mean()),
                       "max_over_mean_load": float((cnt.max(axis=1) / cnt.mean(axis=1)).mean())}
    print(json.dumps(line), flush=True)
    m.close()
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
