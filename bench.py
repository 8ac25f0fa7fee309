"""Benchmark of the KIVI quantized KV cache on GB300: one step = append one
new K/V token to every sequence + decode attention over the whole cache,
through the fused kivi_append_decode_attn call (--unfused: kivi_append then
kivi_decode_attn).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  `value` is the effective HBM throughput of the
step: the algorithmic bytes of append + decode (the bytes the method must
move, not what the kernels happen to move) divided by the CUDA-event time of
the K timed steps, summed over ranks.  Inputs are resident in HBM before the
timed region; the caches rotate over replicas whose total footprint is well
above the 129 MB L2, so every step streams from DRAM.

Multi-GPU: the workload is replicated per GPU (independent sequences need no
exchange); time is the max over ranks and `value` the sum of all ranks'
bytes over it ("scaling": "weak").
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-KV decode attn effective HBM GB/s & % of 8 TB/s; append tokens/s"
NOMINAL_HBM_GBS = 8000.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="mha7b")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--replicas", type=int, default=0, help="cache replicas (0 = enough for 4x L2)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--unfused", action="store_true", help="append and decode as two calls (two launches)")
    ap.add_argument("--prefill", type=int, default=0, metavar="M",
                    help="chunked prefill instead of decode: a step appends M tokens per sequence and runs "
                         "the causal attention of those M queries (kivi_append + kivi_prefill_attn)")
    ap.add_argument("--ragged", action="store_true",
                    help="ragged batch: decode with sequence b holding T - T*b/(2B) tokens; with --prefill, "
                         "sequence b takes a chunk of M - M*b/(2B) tokens (all lengths differ)")
    ap.add_argument("--repeats", type=int, default=5,
                    help="timed windows of exactly --steps steps each; the line reports the median window")
    ap.add_argument("--sweep", action="store_true",
                    help="every cell of the 32-layer decode-step sweep, one JSON line per cell")
    return ap.parse_args()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def workload(name):
    from kivi_quantized_kv_gb300.synth import WORKLOADS, sweep_workload
    if name in WORKLOADS:
        return WORKLOADS[name]
    if name.startswith("sweep_"):   # sweep_B<batch>_T<tokens>_b<bits>
        _, b, t, bits = name.split("_")
        return sweep_workload(int(b[1:]), int(t[1:]), int(bits[1:]))
    raise SystemExit(f"unknown workload {name}")


def workload_config(w, extra=None):
    cfg = {"workload": w.name, "batch": w.batch, "h_q": w.h_q, "h_kv": w.h_kv, "head_dim": w.head_dim,
           "tokens": w.tokens, "bits": w.bits, "group": w.group, "residual": w.residual, "sinks": w.sinks,
           "window": w.window, "layers": 1}
    if extra:
        cfg.update(extra)
    return cfg


# --------------------------------------------------------------- clocks
class ClockSampler:
    """SM clock and throttle reasons sampled while the timed region runs.

    Reads NVML (libnvidia-ml, the driver's management library) through ctypes
    every 2 ms from a thread, so that even a timed region of a few tens of
    milliseconds gets samples; falls back to `nvidia-smi -lms 200` when NVML
    cannot be loaded.  Only samples taken between mark_begin() and mark_end()
    count.  Nothing here changes a GPU setting."""

    # NVML clock-event reason bits (nvml.h: nvmlClocksEventReason*)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.device = device
        self.rows = []          # (t, sm_mhz, max_mhz, set of reasons)
        self.proc = None
        self.nvml = None
        self.running = False
        self.t_begin = self.t_end = None

    def _nvml_handle(self):
        import ctypes
        import torch
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return None
        if nv.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        idx = self.device.index if self.device.index is not None else 0
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(self.device).uuid)
            ok = nv.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(uuid.encode()), ctypes.byref(h)) == 0
        except Exception:
            ok = False
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(h)) != 0:
            return None
        self.index = idx
        return nv, h

    def start(self):
        self.nvml = self._nvml_handle()
        self.running = True
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._poll_nvml, daemon=True)
            self.thread.start()
            return
        try:
            idx = self.device.index if self.device.index is not None else 0
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(idx)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read_smi, daemon=True)
        self.thread.start()

    def _poll_nvml(self):
        import ctypes
        nv, h = self.nvml
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while self.running:
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                    nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and \
                    get_reasons(h, ctypes.byref(rs)) == 0:
                reasons = {n for bit, n in self.REASONS.items() if rs.value & bit}
                self.rows.append((time.perf_counter(), float(clk.value), float(mx.value), reasons))
            time.sleep(0.002)

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            r = [c.strip() for c in line.split(",")]
            try:
                reasons = {n for i, n in enumerate(names) if r[5 + i].lower().startswith("active")}
                self.rows.append((time.perf_counter(), float(r[1]), float(r[2]), reasons))
            except (ValueError, IndexError):
                continue

    def mark_begin(self):
        self.t_begin = time.perf_counter()

    def mark_end(self):
        self.t_end = time.perf_counter()

    def stop(self):
        self.running = False
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if getattr(self, "thread", None) is not None:
            self.thread.join(timeout=2)
        rows = [r for r in self.rows if self.t_begin is None or self.t_begin <= r[0] <= self.t_end]
        if not rows:
            return None
        reasons = set().union(*(r[3] for r in rows))
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": rows[-1][2],
                "reasons": sorted(reasons), "samples": len(rows),
                "source": "nvml 2 ms" if self.nvml is not None else "nvidia-smi 200 ms"}


# --------------------------------------------------------------- bytes
def append_bytes(w, L_before, L_after, n=1):
    """Algorithmic bytes of appending n tokens per sequence: read the new
    fp16 K/V, write them to the ring (or fp32 sinks), and for every group the
    append freezes read its G fp16 tokens and write its block."""
    units = w.batch * w.h_kv
    d = w.head_dim
    new_groups = L_after["n_groups"] - L_before["n_groups"]
    per_unit = n * 8 * d + new_groups * (4 * d * w.group + L_after["block_bytes"])
    return units * per_unit


def state_at(w, T):
    """(n_sink, n_groups, n_res) after T tokens, the lazy-flush rule the
    library uses (a token that reaches a full ring first freezes its oldest
    G tokens)."""
    n_sink = min(T, w.sinks)
    m = max(T - w.sinks, 0)
    ng = 0 if m <= w.residual else -(-(m - w.residual) // w.group)
    return n_sink, ng, m - ng * w.group


def decode_bytes_at(w, T, n_slots):
    """Algorithmic bytes of one decode after T tokens; the same sum as
    kivi_decode_bytes (checked against it in run_ours)."""
    n_sink, ng, n_res = state_at(w, T)
    first = max(ng - n_slots, 0)
    lo = T - w.window if w.window > 0 else 0
    if w.window > 0 and lo > w.sinks:
        first = max(first, (lo - w.sinks) // w.group)
    first = min(first, ng)
    tq = touched = 0
    for grp in range(first, ng):
        a0 = w.sinks + grp * w.group
        vis = a0 + w.group - max(a0, lo)
        if vis > 0:
            tq += vis
            touched += 1
    d = w.head_dim
    n_out = -(-getattr(w, "outlier_permille", 0) * w.group * d // 1000)   # outlier table entries
    tables = 2 * (2 * (w.group + 1) + 4 * n_out) if n_out else 0          # row pointers + entries, K and V
    per_unit = (2 * tq * d * w.bits // 8 + 4 * d * touched + 4 * tq + 4 * d * n_res + 8 * d * n_sink +
                tables * touched)
    return per_unit * w.batch * w.h_kv + 4 * d * w.batch * w.h_q


def prefill_bytes_at(w, T, m, n_slots):
    """Algorithmic bytes of one causal attention of the m newest tokens
    after T tokens: every token some query sees, counted as decode_bytes_at
    counts them (the oldest query's window reaches furthest back), plus q
    and out for m rows; the same sum as kivi_prefill_bytes."""
    n_sink, ng, n_res = state_at(w, T)
    first = max(ng - n_slots, 0)
    lo = T - m + 1 - w.window if w.window > 0 else 0
    if w.window > 0 and lo > w.sinks:
        first = max(first, (lo - w.sinks) // w.group)
    first = min(first, ng)
    tq = touched = 0
    for grp in range(first, ng):
        a0 = w.sinks + grp * w.group
        vis = a0 + w.group - max(a0, lo)
        if vis > 0:
            tq += vis
            touched += 1
    d = w.head_dim
    n_out = -(-getattr(w, "outlier_permille", 0) * w.group * d // 1000)   # outlier table entries
    tables = 2 * (2 * (w.group + 1) + 4 * n_out) if n_out else 0          # row pointers + entries, K and V
    per_unit = (2 * tq * d * w.bits // 8 + 4 * d * touched + 4 * tq + 4 * d * n_res + 8 * d * n_sink +
                tables * touched)
    return per_unit * w.batch * w.h_kv + 4 * d * w.batch * m * w.h_q


def prefill_flops_at(w, T, m, n_slots):
    """Algorithmic FLOPs of that attention: 4 d per (query row, visible
    token) (q·k and p·v, a multiply and an add each)."""
    _, ng, _ = state_at(w, T)
    first_pos = w.sinks + max(ng - n_slots, 0) * w.group if w.window > 0 else 0   # oldest resident non-sink
    pairs = 0
    for j in range(m):
        P = T - m + j
        start = max(w.sinks, first_pos, P + 1 - w.window) if w.window > 0 else w.sinks
        pairs += min(P + 1, w.sinks) + max(0, P - start + 1)
    return 4 * w.head_dim * pairs * w.batch * w.h_q


def append_bytes_at(w, T, block_bytes):
    """Algorithmic bytes of appending one token per sequence to T tokens."""
    new_groups = state_at(w, T + 1)[1] - state_at(w, T)[1]
    d = w.head_dim
    return w.batch * w.h_kv * (8 * d + new_groups * (4 * d * w.group + block_bytes))


# --------------------------------------------------------------- our arm
def across_ranks(ms, nbytes, world, device):
    """(max of the ranks' timed spans, sum of their bytes) over the process
    group: every rank runs its own replica of the workload (weak scaling; the
    path needs no exchange), so the job moved the sum of the bytes in the
    slowest rank's time."""
    if world == 1:
        return ms, nbytes
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    b = torch.tensor([float(nbytes)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(b, op=torch.distributed.ReduceOp.SUM)
    return float(t.item()), float(b.item())


def run_ours(args, rank, world, device):
    import torch
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig
    from kivi_quantized_kv_gb300.synth import KVStream, queries

    w = workload(args.workload)
    # W warm-up steps, R timed windows of K steps, then K steps timed one by
    # one for the decode kernel's own time
    total_steps = args.warmup + (args.repeats + 1) * args.steps
    cap_extra = total_steps + 64
    cfg = KiviConfig.from_workload(w)
    if w.window == 0:
        cfg = KiviConfig(**{**cfg.__dict__, "max_tokens": w.tokens + cap_extra})
    from kivi_quantized_kv_gb300 import cache_bytes
    per_cache = cache_bytes(cfg)
    l2 = 129 * 1024 * 1024
    # enough replicas for 4x L2, and for each sequence to grow by at most 64
    # tokens over the run
    n_rep = args.replicas or max(2, -(-4 * l2 // per_cache), -(-total_steps // 64))
    stream = torch.cuda.current_stream(device)

    caches = []
    for r in range(n_rep):
        # ragged: sequence b starts at T - 1 - T*b/(2B) tokens (every length
        # differs).  Replica r starts r*G/n_rep tokens shorter, so that the
        # steps whose token freezes a group (one in G per sequence) fall
        # evenly over any window of consecutive steps, as they do over a long
        # run, instead of all replicas freezing within the same few steps
        stagger = (r * w.group) // n_rep
        targets = [w.tokens - 1 - stagger - ((w.tokens * b) // (2 * w.batch) if args.ragged else 0)
                   for b in range(w.batch)]
        c = KiviCache(cfg, device=device)
        kv = KVStream(w.with_(seed=w.seed + 100 * r), device=device)
        t = [0] * w.batch
        while t != targets:
            n = [min(4096, targets[b] - t[b]) for b in range(w.batch)]
            k, v = kv.next(max(n))
            if args.ragged:
                c.append_ragged(k, v, n)
            else:
                c.append(k, v)
            t = [t[b] + n[b] for b in range(w.batch)]
        caches.append((c, kv))
    # per-step inputs, resident before the timed region
    new_kv = [caches[s % n_rep][1].next(1) for s in range(total_steps)]
    qs = [queries(w, step=s, device=device) for s in range(min(total_steps, 64))]
    out = torch.empty((w.batch, w.h_q, w.head_dim), dtype=torch.float16, device=device)
    torch.cuda.synchronize(device)

    fused = not args.unfused
    import ctypes
    from kivi_quantized_kv_gb300 import _abi
    L = _abi.lib()
    sp = ctypes.c_void_p(stream.cuda_stream)
    vp = ctypes.c_void_p
    for c, _ in caches:   # every call below goes straight through the C ABI; check the shapes once
        c._check_io(new_kv[0][0], (w.batch, w.h_kv, 1, w.head_dim), "k_new")
    # per-step C-ABI arguments, marshalled before the timed region
    args_of = []
    for s in range(total_steps):
        c = caches[s % n_rep][0]
        k, v = new_kv[s]
        args_of.append((c._h, vp(k.data_ptr()), vp(v.data_ptr()), vp(qs[s % len(qs)].data_ptr()),
                        vp(out.data_ptr())))

    def step(s):
        h, kp, vq, qp, op = args_of[s]
        if fused:   # one call: append + decode (a freezing group's flush is a launch of its own)
            st = L.kivi_append_decode_attn(h, kp, vq, qp, op, sp)
        else:
            st = L.kivi_append(h, kp, vq, 1, sp) or L.kivi_decode_attn(h, qp, op, sp)
        if st != 0:
            raise RuntimeError(_abi.status_string(st))

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize(device)
    T_before = [c.tokens_per_sequence() for c, _ in caches]   # tokens of each replica's sequences before the timed steps
    meta = [(c.layout()["n_slots"], c.layout()["block_bytes"]) for c, _ in caches]

    # per timed step (from the first one after the warm-up): its bytes, its
    # launches and whether its token freezes a group, from each replica's
    # token count at that step
    T_now = [list(t) for t in T_before]
    w1 = w.with_(batch=1)
    per_step = []
    for s in range(args.warmup, total_steps):
        r = s % n_rep
        n_slots, block_bytes = meta[r]
        # the library's runs (consecutive sequences of equal length): one run is
        # one decode launch (plus a flush launch when its token freezes a
        # group); several runs share one ragged launch per 64 runs (plus one
        # flush launch when any of them freezes a group)
        runs = [b for b in range(w.batch) if b == 0 or T_now[r][b] != T_now[r][b - 1]]
        freezes = [state_at(w, T_now[r][b0] + 1)[1] > state_at(w, T_now[r][b0])[1] for b0 in runs]
        if not fused:   # kivi_append, one launch pair (flush, write) per run, then the decode
            launches = sum(2 if f else 1 for f in freezes) + -(-len(runs) // 64)
        else:
            launches = sum(1 + (1 if any(freezes[i:i + 64]) else 0) for i in range(0, len(runs), 64))
        dec = app = 0
        for b in range(w.batch):
            app += append_bytes_at(w1, T_now[r][b], block_bytes)
            T_now[r][b] += 1
            dec += decode_bytes_at(w1, T_now[r][b], n_slots)
        per_step.append((dec, app, launches, any(freezes)))
    clocks = ClockSampler(device) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.05)
        clocks.mark_begin()
    # R windows of exactly K steps, each bracketed by a barrier and a device
    # synchronisation on both sides and timed by CUDA events on the stream
    windows = []
    s0 = args.warmup
    for rep in range(args.repeats):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)
        t0.record(stream)
        for i in range(args.steps):
            step(s0 + i)
        t1.record(stream)
        torch.cuda.synchronize(device)
        if world > 1:
            torch.distributed.barrier()
        ms = t0.elapsed_time(t1)
        steps_w = per_step[s0 - args.warmup:s0 - args.warmup + args.steps]
        dec_b = sum(x[0] for x in steps_w)
        app_b = sum(x[1] for x in steps_w)
        ms_max, all_bytes = across_ranks(ms, dec_b + app_b, world, device)
        windows.append({"ms": ms_max, "bytes": all_bytes, "dec_bytes": dec_b, "app_bytes": app_b,
                        "dec_ms": ms, "launches": sum(x[2] for x in steps_w),
                        "freezing_steps": sum(1 for x in steps_w if x[3])})
        s0 += args.steps
    if clocks:
        clocks.mark_end()
    clk = clocks.stop() if clocks else None
    # the median window (by throughput) is the line's value
    order = sorted(range(len(windows)), key=lambda i: windows[i]["bytes"] / windows[i]["ms"])
    med = windows[order[len(order) // 2]]
    value = med["bytes"] / (med["ms"] / 1e3) / 1e9

    # the decode kernel's own time: K more steps, each bracketed by events;
    # the steps that freeze no group are one decode launch each (the fused
    # step), so their mean duration is the decode kernel's launch time
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    torch.cuda.synchronize(device)
    for i in range(args.steps):
        ev[i].record(stream)
        step(s0 + i)
    ev[args.steps].record(stream)
    torch.cuda.synchronize(device)
    dur = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    for r, (c, _) in enumerate(caches):   # the byte count above is the library's own
        assert c.tokens_per_sequence() == T_now[r]
        assert c.decode_bytes() == sum(decode_bytes_at(w1, t, meta[r][0]) for t in T_now[r]), \
            "decode byte count mismatch"
    steps_k = per_step[s0 - args.warmup:s0 - args.warmup + args.steps]
    plain = [(d, x[0]) for d, x in zip(dur, steps_k) if not x[3]] or [(d, x[0]) for d, x in zip(dur, steps_k)]
    flush_steps = [d for d, x in zip(dur, steps_k) if x[3]]
    kern_ms = sum(d for d, _ in plain) / len(plain)
    kern_bytes = sum(b for _, b in plain) / len(plain)
    res = {
        "w": w, "cfg": cfg, "n_rep": n_rep, "per_cache": per_cache, "ms": med["ms"], "value": value,
        "dec_gbs": kern_bytes / (kern_ms / 1e3) / 1e9, "dec_ms": kern_ms, "dec_bytes": kern_bytes,
        "window_dec_gbs": med["dec_bytes"] / (med["dec_ms"] / 1e3) / 1e9,
        "flush_step_ms": (sum(flush_steps) / len(flush_steps)) if flush_steps else None,
        "fused": fused, "step_bytes": med["bytes"] / args.steps, "launches": med["launches"],
        "clocks": clk, "app_tok_s": w.batch * world * args.steps / (med["ms"] / 1e3),
        "windows": [{"ms": round(x["ms"], 4), "gbs": round(x["bytes"] / (x["ms"] / 1e3) / 1e9, 1),
                     "freezing_steps": x["freezing_steps"]} for x in windows],
        "kernel_steps": len(plain),
    }
    if not args.no_e2e and not args.ragged:
        res["e2e"] = run_e2e(args, caches, new_kv, w, device, stream)
    return res


def run_sweep_cell(args, device, w):
    """One cell of the 32-layer decode-step sweep: a step appends one token to
    every sequence of every layer and runs every layer's decode attention
    over its cache (one kivi_append_decode_attn per layer, the 32 layers in
    order).  Layer l's K/V stream is seeded 1000003*seed + l.  Small cells
    rotate over whole-model replicas until 4x the 129 MB L2 is covered; a
    cell whose caches do not fit the free device memory is reported as such,
    with its footprint from kivi_cache_bytes."""
    import ctypes
    import torch
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig, _abi, cache_bytes
    from kivi_quantized_kv_gb300.synth import KVStream, queries

    layers = w.layers
    total_steps = args.warmup + (args.repeats + 1) * args.steps
    cfg = KiviConfig(**{**KiviConfig.from_workload(w).__dict__, "max_tokens": w.tokens + total_steps + 64})
    per_layer = cache_bytes(cfg)
    model = per_layer * layers
    l2 = 129 * 1024 * 1024
    n_rep = max(1, -(-4 * l2 // model))
    free, _total = torch.cuda.mem_get_info(device)
    # the timed steps' inputs and the fill's staging chunks need room too
    inputs = total_steps * layers * 2 * w.batch * w.h_kv * w.head_dim * 2
    staging = 12 * w.batch * w.h_kv * 4096 * w.head_dim * 4
    need = n_rep * model + inputs + staging + (1 << 30)
    base_cfg = workload_config(w, {"layers": layers, "parallelism": "replicas1"})
    if need > free:
        return {"metric": METRIC, "workload": w.name, "does_not_fit": True,
                "footprint_bytes": int(model), "free_bytes": int(free),
                "note": "32 layers of kivi_cache_bytes exceed the free device memory", "config": base_cfg}
    stream = torch.cuda.current_stream(device)
    reps = []   # per replica: list of (cache, stream) per layer
    for r in range(n_rep):
        stagger = (r * w.group) // n_rep
        lay = []
        for l in range(layers):
            c = KiviCache(cfg, device=device)
            kv = KVStream(w.with_(seed=w.seed + 100 * r), layer=l, device=device)
            t = 0
            target = w.tokens - 1 - stagger
            while t < target:
                n = min(4096, target - t)
                k, v = kv.next(n)
                c.append(k, v)
                t += n
            lay.append((c, kv))
        reps.append(lay)
    torch.cuda.synchronize(device)
    # per step and layer: the new token and a query, resident before timing
    new_kv = [[reps[s % n_rep][l][1].next(1) for l in range(layers)] for s in range(total_steps)]
    qs = [[queries(w, step=s, layer=l, device=device) for l in range(layers)] for s in range(min(total_steps, 8))]
    outs = [torch.empty((w.batch, w.h_q, w.head_dim), dtype=torch.float16, device=device) for _ in range(layers)]
    torch.cuda.synchronize(device)
    L = _abi.lib()
    vp = ctypes.c_void_p
    sp = vp(stream.cuda_stream)
    args_of = [[(reps[s % n_rep][l][0]._h, vp(new_kv[s][l][0].data_ptr()), vp(new_kv[s][l][1].data_ptr()),
                 vp(qs[s % len(qs)][l].data_ptr()), vp(outs[l].data_ptr())) for l in range(layers)]
               for s in range(total_steps)]
    fn = L.kivi_append_decode_attn

    def step(s):
        for a in args_of[s]:
            st = fn(*a, sp)
            if st != 0:
                raise RuntimeError(_abi.status_string(st))

    T0 = [reps[r][0][0].tokens for r in range(n_rep)]
    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize(device)
    # bytes of every timed step (the same for every layer of a replica)
    T_now = [reps[r][0][0].tokens for r in range(n_rep)]
    n_slots, block_bytes = reps[0][0][0].layout()["n_slots"], reps[0][0][0].layout()["block_bytes"]
    w1 = w.with_(batch=1)
    per_step = []
    for s in range(args.warmup, total_steps):
        r = s % n_rep
        freeze = state_at(w, T_now[r] + 1)[1] > state_at(w, T_now[r])[1]
        app = append_bytes_at(w1, T_now[r], block_bytes) * w.batch
        T_now[r] += 1
        dec = decode_bytes_at(w1, T_now[r], n_slots) * w.batch
        per_step.append((dec * layers, app * layers, layers * (2 if freeze else 1), freeze, dec))
    clocks = ClockSampler(device)
    clocks.start()
    time.sleep(0.05)
    clocks.mark_begin()
    windows = []
    s0 = args.warmup
    for rep in range(args.repeats):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        t0.record(stream)
        for i in range(args.steps):
            step(s0 + i)
        t1.record(stream)
        torch.cuda.synchronize(device)
        st = per_step[s0 - args.warmup:s0 - args.warmup + args.steps]
        windows.append({"ms": t0.elapsed_time(t1), "bytes": sum(x[0] + x[1] for x in st),
                        "launches": sum(x[2] for x in st), "freezing_steps": sum(1 for x in st if x[3])})
        s0 += args.steps
    clocks.mark_end()
    clk = clocks.stop()
    order = sorted(range(len(windows)), key=lambda i: windows[i]["bytes"] / windows[i]["ms"])
    med = windows[order[len(order) // 2]]
    # the decode kernel's own launch time: K more steps, each layer's call
    # bracketed by events; calls whose token freezes no group are one launch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps * layers + 1)]
    torch.cuda.synchronize(device)
    j = 0
    for i in range(args.steps):
        for a in args_of[s0 + i]:
            ev[j].record(stream)
            st = fn(*a, sp)
            if st != 0:
                raise RuntimeError(_abi.status_string(st))
            j += 1
    ev[j].record(stream)
    torch.cuda.synchronize(device)
    st_k = per_step[s0 - args.warmup:s0 - args.warmup + args.steps]
    plain = [ev[i * layers + l].elapsed_time(ev[i * layers + l + 1]) for i in range(args.steps) if not st_k[i][3]
             for l in range(layers)]
    plain_bytes = [st_k[i][4] for i in range(args.steps) if not st_k[i][3]]
    for r in range(n_rep):
        for c, _ in reps[r]:
            assert c.read_error() == 0
            assert c.tokens == T0[r] + sum(1 for s in range(total_steps) if s % n_rep == r)
    peaks, src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    kern_ms = sum(plain) / len(plain) if plain else None
    kern_bytes = sum(plain_bytes) / len(plain_bytes) if plain_bytes else None
    step_ms = med["ms"] / args.steps
    value = med["bytes"] / (med["ms"] / 1e3) / 1e9
    achieved = kern_bytes / (kern_ms / 1e3) / 1e9 if kern_ms else None
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16xf16->f32", "data": "synthetic",
        "config": {**base_cfg, "l2": f"{n_rep} rotating replicas of the 32-layer caches x {model / 1e6:.0f} MB"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1) if achieved else None, "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4) if achieved else None, "traffic": None,
                     "kernel": "decode_mma_kernel (one launch per layer)", "peak_source": src,
                     "bytes_per_launch": int(kern_bytes) if kern_bytes else None},
        "gpu_launches": med["launches"], "clocks": clk, "repeats": args.repeats,
        "windows": [{"ms": round(x["ms"], 4), "gbs": round(x["bytes"] / (x["ms"] / 1e3) / 1e9, 1),
                     "freezing_steps": x["freezing_steps"]} for x in windows],
        "bytes_per_step": int(med["bytes"] / args.steps),
        "decode_steps_per_s": round(1e3 / step_ms, 2),
        "tokens_per_s": round(w.batch * 1e3 / step_ms, 1),
        "tokens_per_s_kind": "sequence tokens decoded per second (each appended to all 32 layers)",
        "decode_us_per_layer": round(kern_ms * 1e3, 2) if kern_ms else None,
        "footprint_bytes": int(model),
    }


def sweep_cells():
    from kivi_quantized_kv_gb300.synth import SWEEP_BATCH, SWEEP_BITS, SWEEP_TOKENS, sweep_workload
    return [sweep_workload(b, t, bits) for b in SWEEP_BATCH for t in SWEEP_TOKENS for bits in SWEEP_BITS]


def run_prefill(args, device):
    """Chunked prefill: a step appends an M-token chunk to every sequence
    (kivi_append) and runs the causal attention of the chunk's M queries over
    the packed cache (kivi_prefill_attn).  The replicas start M tokens short
    of the workload's length, so the first chunk on each ends at it; later
    chunks grow it (the byte and FLOP counts follow each replica's length).
    The attention launches are timed on their own with CUDA events around
    each call on the launching stream."""
    import ctypes
    import torch
    from kivi_quantized_kv_gb300 import KiviCache, KiviConfig, _abi, cache_bytes
    from kivi_quantized_kv_gb300.synth import KVStream

    w = workload(args.workload)
    m = args.prefill
    counts = [m - (m * b) // (2 * w.batch) for b in range(w.batch)] if args.ragged else [m] * w.batch
    w1 = w.with_(batch=1)
    total_steps = args.steps + args.warmup
    l2 = 129 * 1024 * 1024
    cfg0 = KiviConfig.from_workload(w)
    n_rep = args.replicas or max(2, -(-4 * l2 // cache_bytes(cfg0)))
    per_rep = -(-total_steps // n_rep)
    cfg = cfg0 if w.window else KiviConfig(**{**cfg0.__dict__, "max_tokens": w.tokens + per_rep * m})
    per_cache = cache_bytes(cfg)
    stream = torch.cuda.current_stream(device)
    caches = []
    for r in range(n_rep):
        c = KiviCache(cfg, device=device)
        kv = KVStream(w.with_(seed=w.seed + 100 * r), device=device)
        t = 0
        while t < w.tokens - m:
            n = min(4096, w.tokens - m - t)
            k, v = kv.next(n)
            c.append(k, v)
            t += n
        caches.append((c, kv))
    chunks = [caches[s % n_rep][1].next(m) for s in range(total_steps)]
    g = torch.Generator(device=device).manual_seed(w.seed + 4242)
    qs = [torch.randn((w.batch, m, w.h_q, w.head_dim), generator=g, device=device).half() for _ in range(4)]
    out = torch.empty_like(qs[0])
    need = caches[0][0].prefill_scratch_bytes(m)
    scratch = torch.empty(need, dtype=torch.uint8, device=device)
    torch.cuda.synchronize(device)
    L = _abi.lib()
    vp = ctypes.c_void_p
    sp = vp(stream.cuda_stream)
    args_of = [(caches[s % n_rep][0]._h, vp(chunks[s][0].data_ptr()), vp(chunks[s][1].data_ptr()),
                vp(qs[s % len(qs)].data_ptr())) for s in range(total_steps)]
    counts_arr = (ctypes.c_int64 * w.batch)(*counts)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]

    def step(s, e=None):
        h, kp, vq, qp = args_of[s]
        if args.ragged:
            st = L.kivi_append_ragged(h, kp, vq, counts_arr, m, sp)
        else:
            st = L.kivi_append(h, kp, vq, m, sp)
        if e is not None:
            e[0].record(stream)
        if args.ragged:
            st = st or L.kivi_prefill_attn_ragged(h, qp, vp(out.data_ptr()), counts_arr, m, vp(scratch.data_ptr()),
                                                  need, sp)
        else:
            st = st or L.kivi_prefill_attn(h, qp, vp(out.data_ptr()), m, vp(scratch.data_ptr()), need, sp)
        if e is not None:
            e[1].record(stream)
        if st != 0:
            raise RuntimeError(_abi.status_string(st))

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize(device)
    T_now = [c.tokens_per_sequence() for c, _ in caches]
    meta = [(c.layout()["n_slots"], c.layout()["block_bytes"]) for c, _ in caches]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(device)
    clocks.start()
    time.sleep(0.05)
    clocks.mark_begin()
    t0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i, ev[i])
    t1.record(stream)
    torch.cuda.synchronize(device)
    clocks.mark_end()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    attn_ms = sum(a.elapsed_time(b) for a, b in ev)
    attn_bytes = attn_flops = launches = 0
    for i in range(args.steps):
        r = (args.warmup + i) % n_rep
        T0 = list(T_now[r])
        runs = []   # the library's runs: consecutive sequences of equal (length, count)
        for b in range(w.batch):
            if runs and runs[-1][1] == (T0[b], counts[b]):
                runs[-1][0].append(b)
            else:
                runs.append(([b], (T0[b], counts[b])))
        for seqs, (t0, n) in runs:
            launches += 2 + (1 if state_at(w, t0 + n)[1] > state_at(w, t0)[1] else 0)   # write, prefill, flush
        for b in range(w.batch):
            T_now[r][b] += counts[b]
            attn_bytes += prefill_bytes_at(w1, T_now[r][b], counts[b], meta[r][0])
            attn_flops += prefill_flops_at(w1, T_now[r][b], counts[b], meta[r][0])
    for r, (c, _) in enumerate(caches):   # the byte count above is the library's own
        assert c.tokens_per_sequence() == T_now[r]
        if not args.ragged:
            assert c.prefill_bytes(m) == prefill_bytes_at(w, T_now[r][0], m, meta[r][0]), "prefill byte count mismatch"
        assert c.read_error() == 0
    peaks, src = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    tensor = float(peaks.get("bf16_tflops", 1900.0))
    gbs = attn_bytes / (attn_ms / 1e3) / 1e9
    tflops = attn_flops / (attn_ms / 1e3) / 1e12
    # the roofline the attention launch is bound by: the larger of its
    # memory time and its tensor time at the measured peaks
    t_mem = attn_bytes / (hbm * 1e9)
    t_math = attn_flops / (tensor * 1e12)
    if t_mem >= t_math:
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4)}
    else:
        roof = {"bound": "tensor", "achieved": round(tflops, 2), "peak": tensor, "unit": "TFLOP/s",
                "frac": round(tflops / tensor, 4)}
    roof.update({"traffic": None, "peak_source": src, "kernel": "decode_mma_kernel (several query tokens, causal masks)",
                 "bytes_per_launch": int(attn_bytes / args.steps), "flops_per_launch": int(attn_flops / args.steps),
                 "hbm_frac": round(gbs / hbm, 4), "tensor_frac": round(tflops / tensor, 5)})
    tok = sum(counts) * args.steps
    return {
        "metric": (f"chunked prefill query tokens/s (append {'up to ' if args.ragged else ''}{m} tokens per sequence "
                   f"+ their causal attention over the packed cache)"),
        "value": round(tok / (ms / 1e3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16xf16->f32", "data": "synthetic",
        "config": workload_config(w, {"chunk": m, "chunks_per_sequence": counts if args.ragged else m,
                                      "parallelism": "replicas1",
                                      "l2": f"{n_rep} rotating cache replicas x {per_cache / 1e6:.0f} MB (> 4x 129 MB L2)",
                                      "tokens_at_first_chunk": w.tokens}),
        "roofline": roof, "gpu_launches": launches, "clocks": clk,
        "attn_us": round(attn_ms * 1e3 / args.steps, 2), "attn_gbs": round(gbs, 1), "attn_tflops": round(tflops, 2),
        "step_call": ("kivi_append_ragged + kivi_prefill_attn_ragged" if args.ragged
                      else "kivi_append + kivi_prefill_attn"),
    }


def run_e2e(args, caches, new_kv, w, device, stream):
    """The same step through the public API with host buffers: one
    kivi_append_decode_attn_host call per step (kivi_append on a device copy
    + kivi_decode_attn_host with --unfused).  The step's K/V and q sit in
    pinned host memory and the output goes back to pinned host memory: the
    step reads the inputs over the host mapping and its merge writes the
    output there, every step, inside the timed region."""
    import ctypes
    import torch
    from kivi_quantized_kv_gb300 import _abi
    L = _abi.lib()
    n_rep = len(caches)
    steps = min(args.steps, 200)
    g = torch.Generator().manual_seed(7)
    k_h = [torch.randn((w.batch, w.h_kv, 1, w.head_dim), generator=g).half().pin_memory() for _ in range(steps)]
    v_h = [torch.randn((w.batch, w.h_kv, 1, w.head_dim), generator=g).half().pin_memory() for _ in range(steps)]
    q_h = torch.randn((w.batch, w.h_q, w.head_dim), generator=g).half().pin_memory()
    out_h = torch.empty_like(q_h).pin_memory()
    k_d = torch.empty((w.batch, w.h_kv, 1, w.head_dim), dtype=torch.float16, device=device)
    v_d = torch.empty_like(k_d)
    vp = ctypes.c_void_p
    sp = vp(stream.cuda_stream)
    T_before = [c.tokens for c, _ in caches]
    meta = [(c.layout()["n_slots"], c.layout()["block_bytes"]) for c, _ in caches]
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(steps):
        h = caches[s % n_rep][0]._h
        if args.unfused:
            k_d.copy_(k_h[s], non_blocking=True)
            v_d.copy_(v_h[s], non_blocking=True)
            st = L.kivi_append(h, vp(k_d.data_ptr()), vp(v_d.data_ptr()), 1, sp) or \
                L.kivi_decode_attn_host(h, vp(q_h.data_ptr()), vp(out_h.data_ptr()), sp)
        else:
            st = L.kivi_append_decode_attn_host(h, vp(k_h[s].data_ptr()), vp(v_h[s].data_ptr()),
                                                vp(q_h.data_ptr()), vp(out_h.data_ptr()), sp)
        if st != 0:
            raise RuntimeError(_abi.status_string(st))
    t1.record(stream)
    torch.cuda.synchronize(device)
    ms = t0.elapsed_time(t1)
    total = 0
    T_now = list(T_before)
    for s in range(steps):
        r = s % n_rep
        total += append_bytes_at(w, T_now[r], meta[r][1])
        T_now[r] += 1
        total += decode_bytes_at(w, T_now[r], meta[r][0])
    h2d = (2 * w.batch * w.h_kv + w.batch * w.h_q) * w.head_dim * 2
    d2h = w.batch * w.h_q * w.head_dim * 2
    return {"value": round(total / (ms / 1e3) / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "transfer": "the step reads the pinned host inputs and writes the output to pinned host memory over the host mapping"}


# --------------------------------------------------------------- oracle arm
def oracle_sample(w, units_max, seed=0, extra=4096):
    """An oracle cache holding a bounded sample of the workload: the first
    `units` (sequence, kv head) units, built from the same generator."""
    import numpy as np
    import oracle
    from kivi_quantized_kv_gb300.synth import KVStream
    rep = w.h_q // w.h_kv
    units = min(units_max, w.batch * w.h_kv)
    hk = min(units, w.h_kv)
    bs = max(1, units // hk)
    ws = w.with_(batch=bs, h_kv=hk, h_q=hk * rep)
    p = oracle.Params(bits=w.bits, group=w.group, residual=w.residual, sinks=w.sinks, h_q=ws.h_q, h_kv=ws.h_kv,
                      head_dim=w.head_dim, batch=ws.batch, max_tokens=0 if w.window else w.tokens + extra,
                      window=w.window, outlier_permille=w.outlier_permille, rope_base=w.rope_base)
    c = oracle.Cache(p)
    kv = KVStream(ws, device="cpu")
    t = 0
    while t < w.tokens - 1:
        n = min(4096, w.tokens - 1 - t)
        k, v = kv.next(n)
        c.append(k.numpy(), v.numpy())
        t += n
    return c, ws, kv


def time_oracle(w, budget_s=12.0, units_max=None, steps_exact=None, warmup=0):
    """The oracle on the host cores over a bounded sample of the workload:
    steps of (append one token + fp64 decode).  With steps_exact, `warmup`
    untimed steps then exactly that many timed ones; else timed steps until
    about budget_s seconds (at most 50)."""
    import numpy as np
    import torch
    from kivi_quantized_kv_gb300.synth import queries
    cores = os.cpu_count() or 1
    units_max = units_max or max(cores * 2, 8)
    t_build = time.perf_counter()
    c, ws, kv = oracle_sample(w, units_max, extra=max(4096, (steps_exact or 50) + warmup + 64))
    t_build = time.perf_counter() - t_build
    q = queries(ws).numpy()
    for _ in range(warmup if steps_exact else 0):
        k, v = kv.next(1)
        c.append(k.numpy(), v.numpy())
        c.decode_attn(q, threads=cores)
    steps = 0
    total = 0
    tt = 0.0
    while (steps < steps_exact) if steps_exact else (tt < budget_s and steps < 50):
        k, v = kv.next(1)
        t0 = time.perf_counter()
        c.append(k.numpy(), v.numpy())
        c.decode_attn(q, threads=cores)
        tt += time.perf_counter() - t0
        total += c.decode_bytes() + ws.batch * ws.h_kv * 8 * w.head_dim
        steps += 1
    return {"value": round(total / tt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{ws.batch * ws.h_kv} of {w.batch * w.h_kv} (sequence, kv-head) units of {w.name}, "
                      f"{steps} steps (append 1 token + fp64 decode), {cores} threads, build {t_build:.1f}s excluded",
            "steps": steps, "seconds": round(tt, 2)}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = workload(args.workload)

    if args.impl == "reference":
        if rank != 0:
            return
        base = time_oracle(w, steps_exact=args.steps, warmup=args.warmup)
        line = {"metric": METRIC, "value": base["value"], "unit": "GB/s", "n_gpus": args.gpus, "steps": base["steps"],
                "warmup": args.warmup, "ms_per_step": round(base["seconds"] * 1e3 / max(base["steps"], 1), 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "impl": "reference", "config": workload_config(w),
                "cpu_baseline": {k: base[k] for k in ("value", "unit", "cores", "kind", "sample")},
                "e2e": {"value": base["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import __graft_entry__ as ge
    ge.build()

    if args.prefill > 0:
        if world > 1:
            raise SystemExit("--prefill runs on one GPU")
        print(json.dumps(run_prefill(args, device)), flush=True)
        return
    if args.sweep or w.layers > 1:
        if world > 1:
            raise SystemExit("the sweep runs on one GPU")
        for cell in (sweep_cells() if args.sweep else [w]):
            print(json.dumps(run_sweep_cell(args, device, cell)), flush=True)
            torch.cuda.empty_cache()
        return
    r = run_ours(args, rank, world, device)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    peaks, src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    traffic = load_traffic(w.name)
    line = {
        "metric": METRIC, "value": round(r["value"], 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(r["ms"] / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16xf16->f32", "data": "synthetic",
        "config": workload_config(w, {"parallelism": f"replicas{world}",
                                      "l2": f"{r['n_rep']} rotating cache replicas x {r['per_cache'] / 1e6:.0f} MB "
                                            f"(> 4x 129 MB L2)",
                                      "appended_per_sequence": -(-(args.warmup + (args.repeats + 1) * args.steps) //
                                                                 r["n_rep"]),
                                      "replica_stagger": "replica r starts r*G/replicas tokens short of T - 1",
                                      "ragged": bool(args.ragged)}),
        "roofline": {"bound": "hbm", "achieved": round(r["dec_gbs"], 1), "peak": peak, "unit": "GB/s",
                     "frac": round(r["dec_gbs"] / peak, 4), "traffic": traffic,
                     "kernel": "decode_mma_kernel (stream-K split-K, merge and fresh-token append in the same launch)",
                     "peak_source": src,
                     "bytes_per_launch": int(r["dec_bytes"])},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "repeats": args.repeats,
        "windows": r["windows"],
        "decode_gbs": round(r["dec_gbs"], 1),
        "decode_frac_of_8tbs": round(r["dec_gbs"] / NOMINAL_HBM_GBS, 4),
        "decode_us": round(r["dec_ms"] * 1e3, 2),
        "decode_us_kind": (f"mean CUDA-event time of the {r['kernel_steps']} of {args.steps} steps (timed one by "
                           f"one after the windows) whose token freezes no group: one decode launch each"),
        "flush_step_us": round(r["flush_step_ms"] * 1e3, 2) if r["flush_step_ms"] else None,
        "window_decode_gbs": round(r["window_dec_gbs"], 1),
        "decode_steps_per_s": round(1e3 / r["dec_ms"], 1),
        "step_call": "kivi_append_decode_attn" if r["fused"] else "kivi_append + kivi_decode_attn",
        "append_tokens_per_s": round(r["app_tok_s"], 1),
        "append_tokens_per_s_kind": "tokens appended per second by the whole step (append + decode)",
    }
    if "e2e" in r:
        line["e2e"] = r["e2e"]
    if not args.no_cpu_baseline:
        base = time_oracle(w)
        line["cpu_baseline"] = {k: base[k] for k in ("value", "unit", "cores", "kind", "sample")}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def decode_sources():
    """The decode kernels' sources: the shared internal header, the rotation
    table and every decode* file, in name order."""
    csrc = os.path.join(ROOT, "kivi_quantized_kv_gb300", "csrc")
    return ["kivi_internal.cuh", "rope.cu"] + sorted(f for f in os.listdir(csrc) if f.startswith("decode"))


def decode_sources_sha():
    """sha256 over the decode kernel's sources, in a fixed order."""
    import hashlib
    h = hashlib.sha256()
    for n in decode_sources():
        with open(os.path.join(ROOT, "kivi_quantized_kv_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def load_traffic(name):
    """DRAM bytes (read + write) per decode launch from the committed ncu
    summary profiles/traffic.json, or None when that capture does not cover
    this workload or was taken on other decode sources than the ones built."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        if t.get("decode_sources_sha256") != decode_sources_sha():
            return None
        e = t["workloads"][name]
        return int(e["dram_bytes_read"] + e["dram_bytes_write"])
    except Exception:
        return None


if __name__ == "__main__":
    main()
