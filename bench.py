"""Benchmark: the Q4_K decode-layer mat-vec set of an 8B-shaped model, batch 1.

One step = the four batch-1 GEMVs of one transformer layer with hidden 4096,
32 query / 8 key-value heads of 128 and a 14336-wide MLP:
  QKV 4096 -> 6144, O 4096 -> 4096, fused gate+up 4096 -> 28672, down 14336 -> 4096,
122,683,392 bytes of Q4_K weights.  The weights of L distinct layers (20 by
default, 2.45 GB, 19 times the 129 MB L2) stay resident in HBM and step s
uses layer s mod L, so each step's weights were evicted from L2 by the L-1
layers in between (inputs larger than L2; no flush needed).  A rotation of
only a few times the L2 leaves part of the weights in it from one pass to
the next: with 0.43 GB of 14336x4096 copies the DRAM reads were 0.88 of the
weight bytes (ncu over the whole CUDA graph), with 1.3 GB and more 1.00 --
so every rotation here spans at least ten times the L2.

metric: effective weight GB/s = weight bytes / time; also microseconds per set.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (dequantize, then f64 dot) on the
host's cores on a bounded sample of the same workload.  Under torchrun each
rank runs the same per-GPU workload (replicas, weak scaling); rank 0 prints
one JSON line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import shutil
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

HIDDEN, N_Q, N_KV, HEAD, FFN = 4096, 32, 8, 128, 14336
SET = [  # (name, n_out, k)
    ("qkv", (N_Q + 2 * N_KV) * HEAD, HIDDEN),
    ("o", HIDDEN, N_Q * HEAD),
    ("gate_up", 2 * FFN, HIDDEN),
    ("down", HIDDEN, FFN),
]
FMT = "q4_k"
DOMINANT = "gate_up"
METRIC = "Q4_K GEMV effective weight GB/s (decode-layer set, batch 1)"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, nominal

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant
# kernel from one ncu capture, keyed by the sha256 of the kernel source it was
# taken on (the code up to the kernel's namespace end, comments removed); any
# edit of that code makes the figure stale (reported as null).
NCU_TRAFFIC = {"7217d3a290f0653e": 66_158_080}
# The same launch under ncu, cold and alone (gpu__time_duration.sum in us,
# dram__throughput.avg.pct_of_peak_sustained_elapsed), from the same capture.
NCU_ISOLATED = {"7217d3a290f0653e": {"us": 18.24, "dram_throughput_pct": 45.90}}


def set_bytes():
    return sum(synth.weight_bytes(FMT, n, k) for _, n, k in SET)


def kernel_source_hash():
    """sha256 prefix of the dominant kernel's source (gemv_stream.cu up to the
    end of the whole-row kernel's namespace: its helpers and the kernel) with
    comments and blank space removed (an edit of a comment, or of the kernels
    after it, leaves the captured figure valid)."""
    p = os.path.join(ROOT, "quantized_weight_mat_gb300", "csrc", "gemv_stream.cu")
    with open(p, encoding="utf-8") as f:
        src = f.read()
    end = src.find("}  // namespace rowk")
    if end > 0:
        src = src[:end]
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    src = "\n".join(line.strip() for line in src.splitlines() if line.strip())
    return hashlib.sha256(src.encode()).hexdigest()[:16]


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm_gb_s"):
            if key in d and d[key]:
                return float(d[key]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons in the background."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.rows, self.proc = index, [], None
        self.t_on = self.t_off = None

    def start(self):
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        self.proc = subprocess.Popen([exe, f"--id={self.index}", f"--query-gpu={self.Q}",
                                      "--format=csv,noheader,nounits", "-lms", "100"],
                                     stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.monotonic(), [c.strip() for c in line.split(",")]))

    def mark_on(self):
        self.t_on = time.monotonic()

    def mark_off(self):
        self.t_off = time.monotonic()

    def stop(self):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        inside = [r for t, r in self.rows if self.t_on and self.t_on <= t <= self.t_off + 0.15]
        window = "timed"
        if not inside:
            inside, window = [r for _, r in self.rows], "run"
        sm = [float(r[1]) for r in inside if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "window": window}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, world, device=None):
    """Each value's maximum over all ranks (one all-reduce; the identity on
    one rank).  Times are taken as the slowest rank's."""
    if world == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(bytes_per_step, steps, world, ms):
    """Whole-job throughput in GB/s: every rank processed `steps` steps of
    `bytes_per_step` in `ms` milliseconds (the slowest rank's time)."""
    return bytes_per_step * steps * world / (ms * 1e-3) / 1e9


# The workloads of the method, each timed alone (config name, fmt, n_out, k, batch).
CONFIGS = [
    ("Q8_0 896x896, batch 1", "q8_0", 896, 896, 1),
    ("Q4_K 4096x4096, batch 1", "q4_k", 4096, 4096, 1),
    ("Q6_K LM head 128256x4096, batch 1", "q6_k", 128256, 4096, 1),
] + [(f"Q4_K {n}x{k}, batch {b}", "q4_k", n, k, b)
     for (n, k) in ((14336, 4096), (4096, 14336)) for b in (1, 2, 4, 8, 16)
] + [(f"Q6_K LM head 128256x4096, batch {b}", "q6_k", 128256, 4096, b) for b in (2, 4, 8)
] + [("Q8_0 4096x4096, batch 1", "q8_0", 4096, 4096, 1),
     ("Q8_0 14336x4096, batch 1", "q8_0", 14336, 4096, 1),
     ("I8_ROW 14336x4096, batch 1", "i8_row", 14336, 4096, 1),
     ("I8_ROW 4096x4096, batch 1", "i8_row", 4096, 4096, 1),
] + [(f"{f.upper()} 14336x4096, batch 1", f, 14336, 4096, 1)
     for f in ("q5_k", "q3_k", "q2_k", "i4_row")
] + [("Q4_K QKV 6144x4096 with bias, batch 1", "q4_k", 6144, 4096, 1, "bias"),
     ("Q4_K gate+up 28672x4096 with SwiGLU, batch 1", "q4_k", 28672, 4096, 1, "swiglu"),
     ("Q4_K gate+up 28672x4096 with SwiGLU, batch 8", "q4_k", 28672, 4096, 8, "swiglu"),
     ("Q4_K gate+up 28672x4096, batch 8", "q4_k", 28672, 4096, 8),
     ("Q4_K 14336x4096, batch 32 (prompt width)", "q4_k", 14336, 4096, 32),
     ("Q4_K 4096x14336, batch 32 (prompt width)", "q4_k", 4096, 14336, 32)]


def per_config(pq, dev, peak, l2_bytes):
    """Each workload alone: pq_gemv launched back to back in a CUDA graph, the
    weights rotating over copies that together exceed ten times the L2 (no
    weight bytes left in L2 from the previous pass), CUDA events around one
    replay.  Returns one record per workload."""
    import torch
    out = []
    for name, fmt, n, k, b, *epi in CONFIGS:
        epi = epi[0] if epi else None
        nbytes = synth.weight_bytes(fmt, n, k)
        copies = max(2, -(-10 * l2_bytes // nbytes))
        base = torch.from_numpy(synth.random_records(fmt, n, k, seed=11)).to(dev)
        W = [base] + [base.clone() for _ in range(copies - 1)]
        x = torch.from_numpy(synth.normal_x(b, k, seed=12)).to(dev)
        y = torch.empty(b * n, dtype=torch.float32, device=dev)
        bias = torch.zeros(n, dtype=torch.float32, device=dev)
        # enough launches that the graph's own start-up is spread thin (a
        # decode step issues hundreds of these calls back to back)
        launches = 400 if nbytes < 4_000_000 else 200

        def call(i, stream=None):
            if epi == "bias":
                pq.pq_gemv_bias(fmt, W[i % copies], n, k, x, b, bias, y, stream)
            elif epi == "swiglu":
                pq.pq_gemv_swiglu(fmt, W[i % copies], n // 2, k, x, b, y, stream)
            else:
                pq.pq_gemv(fmt, W[i % copies], n, k, x, b, y, stream)

        for i in range(3):
            call(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cur = torch.cuda.current_stream()
            for i in range(launches):
                call(i, cur)
        g.replay()
        torch.cuda.synchronize()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        e.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(e) * 1e3 / launches
        gbs = nbytes / (us * 1e-6) / 1e9
        out.append({"workload": name, "kernel": int(pq.pq_gemv_choice(fmt, n, k, b)), "us": round(us, 3),
                    "weight_GBs": round(gbs, 1), "hbm_frac": round(gbs / peak, 4)})
        del W, base, g
        torch.cuda.empty_cache()
    # one labelled L2-warm figure: the 4096 -> 14336 batch-1 GEMV on a single
    # weight buffer (33 MB, resident in the 129 MB L2 after the first call)
    n, k = 14336, 4096
    w1 = torch.from_numpy(synth.random_records("q4_k", n, k, seed=11)).to(dev)
    x = torch.from_numpy(synth.normal_x(1, k, seed=12)).to(dev)
    y = torch.empty(n, dtype=torch.float32, device=dev)
    for _ in range(3):
        pq.pq_gemv("q4_k", w1, n, k, x, 1, y)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cur = torch.cuda.current_stream()
        for _ in range(200):
            pq.pq_gemv("q4_k", w1, n, k, x, 1, y, cur)
    g.replay()
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    e.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(e) * 1e3 / 200
    out.append({"workload": "Q4_K 14336x4096, batch 1, L2-WARM (one weight buffer, not an HBM figure)",
                "kernel": int(pq.pq_gemv_choice("q4_k", n, k, 1)), "us": round(us, 3),
                "weight_GBs": round(synth.weight_bytes("q4_k", n, k) / (us * 1e-6) / 1e9, 1), "hbm_frac": None})
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist
    from quantized_weight_mat_gb300 import build
    import quantized_weight_mat_gb300 as pq

    world, rank, local = dist_init()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    # decode weights are loaded once and only read: let each GEMV start
    # streaming its weights while the previous kernel finishes
    pq.pq_set_weight_prefetch(True)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    L = args.layers

    # resident weights of L layers; x and y per GEMV
    W = []
    for layer in range(L):
        W.append([torch.from_numpy(synth.random_records(FMT, n, k, seed=1000 * layer + j)).to(dev)
                  for j, (_, n, k) in enumerate(SET)])
    # x and y of the four GEMVs live in one device buffer each (views), so an
    # end-to-end step moves its inputs in and its outputs out with one copy each;
    # two such buffers (steps alternate) let the copies of one step overlap the
    # GEMVs of its neighbours
    xs = [synth.normal_x(1, k, seed=7 + j).ravel() for j, (_, n, k) in enumerate(SET)]
    x_off = np.cumsum([0] + [x.size for x in xs])
    y_off = np.cumsum([0] + [n for _, n, _ in SET])
    XA = [torch.from_numpy(np.concatenate(xs)).to(dev) for _ in range(2)]
    YA = [torch.empty(int(y_off[-1]), dtype=torch.float32, device=dev) for _ in range(2)]
    XB = [[xa[int(x_off[j]):int(x_off[j + 1])] for j in range(len(SET))] for xa in XA]
    YB = [[ya[int(y_off[j]):int(y_off[j + 1])] for j in range(len(SET))] for ya in YA]
    Xall, Yall, X, Y = XA[0], YA[0], XB[0], YB[0]
    launches_per_step = sum(pq.pq_gemv_launches(FMT, n, k, 1) for _, n, k in SET)
    dom = [name for name, _, _ in SET].index(DOMINANT)
    torch.cuda.synchronize()

    # one step = the four GEMVs of layer s mod L.  e2e: the step's x is copied
    # in from pinned host memory and its y copied back; step s uses buffer s % 2,
    # its input copy runs on one side stream while step s - 1 computes, its
    # output copy on another while step s + 1 computes (events order each copy
    # against the GEMVs that use the same buffer)
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()

    def steps_body(s0, count, e2e=False):
        cur = torch.cuda.current_stream()
        if e2e != "overlap":
            # plain steps, or (e2e "serial") each step's copies in line with its GEMVs
            for s in range(s0, s0 + count):
                ws = W[s % L]
                if e2e:
                    Xall.copy_(Xh, non_blocking=True)
                for j, (_, n, k) in enumerate(SET):
                    pq.pq_gemv(FMT, ws[j], n, k, X[j], 1, Y[j], cur)
                if e2e:
                    Yh.copy_(Yall, non_blocking=True)
            return
        start = torch.cuda.Event()
        start.record(cur)
        h2d_stream.wait_event(start)
        d2h_stream.wait_event(start)
        gemv_done = [None, None]
        d2h_done = [None, None]
        for s in range(s0, s0 + count):
            b = s % 2
            ws = W[s % L]
            with torch.cuda.stream(h2d_stream):
                if gemv_done[b] is not None:
                    h2d_stream.wait_event(gemv_done[b])      # step s - 2 has read XA[b]
                XA[b].copy_(Xh, non_blocking=True)
                h2d = torch.cuda.Event()
                h2d.record(h2d_stream)
            cur.wait_event(h2d)
            if d2h_done[b] is not None:
                cur.wait_event(d2h_done[b])                   # step s - 2's y has left YA[b]
            for j, (_, n, k) in enumerate(SET):
                pq.pq_gemv(FMT, ws[j], n, k, XB[b][j], 1, YB[b][j], cur)
            done = torch.cuda.Event()
            done.record(cur)
            gemv_done[b] = done
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(done)
                Yh.copy_(YA[b], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(d2h_stream)
                d2h_done[b] = ev
        # join the side streams
        for st in (h2d_stream, d2h_stream):
            ev = torch.cuda.Event()
            ev.record(st)
            cur.wait_event(ev)

    def capture(count, e2e=False):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            steps_body(0, count, e2e)
        return g

    def timed(K, e2e=False):
        """Replay graphs covering exactly K steps; returns milliseconds."""
        P = min(K, args.graph_steps - args.graph_steps % L if args.graph_steps >= L else L)
        gA = capture(P, e2e)
        rest = K % P
        gB = capture(rest, e2e) if rest else None
        gA.replay()            # upload + warm
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks.mark_on()
        t0.record()
        for _ in range(K // P):
            gA.replay()
        if gB is not None:
            gB.replay()
        t1.record()
        torch.cuda.synchronize()
        clocks.mark_off()
        if world > 1:
            dist.barrier()
        return t0.elapsed_time(t1)

    def dominant_alone(n_launch):
        """Average duration of the dominant GEMV launched back to back (layers
        rotating), CUDA events around a graph of n_launch launches."""
        _, n, k = SET[dom]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cur = torch.cuda.current_stream()
            for i in range(n_launch):
                pq.pq_gemv(FMT, W[i % L][dom], n, k, X[dom], 1, Y[dom], cur)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n_launch

    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        gpu_id = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        gpu_id = str(local)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    for s0 in range(0, args.warmup, L):        # warm-up: plain stream launches
        steps_body(s0, min(L, args.warmup - s0))
    torch.cuda.synchronize()
    ms = timed(args.steps)
    dom_ms = dominant_alone(args.dominant_launches)

    # the same layer with the epilogues fused (PESTI README, "Conformance"):
    # QKV with its bias, O, gate+up with SwiGLU writing h (14336 values), and
    # the down projection reading h; same weights and bytes per step
    qkv_bias = torch.from_numpy(np.random.default_rng(9).normal(0.0, 0.5, SET[0][1]).astype(np.float32)).to(dev)
    H = torch.empty(FFN, dtype=torch.float32, device=dev)

    def fused_body(count):
        cur = torch.cuda.current_stream()
        for s in range(count):
            ws = W[s % L]
            pq.pq_gemv_bias(FMT, ws[0], SET[0][1], SET[0][2], X[0], 1, qkv_bias, Y[0], cur)
            pq.pq_gemv(FMT, ws[1], SET[1][1], SET[1][2], X[1], 1, Y[1], cur)
            pq.pq_gemv_swiglu(FMT, ws[2], FFN, SET[2][2], X[2], 1, H, cur)
            pq.pq_gemv(FMT, ws[3], SET[3][1], SET[3][2], H, 1, Y[3], cur)

    fused_body(min(L, args.warmup))
    torch.cuda.synchronize()
    fused_steps = min(args.steps, args.graph_steps)
    gF = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gF):
        fused_body(fused_steps)
    gF.replay()
    torch.cuda.synchronize()
    fa, fb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fa.record()
    gF.replay()
    fb.record()
    torch.cuda.synchronize()
    fused_us = fa.elapsed_time(fb) * 1e3 / fused_steps
    del gF
    # the same steps as plain stream launches (no graph), for comparison
    stream_steps = min(args.steps, 400)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sa.record()
    steps_body(0, stream_steps)
    sb.record()
    torch.cuda.synchronize()
    stream_ms = sa.elapsed_time(sb)

    # end to end through the same calls: each step copies its x in from pinned
    # host memory and its y back out, inside the timed region; "overlap" runs
    # those copies beside the neighbouring steps' GEMVs (independent steps),
    # "serial" in line with the step's own GEMVs (a dependent decode loop)
    Xh = Xall.cpu().pin_memory()
    Yh = torch.empty(Yall.numel(), dtype=torch.float32).pin_memory()
    e2e_ms = {}
    for mode in ("serial", "overlap"):
        steps_body(0, min(args.warmup, L), e2e=mode)
        torch.cuda.synchronize()
        e2e_ms[mode] = timed(args.steps, e2e=mode)
    clocks.stop()
    peak, peak_src = measured_hbm_peak()
    configs = per_config(pq, dev, peak, torch.cuda.get_device_properties(local).L2_cache_size) \
        if not args.no_per_config else None

    ms, e2e_ms, e2e_serial_ms, dom_ms = max_over_ranks([ms, e2e_ms["overlap"], e2e_ms["serial"], dom_ms],
                                                       world, dev)

    nbytes = set_bytes()
    gbs = whole_job_rate(nbytes, args.steps, world, ms)
    e2e_gbs = whole_job_rate(nbytes, args.steps, world, e2e_ms)
    e2e_serial_gbs = whole_job_rate(nbytes, args.steps, world, e2e_serial_ms)
    dom_bytes = synth.weight_bytes(FMT, *[(n, k) for name, n, k in SET if name == DOMINANT][0])
    dom_gbs = dom_bytes / (dom_ms * 1e-3) / 1e9 if dom_ms else float("nan")
    src_hash = kernel_source_hash()
    traffic = NCU_TRAFFIC.get(src_hash)
    ncu_isolated = NCU_ISOLATED.get(src_hash)
    result = {
        "metric": METRIC,
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 6),
        "us_per_set": round(1e3 * ms / args.steps, 3),
        "hbm_frac": round(gbs / world / peak, 4),
        "hbm_frac_nominal_8000": round(gbs / world / NOMINAL_HBM_GBS, 4),
        "us_per_set_stream_launches": round(1e3 * stream_ms / stream_steps, 3),
        "fused_epilogue_set": {"us_per_set": round(fused_us, 3),
                               "workload": "QKV 6144x4096 + bias, O 4096x4096, gate+up 28672x4096 with SwiGLU "
                                           "(h of 14336), down 4096x14336 reading h; batch 1, CUDA graph",
                               "weight_GBs": round(set_bytes() / (fused_us * 1e-6) / 1e9, 1)},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "q4_k weights, f32 x/accumulate",
        "data": "synthetic",
        "config": {"workload": "Q4_K decode-layer set, batch 1 (QKV 6144x4096, O 4096x4096, "
                               "gate+up 28672x4096, down 4096x14336)",
                   "weight_bytes_per_step": nbytes, "batch": 1, "layers_resident": L,
                   "l2": f"inputs larger than L2: {L} layers x {nbytes} B rotate",
                   "weights": "synth.random_records (uniform packed fields, fp16 d/dmin)",
                   "launch": f"CUDA graph replay, {min(args.steps, args.graph_steps)} steps per graph",
                   "weight_prefetch": True,
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s",
                "h2d_bytes_per_step": sum(4 * k for _, _, k in SET),
                "d2h_bytes_per_step": sum(4 * n for _, n, _ in SET),
                "copies": "x in and y out every step on side streams, overlapping the neighbouring "
                          "steps' GEMVs (two x/y buffers)",
                "serial_value": round(e2e_serial_gbs, 2),
                "serial": "the same copies in line with the step's own GEMVs"},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"bound": "hbm", "kernel": f"pq_gemv {FMT} {DOMINANT} "
                     f"{[(n, k) for name, n, k in SET if name == DOMINANT][0]}",
                     "achieved": round(dom_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(dom_gbs / peak, 4), "peak_source": f"{peak_src} hbm copy",
                     "frac_of_nominal_8000": round(dom_gbs / NOMINAL_HBM_GBS, 4),
                     "traffic": traffic, "algorithmic_bytes": dom_bytes,
                     "method": f"dominant GEMV alone, {args.dominant_launches} launches back to back "
                               f"in one CUDA graph, weights of {L} layers rotating, CUDA events",
                     "kernel_source": src_hash,
                     "ncu_isolated": None if ncu_isolated is None else dict(
                         ncu_isolated, frac=round(dom_bytes / (ncu_isolated["us"] * 1e-6) / 1e9 / peak, 4),
                         method="the same launch under ncu, cold and alone (no neighbour to overlap)")},
        "clocks": clocks.summary(),
    }
    if configs is not None:
        result["per_config"] = {"method": "each workload alone, pq_gemv back to back in one CUDA graph, "
                                          "weights rotating over copies larger than ten times the L2, "
                                          "CUDA events; kernel = pq_gemv_choice id (0 generic, "
                                          "1 stream, 2 tensor core)",
                                "peak_GBs": peak, "results": configs}
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        result["cpu_detail"] = cpu_detail()
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


def _oracle_sample(budget_s: float):
    """Time the oracle on the set for about budget_s seconds: whole passes
    over the four GEMVs of one layer when one pass is shorter than the
    budget, else the same leading fraction of every GEMV's rows."""
    import oracle
    layer = [(n, k, synth.random_records(FMT, n, k, seed=j)) for j, (_, n, k) in enumerate(SET)]
    xs = [synth.normal_x(1, k, seed=7 + j) for j, (_, _, k) in enumerate(SET)]
    cores = oracle.threads(0)

    def one_pass(frac):
        done = 0
        for (n, k, w), x in zip(layer, xs):
            rows = np.arange(max(1, int(round(n * frac))))
            oracle.gemv_rows(FMT, w, n, k, x, rows)
            done += synth.weight_bytes(FMT, rows.size, k)
        return done

    t = time.perf_counter()
    probe = one_pass(0.02)
    rate = probe / max(time.perf_counter() - t, 1e-6)
    frac = min(1.0, rate * budget_s / set_bytes())
    reps = max(1, int(rate * budget_s / set_bytes())) if frac >= 1.0 else 1
    t = time.perf_counter()
    done = sum(one_pass(frac) for _ in range(reps))
    dt = time.perf_counter() - t
    return done, dt, cores, frac, reps


def cpu_detail(budget_each=0.6):
    """The oracle per format on a bounded row sample: f64 mat-vec and dequant,
    one thread and all cores (GB/s of weight bytes read)."""
    import oracle
    cores = oracle.threads(0)
    out = []
    for name, fmt, n, k in (("Q8_0 896x896", "q8_0", 896, 896), ("Q4_K 4096x4096", "q4_k", 4096, 4096),
                            ("Q6_K 128256x4096", "q6_k", 128256, 4096)):
        rows = min(n, 1024)
        w = synth.random_records(fmt, rows, k, seed=21)
        x = synth.normal_x(1, k, seed=22)
        rec = {"workload": name, "rows_sampled": rows}

        def rate(fn, nbytes):
            fn()
            reps, t0 = 0, time.perf_counter()
            while True:
                fn()
                reps += 1
                dt = time.perf_counter() - t0
                if dt >= budget_each or reps >= 200:
                    return round(nbytes * reps / dt / 1e9, 4)

        nbytes = synth.weight_bytes(fmt, rows, k)
        for label, nt in (("gemv_f64_1_thread", 1), ("gemv_f64_all_cores", 0)):
            rec[label] = rate(lambda: oracle.gemv_rows(fmt, w, rows, k, x, np.arange(rows), nthreads=nt), nbytes)
        for label, nt in (("dequant_1_thread", 1), ("dequant_all_cores", 0)):
            rec[label] = rate(lambda: oracle.dequant(fmt, w, rows, k, nthreads=nt), nbytes)
        out.append(rec)
    return {"unit": "GB/s of weight bytes", "cores": cores, "kind": "oracle", "results": out}


def cpu_baseline(budget_s):
    done, dt, cores, frac, reps = _oracle_sample(budget_s)
    what = (f"{reps} pass(es) over all rows of the 4 GEMVs of one layer" if frac >= 1.0 else
            f"first {100 * frac:.1f}% of the rows of each of the 4 GEMVs of one layer")
    return {"value": round(done / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{what} ({done} weight bytes, {dt:.1f} s, OpenMP over rows)"}


def run_reference(args):
    world, rank, _ = dist_init()
    if rank != 0:
        return
    total = args.warmup + args.steps
    per_step = max(0.05, args.ref_seconds / total)
    import oracle
    layer = [(n, k, synth.random_records(FMT, n, k, seed=j)) for j, (_, n, k) in enumerate(SET)]
    xs = [synth.normal_x(1, k, seed=7 + j) for j, (_, _, k) in enumerate(SET)]
    cores = oracle.threads(0)
    # rows per GEMV so that one step (a proportional sample of the set) takes ~per_step s
    t = time.perf_counter()
    probe = 0
    for (n, k, w), x in zip(layer, xs):
        oracle.gemv_rows(FMT, w, n, k, x, np.arange(max(1, n // 100)))
        probe += synth.weight_bytes(FMT, max(1, n // 100), k)
    rate = probe / max(time.perf_counter() - t, 1e-6)
    frac = min(1.0, rate * per_step / set_bytes())
    rows = [np.arange(max(1, int(n * frac))) for _, n, _ in SET]
    step_bytes = sum(synth.weight_bytes(FMT, r.size, k) for r, (_, _, k) in zip(rows, SET))

    def step():
        for (n, k, w), x, r in zip(layer, xs, rows):
            oracle.gemv_rows(FMT, w, n, k, x, r)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t
    value = step_bytes * args.steps / dt / 1e9
    sample = (f"each step: first {100 * frac:.2f}% of the rows of each of the 4 GEMVs "
              f"({step_bytes} weight bytes)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * dt / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 dot of decoded f32 weights",
        "data": "synthetic",
        "config": {"workload": "Q4_K decode-layer set, batch 1 (QKV 6144x4096, O 4096x4096, "
                               "gate+up 28672x4096, down 4096x14336)", "batch": 1},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_shape(args):
    """One shape launched back to back (for profiler captures and sweeps):
    --shape fmt:NxK[:batch], weights rotating over --rotate-mb of copies."""
    import torch
    from quantized_weight_mat_gb300 import build
    import quantized_weight_mat_gb300 as pq
    build.build()
    parts = args.shape.split(":")
    fmt = parts[0]
    n, k = (int(v) for v in parts[1].split("x"))
    batch = int(parts[2]) if len(parts) > 2 else 1
    nbytes = synth.weight_bytes(fmt, n, k)
    copies = max(2, -(-int(args.rotate_mb * 1e6) // nbytes))
    base = torch.from_numpy(synth.random_records(fmt, n, k, seed=5)).cuda()
    W = [base] + [base.clone() for _ in range(copies - 1)]
    x = torch.from_numpy(synth.normal_x(batch, k, seed=6)).cuda()
    y = torch.empty(batch * n, device="cuda")
    torch.cuda.synchronize()
    if not args.graph:
        for i in range(args.launches):
            pq.pq_gemv_kernel(fmt, W[i % copies], n, k, x, batch, y, kernel=args.kernel)
        torch.cuda.synchronize()
        print(json.dumps({"shape": args.shape, "launches": args.launches, "kernel": args.kernel,
                          "checksum": float(y.double().abs().sum())}))
        return
    # --graph: the launches captured in one CUDA graph with the weights
    # declared static, as the bench's per_config times them (so that a
    # profiler can take the whole graph as one workload); replayed once to
    # warm up, then once more, timed with CUDA events
    pq.pq_set_weight_prefetch(True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(3):
            pq.pq_gemv_kernel(fmt, W[i % copies], n, k, x, batch, y, kernel=args.kernel, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(args.launches):
                pq.pq_gemv_kernel(fmt, W[i % copies], n, k, x, batch, y, kernel=args.kernel, stream=s)
        g.replay()
        s.synchronize()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        g.replay()
        e.record(s)
    torch.cuda.synchronize()
    us = a.elapsed_time(e) * 1e3 / args.launches
    print(json.dumps({"shape": args.shape, "launches": args.launches, "kernel": args.kernel, "graph": True,
                      "us_per_launch": round(us, 3), "weight_GBs": round(nbytes / us / 1e3, 1),
                      "checksum": float(y.double().abs().sum())}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--graph-steps", type=int, default=400)
    ap.add_argument("--dominant-launches", type=int, default=400)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip timing each workload alone")
    ap.add_argument("--shape", default=None, help="fmt:NxK[:batch]: launch one shape only")
    ap.add_argument("--launches", type=int, default=6)
    ap.add_argument("--kernel", default="auto")
    ap.add_argument("--graph", action="store_true", help="--shape: the launches in one CUDA graph (weights static)")
    ap.add_argument("--rotate-mb", type=float, default=1400.0, help="--shape: MB of weight copies to rotate over")
    args = ap.parse_args()
    if args.shape:
        run_shape(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
