"""Benchmark: the Q4_K decode-layer mat-vec set of an 8B-shaped model, batch 1.

One step = the four batch-1 GEMVs of one transformer layer with hidden 4096,
32 query / 8 key-value heads of 128 and a 14336-wide MLP:
  QKV 4096 -> 6144, O 4096 -> 4096, fused gate+up 4096 -> 28672, down 14336 -> 4096,
122,683,392 bytes of Q4_K weights.  The weights of L distinct layers stay
resident in HBM and step s uses layer s mod L, so each step's weights were
evicted from L2 by the L-1 layers in between (inputs larger than L2; no
flush needed).

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

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant
# kernel from one ncu capture, keyed by the sha256 of the kernel source it was
# taken on; any edit of that source makes the figure stale (reported as null).
NCU_TRAFFIC = {}


def set_bytes():
    return sum(synth.weight_bytes(FMT, n, k) for _, n, k in SET)


def kernel_source_hash():
    p = os.path.join(ROOT, "quantized_weight_mat_gb300", "csrc", "gemv_stream.cu")
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


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
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    L = args.layers

    # resident weights of L layers; x and y per GEMV
    W = []
    for layer in range(L):
        W.append([torch.from_numpy(synth.random_records(FMT, n, k, seed=1000 * layer + j)).to(dev)
                  for j, (_, n, k) in enumerate(SET)])
    X = [torch.from_numpy(synth.normal_x(1, k, seed=7 + j)).to(dev) for j, (_, n, k) in enumerate(SET)]
    Y = [torch.empty(n, dtype=torch.float32, device=dev) for _, n, _ in SET]
    launches_per_step = sum(pq.pq_gemv_launches(FMT, n, k, 1) for _, n, k in SET)
    dom = [name for name, _, _ in SET].index(DOMINANT)
    torch.cuda.synchronize()

    def step(s, ev=None):
        ws = W[s % L]
        for j, (_, n, k) in enumerate(SET):
            if ev is not None and j == dom:
                ev[0].record(stream)
            pq.pq_gemv(FMT, ws[j], n, k, X[j], 1, Y[j], stream)
            if ev is not None and j == dom:
                ev[1].record(stream)

    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        gpu_id = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        gpu_id = str(local)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    dom_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark_on()
    t0.record(stream)
    for s in range(args.steps):
        step(s, dom_ev[s])
    t1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_off()
    if world > 1:
        dist.barrier()
    ms = t0.elapsed_time(t1)
    dom_ms = float(np.mean([a.elapsed_time(b) for a, b in dom_ev]))

    # end to end through the same calls: x copied in from pinned host memory
    # and y copied back, every step, inside the timed region
    Xh = [x.cpu().pin_memory() for x in X]
    Yh = [torch.empty(y.numel(), dtype=torch.float32).pin_memory() for y in Y]

    def e2e_step(s):
        ws = W[s % L]
        for j, (_, n, k) in enumerate(SET):
            X[j].copy_(Xh[j], non_blocking=True)
            pq.pq_gemv(FMT, ws[j], n, k, X[j], 1, Y[j], stream)
            Yh[j].copy_(Y[j], non_blocking=True)

    for s in range(args.warmup):
        e2e_step(s)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(args.steps):
        e2e_step(s)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    clocks.stop()

    if world > 1:
        t = torch.tensor([ms, e2e_ms, dom_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms, e2e_ms, dom_ms = t.tolist()

    nbytes = set_bytes()
    gbs = nbytes * args.steps * world / (ms * 1e-3) / 1e9
    e2e_gbs = nbytes * args.steps * world / (e2e_ms * 1e-3) / 1e9
    peak, peak_src = measured_hbm_peak()
    dom_bytes = synth.weight_bytes(FMT, *[(n, k) for name, n, k in SET if name == DOMINANT][0])
    dom_gbs = dom_bytes / (dom_ms * 1e-3) / 1e9
    src_hash = kernel_source_hash()
    traffic = NCU_TRAFFIC.get(src_hash)
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
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s",
                "h2d_bytes_per_step": sum(4 * k for _, _, k in SET),
                "d2h_bytes_per_step": sum(4 * n for _, n, _ in SET)},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"bound": "hbm", "kernel": f"pq_gemv {FMT} {DOMINANT} "
                     f"{[(n, k) for name, n, k in SET if name == DOMINANT][0]}",
                     "achieved": round(dom_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(dom_gbs / peak, 4), "peak_source": f"{peak_src} hbm copy",
                     "traffic": traffic, "algorithmic_bytes": dom_bytes,
                     "kernel_source": src_hash},
        "clocks": clocks.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


def _oracle_sample(budget_s: float):
    """Time the oracle on the set: every GEMV on a prefix of its rows sized
    so that the whole sample takes about budget_s seconds."""
    import oracle
    layer = [(n, k, synth.random_records(FMT, n, k, seed=1000 * 0 + j))
             for j, (_, n, k) in enumerate(SET)]
    xs = [synth.normal_x(1, k, seed=7 + j) for j, (_, _, k) in enumerate(SET)]
    cores = oracle.threads(0)
    # calibrate on 2% of the rows
    t = time.perf_counter()
    done = 0
    for (n, k, w), x in zip(layer, xs):
        rows = np.arange(max(1, n // 50))
        oracle.gemv_rows(FMT, w, n, k, x, rows)
        done += synth.weight_bytes(FMT, rows.size, k)
    rate = done / max(time.perf_counter() - t, 1e-6)
    frac = min(1.0, rate * budget_s / set_bytes())
    t = time.perf_counter()
    done = 0
    for (n, k, w), x in zip(layer, xs):
        rows = np.arange(max(1, int(n * frac)))
        oracle.gemv_rows(FMT, w, n, k, x, rows)
        done += synth.weight_bytes(FMT, rows.size, k)
    dt = time.perf_counter() - t
    return done, dt, cores, frac


def cpu_baseline(budget_s):
    done, dt, cores, frac = _oracle_sample(budget_s)
    return {"value": round(done / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"first {100 * frac:.1f}% of the rows of each of the 4 GEMVs of one layer "
                      f"({done} weight bytes, {dt:.1f} s)"}


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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
