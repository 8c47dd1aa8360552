#!/usr/bin/env python3
"""Benchmark of the NVFP4 weight-only SwiGLU FFN decode on GB300.

One step = one decode FFN forward (gate/up dual GEMV + activation, then the
down GEMV) through each of L distinct layers for one batch of M token rows.
The layers' packed weights (L x 3 x H x I x 0.5625 bytes) are far larger than
L2, so every step streams weights from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--m M]
  python bench.py --impl reference ...     (the CPU oracle on the host cores)

Prints ONE JSON line (rank 0).  `value` is the effective HBM bandwidth of the
whole job: algorithmic bytes (3*H*I*0.5625 weight bytes + 2*M*H*2 activation
bytes per layer) / device time, summed over ranks.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per FFN layer and effective HBM GB/s (% of GB300 peak), M=1..16"

WORKLOADS = {
    "single_token": dict(H=5120, I=17408, M=1, act=0, layers=48, outliers=0.0,
                         desc="single-token SwiGLU FFN decode H=5120 I=17408 M=1 SiLU, "
                              "48 distinct NVFP4 layers"),
    "spec_verify": dict(H=4096, I=12288, M=2, act=0, layers=32, outliers=0.0,
                        desc="speculative-verify FFN H=4096 I=12288 M=2|3 SiLU, 32 layers"),
    "batch_m": dict(H=5120, I=17408, M=8, act=0, layers=48, outliers=0.01,
                    desc="batch-M verify FFN H=5120 I=17408 M=4|8|16, x with 1% outliers x20, "
                         "48 layers"),
    "large": dict(H=5376, I=21504, M=1, act=0, layers=62, outliers=0.0,
                  desc="large dense FFN H=5376 I=21504 M=1..16 SiLU, 62 layers"),
}

KERNEL_SOURCES = ["nvfp4_weight_only_gb300/csrc/stream_gemv.cu",
                  "nvfp4_weight_only_gb300/csrc/device_util.cuh",
                  "nvfp4_weight_only_gb300/csrc/layout.h"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dual_gate_up_single_token_traffic.json")


def layer_bytes(H, I, M):
    return 3 * H * I * 0.5625 + 2 * M * H * 2


def dual_kernel_bytes(H, I, M):
    # gate+up weights, x read, h written
    return 2 * H * I * 0.5625 + M * H * 2 + M * I * 2


def down_kernel_bytes(H, I, M):
    return H * I * 0.5625 + M * I * 2 + M * H * 2


def kernel_source_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.file = None
        self.windows = []

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self, t0, t1):
        """Keep only samples taken between wall-clock times t0 and t1."""
        self.windows.append((t0, t1))

    def _in_window(self, stamp):
        from datetime import datetime
        try:
            t = datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return True
        return any(a - 0.05 <= t <= b + 0.05 for a, b in self.windows) if self.windows else True

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9 or not self._in_window(r[0]):
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def reduce_max(values, device=None):
    """Element-wise maximum of `values` over all ranks of the default process
    group (identity on a single process)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def whole_job_gbs(world, bytes_per_step, steps, seconds):
    """Whole-job effective bandwidth: every rank's bytes over the slowest rank's time."""
    return world * bytes_per_step * steps / seconds / 1e9


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------------- our arm

def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    from nvfp4_weight_only_gb300 import ffi, synth

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    ffi.load(build_if_missing=True)
    H, I, M, L = wl["H"], wl["I"], args.m or wl["M"], args.layers or wl["layers"]
    act = wl["act"] if args.act is None else args.act

    # ---- load time: quantise + repack every layer on the device (untimed)
    layers = []
    for li in range(L):
        q = []
        for proj, (n, k) in ((synth.GATE, (I, H)), (synth.UP, (I, H)), (synth.DOWN, (H, I))):
            w = synth.weights_f32(n, k, seed=synth.layer_seed(li, proj) + 7919 * rank, device=dev)
            q.append(ffi.nvfp4_quantize(w))
            del w
        gu = ffi.nvfp4_repack_gate_up(q[0][0], q[0][1], q[1][0], q[1][1], I, H)
        dn = ffi.nvfp4_repack(q[2][0], q[2][1], H, I)
        layers.append((gu, q[0][2], q[1][2], dn, q[2][2]))
        del q
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    x = synth.activations_bf16(M, H, seed=0, outlier_frac=wl["outliers"], device=dev)
    out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    ws = ffi.workspace(ffi.ffn_swiglu_nvfp4_workspace_bytes(M, H, I), dev)
    h = torch.empty((M, I), dtype=torch.bfloat16, device=dev)
    ws_gu = ffi.workspace(ffi.ffn_gate_up_nvfp4_workspace_bytes(M, H, I), dev)
    ws_dn = ffi.workspace(ffi.nvfp4_gemv_workspace_bytes(M, H, I), dev)

    def step():
        for (gu, g2, u2, dn, d2) in layers:
            ffi.ffn_swiglu_nvfp4(x, gu, g2, u2, dn, d2, I, act, ws=ws, out=out)

    def dual_only():
        for (gu, g2, u2, dn, d2) in layers:
            ffi.ffn_gate_up_nvfp4(x, gu, g2, u2, I, act, ws=ws_gu, h=h)

    def down_only():
        for (gu, g2, u2, dn, d2) in layers:
            ffi.nvfp4_gemv(h, dn, d2, H, ws=ws_dn, out=out)

    stream = torch.cuda.Stream(device=dev)
    graphs = {}
    with torch.cuda.stream(stream):
        for name, fn in (("step", step), ("dual", dual_only), ("down", down_only)):
            fn()  # first launch sets kernel attributes outside capture
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            graphs[name] = g
    torch.cuda.synchronize()

    def timed(graph, reps):
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(reps):
                graph.replay()
            ev1.record(stream)
        ev1.synchronize()
        return ev0.elapsed_time(ev1) / 1e3

    # ---- warm-up, then the timed region (barrier + sync on both sides)
    for _ in range(args.warmup):
        graphs["step"].replay()
    torch.cuda.synchronize()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    w0 = time.time()
    t_step = timed(graphs["step"], args.steps)
    torch.cuda.synchronize()
    sampler.mark(w0, time.time())
    if world > 1:
        dist.barrier()
    # per-kernel averages (same process, same stream, CUDA events)
    kreps = max(3, min(args.steps, 200))
    for _ in range(2):
        graphs["dual"].replay()
    w0 = time.time()
    t_dual = timed(graphs["dual"], kreps) / (kreps * L)
    t_down = timed(graphs["down"], kreps) / (kreps * L)
    sampler.mark(w0, time.time())
    time.sleep(0.15)
    clocks = sampler.stop()

    # ---- end to end through the public API with host buffers
    x_host = x.cpu().pin_memory()
    out_host = torch.empty((M, H), dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    with torch.cuda.stream(stream):
        for _ in range(2):
            x.copy_(x_host, non_blocking=True)
            step()
            out_host.copy_(out, non_blocking=True)
        stream.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(e2e_steps):
            x.copy_(x_host, non_blocking=True)
            step()
            out_host.copy_(out, non_blocking=True)
        ev1.record(stream)
        ev1.synchronize()
    t_e2e_eager = ev0.elapsed_time(ev1) / 1e3 / e2e_steps

    # The same step as a serving loop would run it: the pinned-host copy of x,
    # the 48 public-API calls and the read-back of out, captured once into a
    # CUDA graph and replayed (the calls only enqueue work on the stream).
    with torch.cuda.stream(stream):
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e, stream=stream):
            x.copy_(x_host, non_blocking=True)
            step()
            out_host.copy_(out, non_blocking=True)
        for _ in range(2):
            g_e2e.replay()
        stream.synchronize()
        ev0.record(stream)
        for _ in range(e2e_steps):
            g_e2e.replay()
        ev1.record(stream)
        ev1.synchronize()
    t_e2e = ev0.elapsed_time(ev1) / 1e3 / e2e_steps
    status = ffi.nvfp4_workspace_status(ws)
    if status != 0:
        raise RuntimeError(f"device status word reports {status} (bounded wait abandoned)")

    t_max, t_e2e, t_e2e_eager = reduce_max([t_step, t_e2e, t_e2e_eager], device=dev)
    per_step = layer_bytes(H, I, M) * L
    value = whole_job_gbs(world, per_step, args.steps, t_max)
    us_layer = t_max / (args.steps * L) * 1e6
    peak, peak_kind = measured_peaks()
    dual_gbs = dual_kernel_bytes(H, I, M) / t_dual / 1e9
    traffic = None
    if os.path.exists(TRAFFIC_FILE):
        with open(TRAFFIC_FILE) as f:
            tr = json.load(f)
        if (tr.get("source_hash") == kernel_source_hash() and tr.get("H") == H
                and tr.get("I") == I and tr.get("M") == M):
            traffic = tr.get("bytes_per_launch")
    line = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t_max / args.steps * 1e3, 4),
            "us_per_layer": round(us_layer, 3),
            "pct_of_peak": round(100.0 * value / world / peak, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded N(0,0.02) weights quantised on device, "
                                    "N(0,1) bf16 activations)",
            "config": {"workload": wl["desc"], "H": H, "I": I, "M": M,
                       "act": "silu" if act == 0 else "gelu_tanh", "layers": L,
                       "outliers": wl["outliers"], "graph": "one CUDA graph per step",
                       "l2": f"inputs larger than L2: {L} distinct layers, "
                             f"{L * 3 * H * I * 0.5625 / 1e9:.2f} GB packed weights",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": "dual gate+up GEMV + activation",
                         "achieved": round(dual_gbs, 1), "peak": peak, "peak_kind": peak_kind,
                         "unit": "GB/s", "frac": round(dual_gbs / peak, 4), "traffic": traffic,
                         "algorithmic_bytes_per_launch": dual_kernel_bytes(H, I, M),
                         "us_per_launch": round(t_dual * 1e6, 3)},
            "down_kernel": {"achieved": round(down_kernel_bytes(H, I, M) / t_down / 1e9, 1),
                            "unit": "GB/s", "frac": round(down_kernel_bytes(H, I, M) / t_down
                                                          / 1e9 / peak, 4),
                            "us_per_launch": round(t_down * 1e6, 3)},
            "e2e": {"value": round(whole_job_gbs(world, per_step, 1, t_e2e), 1), "unit": "GB/s",
                    "h2d_bytes_per_step": M * H * 2, "d2h_bytes_per_step": M * H * 2,
                    "path": "pinned-host x copy, per-layer ffn_swiglu_nvfp4 C-ABI calls, "
                            "out read-back, captured in one CUDA graph per step",
                    "eager_value": round(whole_job_gbs(world, per_step, 1, t_e2e_eager), 1),
                    "eager_path": "the same calls issued one by one from Python (ctypes) "
                                  "each step"},
            "gpu_launches": 2 * L * args.steps,
            "clocks": clocks,
        }
    if world > 1:
        dist.barrier()
    return line


def cpu_baseline(wl, M, budget_s=10.0):
    """The oracle FFN on the host cores for one layer of the workload."""
    import numpy as np

    import oracle
    from nvfp4_weight_only_gb300 import synth

    H, I = wl["H"], wl["I"]
    act = wl["act"]
    cores = oracle.set_threads(os.cpu_count() or 1)
    q = [oracle.quantize(synth.weights_f32(n, k, seed=synth.layer_seed(0, p)).numpy())
         for p, (n, k) in ((synth.GATE, (I, H)), (synth.UP, (I, H)), (synth.DOWN, (H, I)))]
    x = synth.bf16_bits(synth.activations_bf16(M, H, seed=0, outlier_frac=wl["outliers"]))
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.ffn(x, I, q[0], q[1], q[2], act)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 1000:
            break
    per = el / reps
    return {"value": round(layer_bytes(H, I, M) / per / 1e9, 3), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{reps} oracle FFN forward(s) of layer 0 (H={H}, I={I}, M={M}), "
                      f"{el:.1f} s, {per * 1e3:.1f} ms/layer"}, q, x


def run_reference(args, wl):
    """--impl reference: the CPU oracle timed on the host cores, same config/metric."""
    import oracle

    world, rank, _ = dist_setup()
    if rank != 0:
        return None
    H, I, M = wl["H"], wl["I"], args.m or wl["M"]
    cb, q, x = cpu_baseline(wl, M, budget_s=0.0)
    for _ in range(args.warmup):
        oracle.ffn(x, I, q[0], q[1], q[2], wl["act"])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.ffn(x, I, q[0], q[1], q[2], wl["act"])
    el = time.perf_counter() - t0
    value = layer_bytes(H, I, M) * args.steps / el / 1e9
    cores = oracle.set_threads(0)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl["desc"], "H": H, "I": I, "M": M,
                   "act": "silu" if wl["act"] == 0 else "gelu_tanh",
                   "sample": "one layer per step (the oracle is the reference arm)"},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} oracle FFN forwards of layer 0"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="single_token")
    ap.add_argument("--m", type=int, default=None, help="token rows (overrides the workload)")
    ap.add_argument("--act", type=int, default=None, choices=[0, 1])
    ap.add_argument("--layers", type=int, default=None,
                    help="distinct layers (fewer only for small profiling runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    wl = WORKLOADS[args.workload]
    if args.impl == "reference":
        line = run_reference(args, wl)
    else:
        line = run_ours(args, wl)
        world, rank, _ = dist_setup()
        if line is not None and rank == 0 and world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl, line["config"]["M"], args.cpu_budget)[0]
    if line is not None:
        print(json.dumps(line), flush=True)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and args.impl == "ours":
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
