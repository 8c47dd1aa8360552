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
bytes per layer) / device time, summed over ranks.  On one GPU the line also
carries `sweep`: the same metric for M = 1..16 on the headline layer (with the
gate/up and down kernels timed on their own), the 1%-outlier batch-M variants
with SiLU and GeLU, the speculative-verify and large dense layers, and points of
the standalone GEMV sweep (`--no-sweep` skips it).
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

KERNEL_SOURCES = ["nvfp4_weight_only_gb300/csrc/stream_kernel.cuh",
                  "nvfp4_weight_only_gb300/csrc/stream_gemv.cu",
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


def grid_bytes(N, K):
    return ((N + 127) // 128) * ((K + 127) // 128) * 4


def w8a16_layer_bytes(H, I, M):
    # FP8 codes and block grids of gate, up and down, x read, out written
    return 3 * H * I + 2 * grid_bytes(I, H) + grid_bytes(H, I) + 2 * M * H * 2


def w8a16_dual_bytes(H, I, M):
    return 2 * H * I + 2 * grid_bytes(I, H) + M * H * 2 + M * I * 2


def w8a16_down_bytes(H, I, M):
    return H * I + grid_bytes(H, I) + M * I * 2 + M * H * 2


def build_w8a16_layers(ffi, synth, H, I, L, dev):
    """L distinct block-scaled FP8 FFN layers (seeded stand-ins for an FP8
    checkpoint), repacked on the device (load time, untimed)."""
    import torch

    layers = []
    for li in range(L):
        proj = [synth.fp8_weights(n, k, seed=synth.layer_seed(li, p) + 77, device=dev)
                for p, (n, k) in ((synth.GATE, (I, H)), (synth.UP, (I, H)), (synth.DOWN, (H, I)))]
        gu = ffi.w8a16_repack_gate_up(proj[0][0], proj[0][1], proj[1][0], proj[1][1])
        dn = ffi.w8a16_repack(*proj[2])
        layers.append((gu, dn))
        del proj
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return layers


def w8a16_case(ffi, synth, timer, dev, lyrs, H, I, M, act, reps, peak, kernels=True):
    """µs per layer of ffn_swiglu_w8a16 over the distinct layers in one CUDA
    graph, and (kernels) each of its two kernels alone.  Returns (entry,
    launches, wall-clock window)."""
    import torch

    x = synth.activations_bf16(M, H, seed=M, device=dev)
    out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    L = ffi.load()
    ws = ffi.workspace(L.ffn_swiglu_w8a16_workspace_bytes(M, H, I), dev)

    def fn():
        for gu, dn in lyrs:
            ffi.ffn_swiglu_w8a16(x, gu, dn, I, act, ws=ws, out=out)

    g = timer.capture(fn)
    w0 = time.time()
    t = timer.time(g, reps, warmup=3) / (reps * len(lyrs))
    launches = 2 * len(lyrs) * reps
    gbs = w8a16_layer_bytes(H, I, M) / t / 1e9
    entry = {"us_per_layer": round(t * 1e6, 3), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}
    del g
    if kernels:
        # the down kernel alone through w8a16_gemv; the gate/up kernel is the
        # layer minus it (the two run back to back in the FFN)
        h = synth.activations_bf16(M, I, seed=M + 1, device=dev)
        ws_g = ffi.workspace(L.w8a16_gemv_workspace_bytes(M, H, I), dev)

        def down():
            for gu, dn in lyrs:
                ffi.w8a16_gemv(h, dn, H, ws=ws_g, out=out)

        gk = timer.capture(down)
        tk = timer.time(gk, reps, warmup=3) / (reps * len(lyrs))
        launches += len(lyrs) * reps
        del gk
        entry["down"] = {"us_per_launch": round(tk * 1e6, 3),
                         "frac": round(w8a16_down_bytes(H, I, M) / tk / 1e9 / peak, 4)}
        td = t - tk  # the layer is the two kernels back to back
        entry["dual"] = {"us_per_launch": round(td * 1e6, 3), "derived": "layer minus down",
                         "frac": round(w8a16_dual_bytes(H, I, M) / td / 1e9 / peak, 4)}
        if ffi.nvfp4_workspace_status(ws_g) != 0:
            raise RuntimeError("device status word reports a bounded wait abandoned")
    if ffi.nvfp4_workspace_status(ws) != 0:
        raise RuntimeError("device status word reports a bounded wait abandoned")
    return entry, launches, (w0, time.time())


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

def build_layers(ffi, synth, H, I, L, dev, seed_offset=0):
    """Quantise + repack L distinct FFN layers on the device (load time, untimed)."""
    import torch

    layers = []
    for li in range(L):
        q = []
        for proj, (n, k) in ((synth.GATE, (I, H)), (synth.UP, (I, H)), (synth.DOWN, (H, I))):
            w = synth.weights_f32(n, k, seed=synth.layer_seed(li, proj) + seed_offset, device=dev)
            q.append(ffi.nvfp4_quantize(w))
            del w
        gu = ffi.nvfp4_repack_gate_up(q[0][0], q[0][1], q[1][0], q[1][1], I, H)
        dn = ffi.nvfp4_repack(q[2][0], q[2][1], H, I)
        layers.append((gu, q[0][2], q[1][2], dn, q[2][2]))
        del q
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return layers


class GraphTimer:
    """Captures a callable into a CUDA graph on one stream and times replays
    with CUDA events recorded on that stream."""

    def __init__(self, stream):
        self.stream = stream

    def capture(self, fn):
        import torch

        with torch.cuda.stream(self.stream):
            fn()  # first launch sets kernel attributes outside capture
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                fn()
        torch.cuda.synchronize()
        return g

    def time(self, graph, reps, warmup=0):
        import torch

        with torch.cuda.stream(self.stream):
            for _ in range(warmup):
                graph.replay()
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            ev0.record(self.stream)
            for _ in range(reps):
                graph.replay()
            ev1.record(self.stream)
        ev1.synchronize()
        return ev0.elapsed_time(ev1) / 1e3


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
    layers = build_layers(ffi, synth, H, I, L, dev, seed_offset=7919 * rank)
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
    timer = GraphTimer(stream)
    graphs = {name: timer.capture(fn)
              for name, fn in (("step", step), ("dual", dual_only), ("down", down_only))}

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
    t_step = timer.time(graphs["step"], args.steps)
    torch.cuda.synchronize()
    sampler.mark(w0, time.time())
    if world > 1:
        dist.barrier()
    # per-kernel averages (same process, same stream, CUDA events)
    kreps = max(3, min(args.steps, 200))
    w0 = time.time()
    t_dual = timer.time(graphs["dual"], kreps, warmup=2) / (kreps * L)
    t_down = timer.time(graphs["down"], kreps, warmup=2) / (kreps * L)
    sampler.mark(w0, time.time())

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
    # the per-layer public-API calls and the read-back of out, captured once
    # into a CUDA graph and replayed (the calls only enqueue work on the stream).
    def e2e_step():
        x.copy_(x_host, non_blocking=True)
        step()
        out_host.copy_(out, non_blocking=True)

    g_e2e = timer.capture(e2e_step)
    t_e2e = timer.time(g_e2e, e2e_steps, warmup=2) / e2e_steps
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

    # ---- the metric's whole M range and the other configured shapes (one GPU)
    sweep, sweep_launches = None, 0
    if world == 1 and not args.no_sweep:
        sweep, sweep_launches = run_sweep(args, ffi, synth, dev, timer, sampler, layers, H, I,
                                          peak)
    time.sleep(0.15)
    clocks = sampler.stop()

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
        if sweep is not None:
            line["sweep"] = sweep
            line["sweep_gpu_launches"] = sweep_launches
    if world > 1:
        dist.barrier()
    return line


def _layer_entry(t_layer, H, I, M, peak):
    gbs = layer_bytes(H, I, M) / t_layer / 1e9
    return {"us_per_layer": round(t_layer * 1e6, 3), "gbs": round(gbs, 1),
            "frac": round(gbs / peak, 4)}


def run_sweep(args, ffi, synth, dev, timer, sampler, layers, H, I, peak):
    """M = 1..16 on the headline layer (with per-kernel times), the batch-M
    outlier variants (SiLU and GeLU), the speculative-verify layer, the large
    dense layer and points of the standalone GEMV sweep.  Every entry is a CUDA
    graph of all its distinct layers (or weight copies), larger than L2,
    replayed `--sweep-reps` times after warm-up and timed with CUDA events."""
    import torch

    reps = args.sweep_reps
    launches = 0
    res = {"reps": reps, "note": "µs per layer, effective GB/s and fraction of the measured "
                                 "HBM copy peak; per-kernel figures for the headline layer"}

    def ffn_case(lyrs, H, I, M, act, outliers, kernels=False):
        nonlocal launches
        x = synth.activations_bf16(M, H, seed=M, outlier_frac=outliers, device=dev)
        out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        ws = ffi.workspace(ffi.ffn_swiglu_nvfp4_workspace_bytes(M, H, I), dev)

        def fn():
            for (gu, g2, u2, dn, d2) in lyrs:
                ffi.ffn_swiglu_nvfp4(x, gu, g2, u2, dn, d2, I, act, ws=ws, out=out)

        g = timer.capture(fn)
        w0 = time.time()
        t = timer.time(g, reps, warmup=3) / (reps * len(lyrs))
        launches += 2 * len(lyrs) * reps
        entry = _layer_entry(t, H, I, M, peak)
        if kernels:
            h = torch.empty((M, I), dtype=torch.bfloat16, device=dev)
            ws_gu = ffi.workspace(ffi.ffn_gate_up_nvfp4_workspace_bytes(M, H, I), dev)
            ws_dn = ffi.workspace(ffi.nvfp4_gemv_workspace_bytes(M, H, I), dev)

            def dual():
                for (gu, g2, u2, dn, d2) in lyrs:
                    ffi.ffn_gate_up_nvfp4(x, gu, g2, u2, I, act, ws=ws_gu, h=h)

            def down():
                for (gu, g2, u2, dn, d2) in lyrs:
                    ffi.nvfp4_gemv(h, dn, d2, H, ws=ws_dn, out=out)

            for name, f, nbytes in (("dual", dual, dual_kernel_bytes(H, I, M)),
                                    ("down", down, down_kernel_bytes(H, I, M))):
                gk = timer.capture(f)
                tk = timer.time(gk, reps, warmup=3) / (reps * len(lyrs))
                launches += len(lyrs) * reps
                entry[name] = {"us_per_launch": round(tk * 1e6, 3),
                               "frac": round(nbytes / tk / 1e9 / peak, 4)}
                del gk
            if ffi.nvfp4_workspace_status(ws_gu) != 0 or ffi.nvfp4_workspace_status(ws_dn) != 0:
                raise RuntimeError("device status word reports a bounded wait abandoned")
        sampler.mark(w0, time.time())
        if ffi.nvfp4_workspace_status(ws) != 0:
            raise RuntimeError("device status word reports a bounded wait abandoned")
        del g
        return entry

    head = {}
    for M in range(1, 17):
        head[f"M{M}"] = ffn_case(layers, H, I, M, 0, 0.0, kernels=True)
    res[f"ffn_{H}x{I}_silu"] = head
    # verify batches / small prefill beyond one kernel group (16 rows)
    res[f"ffn_{H}x{I}_silu_large_batches"] = {f"M{M}": ffn_case(layers, H, I, M, 0, 0.0)
                                              for M in (17, 24, 32, 48, 64)}
    bm = {}
    for M in (4, 8, 16):
        for act, name in ((0, "silu"), (1, "gelu_tanh")):
            bm[f"M{M}_{name}"] = ffn_case(layers, H, I, M, act, 0.01)
    res[f"ffn_{H}x{I}_outliers_1pct"] = bm
    # LoRA overlay (rank 16 on gate, up and down; one adapter shared by the layers)
    lr = {}
    r = 16
    gen = torch.Generator(device=dev)
    gen.manual_seed(17)

    def rnd(*shape):
        return (torch.randn(shape, generator=gen, device=dev) * 0.05).to(torch.bfloat16)

    pairs = dict(gate=(rnd(r, H), rnd(I, r)), up=(rnd(r, H), rnd(I, r)), down=(rnd(r, I), rnd(H, r)))
    for M in (1, 8):
        x = synth.activations_bf16(M, H, seed=M, device=dev)
        out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        ws = ffi.workspace(ffi.load().ffn_swiglu_nvfp4_lora_workspace_bytes(M, H, I, r), dev)

        def fn():
            for (gu, g2, u2, dn, d2) in layers:
                ffi.ffn_swiglu_nvfp4_lora(x, gu, g2, u2, dn, d2, I, 0, ws=ws, out=out, **pairs)

        g = timer.capture(fn)
        w0 = time.time()
        t = timer.time(g, reps, warmup=3) / (reps * len(layers))
        sampler.mark(w0, time.time())
        launches += 6 * len(layers) * reps
        lr[f"M{M}_r{r}"] = _layer_entry(t, H, I, M, peak)
        if ffi.nvfp4_workspace_status(ws) != 0:
            raise RuntimeError("device status word reports a bounded wait abandoned")
        del g
    res[f"ffn_{H}x{I}_lora_gate_up_down"] = lr
    torch.cuda.empty_cache()

    # the fixed-workspace entry point against the caller-workspace one: the same
    # 48 calls per step issued eagerly from Python, timed with CUDA events on
    # the issuing stream, after the fixed array's one-time set-up
    na = {}
    for M in (1, 8):
        x = synth.activations_bf16(M, H, seed=M, device=dev)
        out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        ws = ffi.workspace(ffi.ffn_swiglu_nvfp4_workspace_bytes(M, H, I), dev)
        entry = {}
        for name, call in (("workspace", lambda l: ffi.ffn_swiglu_nvfp4(
                               x, l[0], l[1], l[2], l[3], l[4], I, 0, ws=ws, out=out)),
                           ("noalloc", lambda l: ffi.ffn_swiglu_nvfp4_noalloc(
                               x, l[0], l[1], l[2], l[3], l[4], I, 0, out=out))):
            st = torch.cuda.Stream(device=dev)
            with torch.cuda.stream(st):
                for _ in range(2):  # warm-up (includes the fixed array's set-up)
                    for lyr in layers:
                        call(lyr)
                st.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                w0 = time.time()
                e0.record(st)
                for _ in range(reps):
                    for lyr in layers:
                        call(lyr)
                e1.record(st)
                e1.synchronize()
                sampler.mark(w0, time.time())
            t = e0.elapsed_time(e1) * 1e-3 / (reps * len(layers))
            launches += 2 * len(layers) * (reps + 2)
            entry[name] = _layer_entry(t, H, I, M, peak)
        if ffi.nvfp4_workspace_status(ws) != 0 or ffi.nvfp4_noalloc_status() != 0:
            raise RuntimeError("device status word reports a bounded wait abandoned")
        na[f"M{M}"] = entry
    res[f"ffn_{H}x{I}_noalloc_vs_workspace_eager"] = na

    # block-scaled FP8 weights (the pages' native FP8 arm) on the headline layer
    f8 = {}
    f8_layers = build_w8a16_layers(ffi, synth, H, I, 24, dev)
    for M in (1, 2, 4, 8, 16):
        entry, n, win = w8a16_case(ffi, synth, timer, dev, f8_layers, H, I, M, 0, reps, peak)
        launches += n
        sampler.mark(*win)
        f8[f"M{M}"] = entry
    res[f"ffn_{H}x{I}_w8a16_silu"] = f8
    del f8_layers
    torch.cuda.empty_cache()

    for key, Hs, Is, Ls, Ms in (("spec_verify", 4096, 12288, 32, (2, 3)),
                                ("large", 5376, 21504, 62, (1, 2, 4, 8, 12, 16))):
        lyrs = build_layers(ffi, synth, Hs, Is, Ls, dev)
        res[f"{key}_{Hs}x{Is}"] = {f"M{M}": ffn_case(lyrs, Hs, Is, M, 0, 0.0) for M in Ms}
        del lyrs
        torch.cuda.empty_cache()

    # standalone nvfp4_gemv: enough identical weight copies (distinct addresses)
    # to exceed 2 GB, so every launch streams from HBM
    gem = {}
    for (N, K) in ((4096, 4096), (17408, 5120), (5120, 17408), (65536, 4096), (4096, 21504),
                   (65536, 21504)):
        w = synth.weights_f32(N, K, seed=N + K, device=dev)
        c, s, s2 = ffi.nvfp4_quantize(w)
        del w
        p = ffi.nvfp4_repack(c, s, N, K)
        del c, s
        nbytes = N * K * 0.5625
        copies = int(min(256, max(3, -(-2.2e9 // nbytes))))
        ps = [p] + [p.clone() for _ in range(copies - 1)]
        for M in (1, 4, 8, 16):
            x = synth.activations_bf16(M, K, seed=M, device=dev)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = ffi.workspace(ffi.nvfp4_gemv_workspace_bytes(M, N, K), dev)

            def fn():
                for pc in ps:
                    ffi.nvfp4_gemv(x, pc, s2, N, ws=ws, out=y)

            g = timer.capture(fn)
            w0 = time.time()
            t = timer.time(g, reps, warmup=3) / (reps * copies)
            sampler.mark(w0, time.time())
            launches += copies * reps
            gbs = (nbytes + M * K * 2 + M * N * 2) / t / 1e9
            gem[f"N{N}_K{K}_M{M}"] = {"us_per_launch": round(t * 1e6, 3), "gbs": round(gbs, 1),
                                      "frac": round(gbs / peak, 4), "copies": copies}
            if ffi.nvfp4_workspace_status(ws) != 0:
                raise RuntimeError("device status word reports a bounded wait abandoned")
            del g
        del ps, p
        torch.cuda.empty_cache()
    res["gemv"] = gem
    return res, launches


def run_gemv(args):
    """--gemv N,K: the standalone nvfp4_gemv on enough weight copies (distinct
    addresses, over 2 GB) that every launch streams from HBM, in one CUDA graph."""
    import torch

    from nvfp4_weight_only_gb300 import ffi, synth

    N, K = (int(v) for v in args.gemv.split(","))
    M = args.m or 1
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ffi.load(build_if_missing=True)
    w = synth.weights_f32(N, K, seed=N + K, device=dev)
    c, s, s2 = ffi.nvfp4_quantize(w)
    del w
    p = ffi.nvfp4_repack(c, s, N, K)
    del c, s
    nbytes = N * K * 0.5625
    copies = args.layers or int(min(256, max(3, -(-2.2e9 // nbytes))))
    ps = [p] + [p.clone() for _ in range(copies - 1)]
    x = synth.activations_bf16(M, K, seed=M, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = ffi.workspace(ffi.nvfp4_gemv_workspace_bytes(M, N, K), dev)

    def fn():
        for pc in ps:
            ffi.nvfp4_gemv(x, pc, s2, N, ws=ws, out=y)

    timer = GraphTimer(torch.cuda.Stream(device=dev))
    g = timer.capture(fn)
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    t = timer.time(g, args.steps) / (args.steps * copies)
    if ffi.nvfp4_workspace_status(ws) != 0:
        raise RuntimeError("device status word reports a bounded wait abandoned")
    peak, kind = measured_peaks()
    gbs = (nbytes + M * K * 2 + M * N * 2) / t / 1e9
    return {"metric": "µs per standalone nvfp4_gemv launch and effective HBM GB/s",
            "value": round(gbs, 1), "unit": "GB/s", "us_per_launch": round(t * 1e6, 3),
            "frac": round(gbs / peak, 4), "peak": peak, "peak_kind": kind, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "config": {"workload": f"standalone GEMV N={N} K={K} M={M}", "copies": copies},
            "gpu_launches": copies * args.steps}


def run_w8a16(args):
    """--w8a16: the block-scaled FP8 FFN on the headline layer (5120 x 17408)
    over distinct layers in one CUDA graph, at --m token rows."""
    import torch

    from nvfp4_weight_only_gb300 import ffi, synth

    H, I, M = 5120, 17408, args.m or 1
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ffi.load(build_if_missing=True)
    L = args.layers or 24
    lyrs = build_w8a16_layers(ffi, synth, H, I, L, dev)
    timer = GraphTimer(torch.cuda.Stream(device=dev))
    peak, kind = measured_peaks()
    entry, launches, _ = w8a16_case(ffi, synth, timer, dev, lyrs, H, I, M, args.act or 0,
                                    args.steps, peak, kernels=True)
    return {"metric": "µs per block-scaled FP8 FFN layer and effective HBM GB/s",
            "value": entry["gbs"], "unit": "GB/s", **entry, "peak": peak, "peak_kind": kind,
            "n_gpus": 1, "steps": args.steps, "warmup": 3, "higher_is_better": True,
            "config": {"workload": f"FP8 (w8a16) SwiGLU FFN H={H} I={I} M={M}, {L} layers"},
            "gpu_launches": launches}


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
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the M=1..16 / other-shape sweep (one GPU only)")
    ap.add_argument("--sweep-reps", type=int, default=10)
    ap.add_argument("--gemv", default=None, metavar="N,K",
                    help="time the standalone GEMV of one N x K projection instead")
    ap.add_argument("--w8a16", action="store_true",
                    help="time the block-scaled FP8 FFN on the headline layer instead")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    wl = WORKLOADS[args.workload]
    if args.w8a16:
        print(json.dumps(run_w8a16(args)), flush=True)
        return
    if args.gemv:
        print(json.dumps(run_gemv(args)), flush=True)
        return
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
