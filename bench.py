#!/usr/bin/env python3
"""Benchmark of the NF4 double-quant hot path on GB300.

One step = one pass of the whole path over the 4096 x 4096 NF4 matrix of the
4096^2 dequant workload (weights N(0, 0.02) with 0.1% of elements x10 as
outliers, blocksize 64, s2_blocksize 256):
    nf4_dequant -> bf16, nf4_dequant -> fp16, nf4_gemv batch 1 (x bf16 N(0,1)).
Inputs are quantized on the GPU by nf4_quantize (outside the timed region) and
copied into R rotation sets whose total footprint exceeds 4x the L2, so every
step reads its weights from HBM. Steps are replayed from CUDA graphs; each
kernel is bracketed by timing events captured in the graph.

Prints ONE JSON line (rank 0). Usage:
    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
For N > 1 run under torch.distributed.run: each rank is an independent replica
(no data-path collective), value = all ranks' bytes / max time over ranks.
"""
from __future__ import annotations

import argparse
import faulthandler
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "NF4 dequant GB/s and NF4-GEMV µs/layer, as % of GB300 HBM roofline"
N_ROWS, K_COLS = 4096, 4096
BS, S2 = 64, 256
W_SEED, OUTLIER_SEED, OUTLIER_FRAC = 1, 101, 0.001
X_SEED = 51                                   # x ~ N(0,1) of the 4096-wide batch-1 GEMV
WORKLOAD = ("nf4 4096x4096 (N(0,0.02) + 0.1% x10 outliers, blocksize 64, s2 256): "
            "dequant->bf16 + dequant->fp16 + fused GEMV batch 1 (fp32 accumulate)")


def replica_env():
    """(world, rank, local_rank) of this process: one independent replica per
    GPU under torch.distributed.run, else a single process."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x, world, device=None):
    """The largest x over all ranks (a job is as slow as its slowest replica);
    x itself for one process."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, bytes_per_replica_step, steps, seconds):
    """Whole-job GB/s: every replica moves bytes_per_replica_step per step;
    `seconds` is the slowest replica's time."""
    return world * bytes_per_replica_step * steps / seconds / 1e9


def algorithmic_bytes():
    n = N_ROWS * K_COLS
    nb = (n + BS - 1) // BS
    ng = (nb + S2 - 1) // S2
    quant = n // 2 + nb + 2 * ng + 2 * 256
    dequant = quant + 2 * n
    gemv = quant + 2 * K_COLS + 4 * N_ROWS
    return {"dequant_bf16": dequant, "dequant_fp16": dequant, "gemv_b1": gemv}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"nf4_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": sorted(reasons), "samples": 0}
        sm_sorted = sorted(sm)
        return {"sm_mhz": sm_sorted[len(sm_sorted) // 2], "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# native arm

def run_native(args, rank, world, local_rank):
    import numpy as np
    import torch

    import synth
    import w4a16_gemv_gb300 as nf4

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    n = N_ROWS * K_COLS
    bytes_ = algorithmic_bytes()
    step_bytes = sum(bytes_.values())

    # inputs: synthetic weights quantized on the GPU, x bf16
    w = torch.from_numpy(synth.weights(W_SEED, n, OUTLIER_FRAC, OUTLIER_SEED)).to(dev)
    code2 = torch.from_numpy(synth.code2_linear().view(np.float16)).to(dev)
    q = nf4.nf4_quantize(w, code2, BS, S2)
    del w
    x_host = synth.activations(X_SEED, 1, K_COLS)
    x0 = torch.from_numpy(x_host.view(np.int16)).to(dev).view(torch.bfloat16)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    set_bytes = (q.packed.numel() + q.absmax_q.numel() + 2 * q.absmax2.numel() + 4 * n + 2 * K_COLS
                 + 4 * N_ROWS)
    R = max(2, math.ceil(4 * l2 / set_bytes))
    sets = []
    for _ in range(R):
        sets.append(dict(packed=q.packed.clone(), absmax_q=q.absmax_q.clone(), absmax2=q.absmax2.clone(),
                         x=x0.clone(), out_bf16=torch.empty(n, dtype=torch.bfloat16, device=dev),
                         out_fp16=torch.empty(n, dtype=torch.float16, device=dev),
                         y=torch.empty((1, N_ROWS), dtype=torch.float32, device=dev)))
    offset = q.offset

    lib = nf4._lib
    ptr_args = []
    for s in sets:
        common = (s["packed"].data_ptr(), s["absmax_q"].data_ptr(), s["absmax2"].data_ptr(),
                  code2.data_ptr(), offset)
        ptr_args.append((common, s))

    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream
    names = ["dequant_bf16", "dequant_fp16", "gemv_b1"]

    def launch(kind, i):
        common, s = ptr_args[i % R]
        if kind == 0:
            st = lib.nf4_dequant(*common, n, BS, S2, s["out_bf16"].data_ptr(), nf4.NF4_BF16, sp)
        elif kind == 1:
            st = lib.nf4_dequant(*common, n, BS, S2, s["out_fp16"].data_ptr(), nf4.NF4_FP16, sp)
        else:
            st = lib.nf4_gemv(*common, N_ROWS, K_COLS, BS, S2, s["x"].data_ptr(), 1, s["y"].data_ptr(), sp)
        if st:
            raise RuntimeError(f"libnf4 call failed with status {st}")

    # A graph runs S steps kernel by kernel: S bf16 dequants, S fp16 dequants,
    # S GEMVs (step i on rotation set i mod R), with timing events only at the
    # three phase boundaries (an event between kernels costs microseconds on
    # this GPU; four per graph amortise over S launches each). Between two uses
    # of one set come R - 1 other launches of the phase (over 4x L2 of other
    # traffic), so every kernel reads its inputs from HBM; the per-kernel
    # average durations come from the phase events.
    K, W = args.steps, args.warmup
    BLOCKS = max(1, min(4, K // R)) if K >= R else 1

    def capture(nsteps):
        g = torch.cuda.CUDAGraph()
        evs = []
        with torch.cuda.stream(stream):
            g.capture_begin()
            e = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
            e[0].record(stream)
            for kind in range(3):
                for i in range(nsteps):
                    launch(kind, i)
                e[kind + 1].record(stream)
            evs.append((e, nsteps))
            g.capture_end()
        return g, evs

    # eager pass over every set (also validates every argument once)
    for i in range(R):
        for kind in range(3):
            launch(kind, i)
    stream.synchronize()

    S = R * BLOCKS if K >= R * BLOCKS else K
    g_main, evs = capture(S)
    rem = K % S
    g_rem = evs_rem = None
    if rem:
        # the graph's event-record nodes refer to these events: keep them alive
        g_rem, evs_rem = capture(rem)

    # warm-up: at least W steps
    done = 0
    with torch.cuda.stream(stream):
        while done < W:
            g_main.replay()
            done += S
    torch.cuda.synchronize()

    clocks = ClockSampler(dev.index)
    clocks.start()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(K // S):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    elapsed_ms = t0.elapsed_time(t1)
    clk = clocks.stop()

    # per-kernel average launch duration over the last replay of the main graph
    per_kernel = {}
    if K >= S:
        for j, name in enumerate(names):
            tot_ms, cnt = 0.0, 0
            for e, steps in evs:
                tot_ms += e[j].elapsed_time(e[j + 1])
                cnt += steps
            per_kernel[name] = tot_ms / cnt * 1e3   # us per launch
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)

    # the timed outputs are finite (a cheap guard; parity is the tests' job)
    assert torch.isfinite(sets[0]["y"]).all().item()

    peak, peak_src = load_peaks()
    ms_per_step = elapsed_ms / K
    value = job_throughput(world, step_bytes, K, elapsed_ms * 1e-3)

    detail = {}
    for name in names:
        us = per_kernel.get(name)
        if us:
            gbs = bytes_[name] / (us * 1e-6) / 1e9
            d = {"us": round(us, 3), "gbs": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak, 4)}
            if name.startswith("dequant"):
                d["gelem_per_s"] = round(N_ROWS * K_COLS / (us * 1e-6) / 1e9, 2)
            if name.startswith("gemv"):
                d["us_per_layer"] = d.pop("us")
            detail[name] = d
    dom = "dequant_bf16"
    roofline = None
    if dom in per_kernel:
        ach = bytes_[dom] / (per_kernel[dom] * 1e-6) / 1e9
        roofline = {"bound": "hbm", "kernel": "nf4_dequant (bf16 out)", "achieved": round(ach, 1),
                    "peak": peak, "peak_source": peak_src, "unit": "GB/s", "frac": round(ach / peak, 4),
                    "traffic": read_traffic(dom), "algorithmic_bytes_per_launch": bytes_[dom]}

    e2e = run_e2e(args, dev, q, code2, x_host, bytes_, world) if not args.no_e2e else None
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "bytes_per_step": step_bytes,
                   "l2_policy": f"rotation over {R} distinct input/output sets "
                                f"({R * set_bytes / 1e6:.0f} MB > 4x L2 {l2 / 1e6:.0f} MB)",
                   "timing": f"CUDA graph of {S} steps, kernel-major (all bf16 dequants, all fp16 "
                             f"dequants, all GEMVs) replayed; events only at the phase boundaries",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roofline, "detail": detail, "gpu_launches": 3 * K, "clocks": clk, "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_step:
        # the fused GEMV inside a recorded decode step (after the timed
        # region): per linear layer, Llama-7B shapes, batch 1
        del sets
        torch.cuda.empty_cache()
        gen = torch.Generator(device=dev)
        gen.manual_seed(4243)
        steps = {}
        for model, desc in (("llama-7b", "llama-7b-shaped (32 layers: q/k/v, o 4096x4096; gate/up 11008x4096; "
                                         "down 4096x11008)"),
                            ("qwen2.5-1.5b", "qwen2.5-1.5b-shaped (28 layers: q/o 1536x1536, k/v 256x1536 with "
                                             "bias; gate/up 8960x1536; down 1536x8960)")):
            st = decode_step(dev, gen, code2, 1, model)
            us = st["time"](reps=3, m=20)
            gbs = st["weight_bytes"] / us / 1e3
            steps[model] = {
                "model": desc, "batch": 1, "us_per_step": round(us, 1),
                "us_per_linear": round(us / st["linears"], 3), "launches_per_step": st["launches"],
                "weight_bytes": st["weight_bytes"], "gbs": round(gbs, 1),
                "frac_of_measured_hbm": round(gbs / peak, 4)}
            st["close"]()
            del st
            torch.cuda.empty_cache()
        result["decode_step"] = steps["llama-7b"]
        result["decode_step_qwen"] = steps["qwen2.5-1.5b"]
    if rank == 0 and world == 1 and not args.no_layers:
        # every GEMV layer shape of the configurations, timed on its own
        # (after the timed region; graphs of back-to-back launches over > 4x L2)
        layers = gemv_layer_times(dev, GEMV_LAYER_CASES, peak)
        result["detail"]["gemv_layers"] = layers
        gate = [d for d in layers if d["case"].startswith("llama-7b") and d["batch"] == 1]
        result["gemv_gate"] = {
            "target": "batch-1 fused GEMV >= 60% of measured HBM on the 4096x4096 and 7B-shaped layers",
            "layers": {f"{d['N']}x{d['K']}": {"us_per_layer": d["us_per_layer"], "gbs": d["gbs"],
                                              "frac_of_measured_hbm": d["frac_of_measured_hbm"]} for d in gate},
            "peak": peak, "peak_source": peak_src}
    if rank == 0 and world == 1 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(args, q, x_host, bytes_)
    return result


def read_traffic(kernel_name):
    """DRAM bytes per launch from the committed ncu summary, if it still
    matches the current source of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        import hashlib
        k = t["kernels"][kernel_name]
        src = os.path.join(ROOT, "w4a16_gemv_gb300", "csrc", k["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
        if h != k["source_sha256"]:
            return None
        return k["dram_bytes_per_launch"]
    except Exception:
        return None


def run_e2e(args, dev, q, code2, x_host, bytes_, world):
    """Same step through the public API with host buffers: H2D of the step's
    inputs from pinned memory and D2H of its outputs inside the timed region.
    Steps are pipelined as a caller would: the two dequant outputs go back to
    the host on two copy streams while the next step's inputs come in and its
    kernels run into the other of two device output sets."""
    import numpy as np
    import torch

    import w4a16_gemv_gb300 as nf4
    n = N_ROWS * K_COLS
    h_packed = q.packed.cpu().pin_memory()
    h_absmax_q = q.absmax_q.cpu().pin_memory()
    h_absmax2 = q.absmax2.cpu().pin_memory()
    h_code2 = code2.cpu().pin_memory()
    h_x = torch.from_numpy(x_host.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_bf16 = torch.empty(n, dtype=torch.bfloat16).pin_memory()
    h_fp16 = torch.empty(n, dtype=torch.float16).pin_memory()
    h_y = torch.empty((1, N_ROWS), dtype=torch.float32).pin_memory()
    d = dict(packed=torch.empty_like(q.packed), absmax_q=torch.empty_like(q.absmax_q),
             absmax2=torch.empty_like(q.absmax2), code2=torch.empty_like(code2),
             x=torch.empty((1, K_COLS), dtype=torch.bfloat16, device=dev),
             y=torch.empty((1, N_ROWS), dtype=torch.float32, device=dev))
    outs = [dict(bf16=torch.empty(n, dtype=torch.bfloat16, device=dev),
                 fp16=torch.empty(n, dtype=torch.float16, device=dev)) for _ in range(2)]
    main = torch.cuda.current_stream(dev)
    copy_streams = (torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev))
    copied = [None, None]   # per output set: events of its last D2H copies
    count = [0]
    h2d = sum(t.numel() * t.element_size() for t in (h_packed, h_absmax_q, h_absmax2, h_code2, h_x))
    d2h = sum(t.numel() * t.element_size() for t in (h_bf16, h_fp16, h_y))

    def step():
        o = outs[count[0] % 2]
        slot = count[0] % 2
        count[0] += 1
        for k, h in (("packed", h_packed), ("absmax_q", h_absmax_q), ("absmax2", h_absmax2),
                     ("code2", h_code2), ("x", h_x)):
            d[k].copy_(h, non_blocking=True)
        if copied[slot] is not None:   # the copies out of this output set two steps ago are done
            for e in copied[slot]:
                main.wait_event(e)
        nf4.nf4_dequant(d["packed"], d["absmax_q"], d["absmax2"], d["code2"], q.offset, n, BS, S2,
                        out=o["bf16"], out_dtype=torch.bfloat16)
        nf4.nf4_dequant(d["packed"], d["absmax_q"], d["absmax2"], d["code2"], q.offset, n, BS, S2,
                        out=o["fp16"], out_dtype=torch.float16)
        nf4.nf4_gemv(d["packed"], d["absmax_q"], d["absmax2"], d["code2"], q.offset, N_ROWS, K_COLS,
                     d["x"], y=d["y"], blocksize=BS, s2_blocksize=S2)
        done = torch.cuda.Event()
        done.record(main)
        h_y.copy_(d["y"], non_blocking=True)
        evs = []
        for cs, src, dst in ((copy_streams[0], o["bf16"], h_bf16), (copy_streams[1], o["fp16"], h_fp16)):
            cs.wait_event(done)
            with torch.cuda.stream(cs):
                dst.copy_(src, non_blocking=True)
            e = torch.cuda.Event()
            e.record(cs)
            evs.append(e)
        copied[slot] = evs

    steps = max(3, min(args.steps, 50))
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    dt = max_over_ranks(time.perf_counter() - t0, world, dev)
    step_bytes = sum(bytes_.values())
    return {"value": round(job_throughput(world, step_bytes, steps, dt), 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(dt / steps * 1e3, 4)}


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)

def _oracle_inputs(q=None, x_host=None):
    import numpy as np

    import oracle
    import synth
    n = N_ROWS * K_COLS
    if q is not None:
        t = oracle.NF4Tensor(q.packed.cpu().numpy(), q.absmax_q.cpu().numpy(),
                             q.absmax2.cpu().numpy().view(np.uint16), synth.code2_linear(), q.offset, n,
                             BS, S2)
    else:
        w = synth.weights(W_SEED, n, OUTLIER_FRAC, OUTLIER_SEED)
        t = oracle.quantize(w, BS, S2, synth.code2_linear())
    if x_host is None:
        x_host = synth.activations(X_SEED, 1, K_COLS)
    return t, x_host


def _oracle_step(t, x_host, rows):
    """One bounded sample of the step: the first `rows` rows of the matrix."""
    import oracle
    sub = oracle.NF4Tensor(t.packed, t.absmax_q, t.absmax2, t.code2, t.offset, rows * K_COLS, BS, S2)
    oracle.dequant(sub, oracle.BF16)
    oracle.dequant(sub, oracle.FP16)
    oracle.gemv(sub, rows, K_COLS, x_host)


def _sample_rows(t, x_host, budget_s):
    t0 = time.perf_counter()
    _oracle_step(t, x_host, 8)
    per_row = (time.perf_counter() - t0) / 8
    return max(1, min(N_ROWS, int(budget_s / per_row)))


def host_cpu():
    """The host's usable core count and a CPU description (the model name on
    x86, implementer/part codes on Arm), for the CPU-oracle figures."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    desc = ""
    try:
        fields = {}
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
        desc = fields.get("model name") or " ".join(
            f"{k} {fields[k]}" for k in ("CPU implementer", "CPU part") if k in fields)
    except OSError:
        pass
    import platform
    return {"host_cores": cores, "cpu": desc or platform.machine()}


def cpu_baseline(args, q, x_host, bytes_):
    t, x_host = _oracle_inputs(q, x_host)
    rows = _sample_rows(t, x_host, 2.0)
    reps = 0
    t0 = time.perf_counter()
    while True:
        _oracle_step(t, x_host, rows)
        reps += 1
        if time.perf_counter() - t0 > 10.0:
            break
    dt = time.perf_counter() - t0
    frac = rows / N_ROWS
    v = sum(bytes_.values()) * frac * reps / dt / 1e9
    return {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first {rows} of {N_ROWS} rows per step (dequant bf16 + fp16 + fp64 GEMV), "
                      f"{reps} steps in {dt:.1f} s, single-threaded C oracle", **host_cpu()}


def run_reference(args):
    bytes_ = algorithmic_bytes()
    t, x_host = _oracle_inputs()
    K, W = args.steps, args.warmup
    budget = max(0.002, 60.0 / max(1, K + W))
    rows = _sample_rows(t, x_host, budget)
    for _ in range(W):
        _oracle_step(t, x_host, rows)
    t0 = time.perf_counter()
    for _ in range(K):
        _oracle_step(t, x_host, rows)
    dt = time.perf_counter() - t0
    frac = rows / N_ROWS
    step_bytes = sum(bytes_.values()) * frac
    v = step_bytes * K / dt / 1e9
    sample = (f"first {rows} of {N_ROWS} rows per step (dequant bf16 + fp16 + fp64 GEMV), "
              f"single-threaded C oracle")
    return {"metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": K,
            "warmup": W, "ms_per_step": round(dt / K * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "impl": "reference", "config": {"workload": WORKLOAD, "parallelism": "single CPU core"},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample, **host_cpu()},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}



# ---------------------------------------------------------------------------
# --sweep: every configuration of the workload list timed on its own

def _sweep_time(launch, nsets, reps=5):
    """us per launch: a CUDA graph of back-to-back launches rotating over the
    input sets (events only at the graph's ends), best of `reps` replays."""
    import torch
    m = max(4 * nsets, 16)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(nsets):
            launch(i, s.cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    e0 = torch.cuda.Event(enable_timing=True, external=True)
    e1 = torch.cuda.Event(enable_timing=True, external=True)
    with torch.cuda.stream(s):
        g.capture_begin()
        e0.record(s)
        for i in range(m):
            launch(i % nsets, s.cuda_stream)
        e1.record(s)
        g.capture_end()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    best = None
    for _ in range(reps):
        g.replay()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / m
        best = us if best is None else min(best, us)
    return best


# The GEMV layer shapes of the configurations: the Qwen2.5-1.5B-shaped layers
# at batch 1 and the Llama-7B-shaped layers at batches 1, 4 and 8.
GEMV_LAYER_CASES = ([("qwen q/o", 1536, 1536, 1), ("qwen k/v", 256, 1536, 1), ("qwen gate/up", 8960, 1536, 1),
                     ("qwen down", 1536, 8960, 1)] +
                    [(f"llama-7b {nm}", N, K, b) for nm, N, K in
                     (("attn", 4096, 4096), ("gate/up", 11008, 4096), ("down", 4096, 11008)) for b in (1, 4, 8)])


def gemv_layer_times(dev, cases, peak, gen=None, l2=None):
    """us per layer of nf4_gemv for each (name, N, K, batch): a CUDA graph of
    back-to-back launches rotating over enough input sets (random codes and
    scales, x ~ N(0,1) bf16, fp32 y) to exceed 4x the L2, best of 5 replays.
    Bytes: packed + absmax_q + absmax2 + code2 + x + y."""
    import numpy as np
    import torch

    import w4a16_gemv_gb300 as nf4
    lib = nf4._lib
    if gen is None:
        gen = torch.Generator(device=dev)
        gen.manual_seed(2468)
    if l2 is None:
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    code2 = torch.from_numpy((((np.arange(256) - 127.5) / 127.5).astype(np.float16))).to(dev)
    out = []
    for name, N, K, batch in cases:
        n = N * K
        nb = (n + BS - 1) // BS
        ng = (nb + S2 - 1) // S2
        bytes_ = n // 2 + nb + 2 * ng + 512 + 2 * batch * K + 4 * batch * N
        r = max(2, int(math.ceil(4 * l2 / bytes_)))
        sets = []
        for _ in range(r):
            sets.append(dict(packed=torch.randint(0, 256, (n // 2,), dtype=torch.uint8, device=dev, generator=gen),
                             absmax_q=torch.randint(0, 256, (nb,), dtype=torch.uint8, device=dev, generator=gen),
                             absmax2=(torch.rand(ng, device=dev, generator=gen) * 0.04 + 0.01).half(),
                             x=torch.randn(batch, K, device=dev, generator=gen).to(torch.bfloat16),
                             y=torch.empty(batch, N, device=dev)))

        def launch(i, sp, N=N, K=K, batch=batch, sets=sets):
            st = sets[i]
            rc = lib.nf4_gemv(st["packed"].data_ptr(), st["absmax_q"].data_ptr(), st["absmax2"].data_ptr(),
                              code2.data_ptr(), 0.01, N, K, BS, S2, st["x"].data_ptr(), batch,
                              st["y"].data_ptr(), sp)
            if rc != 0:
                raise RuntimeError(f"nf4_gemv: {nf4.nf4_status_string(rc)}")
        us = _sweep_time(launch, r)
        gbs = bytes_ / us / 1e3
        out.append({"case": name, "N": N, "K": K, "batch": batch, "bytes": bytes_,
                    "us_per_layer": round(us, 3), "gbs": round(gbs, 1),
                    "frac_of_measured_hbm": round(gbs / peak, 4), "frac_of_8000": round(gbs / 8000.0, 4),
                    "sets": r})
        del sets
        torch.cuda.empty_cache()
    return out


# Linear layers of one decoder layer: (N, K) of q, k, v, o, gate, up, down.
DECODERS = {
    "qwen2.5-1.5b": dict(layers=28, hidden=1536, qkv_bias=True,
                         shapes=[(1536, 1536), (256, 1536), (256, 1536), (1536, 1536), (8960, 1536),
                                 (8960, 1536), (1536, 8960)]),
    "llama-7b": dict(layers=32, hidden=4096, qkv_bias=False,
                     shapes=[(4096, 4096), (4096, 4096), (4096, 4096), (4096, 4096), (11008, 4096),
                             (11008, 4096), (4096, 11008)]),
}


def decode_step(dev, gen, code2, batch, model="qwen2.5-1.5b"):
    """A recorded decode step (nf4_step_create) over the linear layers of a
    decoder of the named shape: per layer q/k/v (with bias for Qwen) from the
    layer input, o from q, gate/up from o, down from gate; bf16 outputs;
    random codes and scales (timing does not depend on the values). Returns
    the step's timer (us per replay, replays back to back on one stream), its
    weight bytes, its linear layers and its kernel launches per replay (q/k/v
    and gate/up grouped)."""
    import torch

    import w4a16_gemv_gb300 as nf4
    cfg = DECODERS[model]
    layers = cfg["layers"]
    shapes = cfg["shapes"]
    inputs = [-1, -1, -1, 0, 3, 3, 4]
    nodes, wbytes = [], 0
    for layer in range(layers):
        base = 7 * layer
        for j, (N, K) in enumerate(shapes):
            n = N * K
            nb = (n + BS - 1) // BS
            ng = (nb + S2 - 1) // S2
            wt = nf4.NF4Weight(torch.randint(0, 256, (n // 2,), dtype=torch.uint8, device=dev, generator=gen),
                               torch.randint(0, 256, (nb,), dtype=torch.uint8, device=dev, generator=gen),
                               (torch.rand(ng, device=dev, generator=gen) * 0.04 + 0.01).half(),
                               code2, 0.01, n, (N, K), BS, S2)
            wbytes += n // 2 + nb + 2 * ng
            inp = inputs[j]
            inp = (-1 if layer == 0 else base - 1) if inp == -1 else base + inp
            bias = (torch.randn(N, device=dev, generator=gen).to(torch.bfloat16)
                    if j < 3 and cfg["qkv_bias"] else None)
            nodes.append(dict(weight=wt, y=torch.empty((batch, N), dtype=torch.bfloat16, device=dev),
                              bias=bias, input=inp))
    x = torch.randn((batch, cfg["hidden"]), device=dev, generator=gen).to(torch.bfloat16)
    step = nf4.DecodeStep(nodes, x)

    def time_step(reps=5, m=50):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for _ in range(5):
                step.launch(s)
        s.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        best = None
        for _ in range(reps):
            with torch.cuda.stream(s):
                e0.record(s)
                for _ in range(m):
                    step.launch(s)
                e1.record(s)
            s.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / m
            best = us if best is None else min(best, us)
        return best
    return {"time": time_step, "weight_bytes": wbytes, "launches": step.kernel_count(), "linears": 7 * layers,
            "close": step.close}


def run_one_gemv(args):
    """--gemv N,K,B: --steps launches of one fused GEMV on random codes and
    scales (a fixed, small command line to put under a profiler)."""
    import numpy as np
    import torch

    import w4a16_gemv_gb300 as nf4
    N, K, B = (int(v) for v in args.gemv.split(","))
    dev = torch.device("cuda:0")
    gen = torch.Generator(device=dev)
    gen.manual_seed(777)
    code2 = torch.from_numpy((((np.arange(256) - 127.5) / 127.5).astype(np.float16))).to(dev)
    n = N * K
    nb = (n + BS - 1) // BS
    packed = torch.randint(0, 256, (n // 2,), dtype=torch.uint8, device=dev, generator=gen)
    aq = torch.randint(0, 256, (nb,), dtype=torch.uint8, device=dev, generator=gen)
    a2 = (torch.rand((nb + S2 - 1) // S2, device=dev, generator=gen) * 0.04 + 0.01).half()
    x = torch.randn(B, K, device=dev, generator=gen).to(torch.bfloat16)
    y = torch.empty(B, N, device=dev)
    for _ in range(args.steps):
        nf4.nf4_gemv(packed, aq, a2, code2, 0.001, N, K, x, y=y)
    torch.cuda.synchronize()
    return {"gemv": [N, K, B], "launches": args.steps, "mean_abs_y": float(y.abs().mean())}


def run_one_dequant(args):
    """--dequant N: --steps launches of nf4_dequant of N elements (bf16 out) on
    random codes and scales (a fixed, small command line to put under a
    profiler; N = 234881024 is the 28672x8192 case, larger than L2)."""
    import numpy as np
    import torch

    import w4a16_gemv_gb300 as nf4
    n = int(args.dequant)
    dev = torch.device("cuda:0")
    gen = torch.Generator(device=dev)
    gen.manual_seed(778)
    code2 = torch.from_numpy((((np.arange(256) - 127.5) / 127.5).astype(np.float16))).to(dev)
    nb = (n + BS - 1) // BS
    packed = torch.randint(0, 256, ((n + 1) // 2,), dtype=torch.uint8, device=dev, generator=gen)
    aq = torch.randint(0, 256, (nb,), dtype=torch.uint8, device=dev, generator=gen)
    a2 = (torch.rand((nb + S2 - 1) // S2, device=dev, generator=gen) * 0.04 + 0.01).half()
    out = torch.empty(n, dtype=torch.bfloat16, device=dev)
    for _ in range(args.steps):
        nf4.nf4_dequant(packed, aq, a2, code2, 0.001, n, BS, S2, out=out, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    return {"dequant": n, "launches": args.steps, "bytes_per_launch": (n + 1) // 2 + nb + 2 * ((nb + S2 - 1) // S2)
            + 512 + 2 * n}


def run_decode_step(args):
    """--decode-step: W replays untimed, then K replays back to back between
    two events; one JSON line."""
    import numpy as np
    import torch
    dev = torch.device("cuda:0")
    peak, peak_kind = load_peaks()
    code2 = torch.from_numpy((((np.arange(256) - 127.5) / 127.5).astype(np.float16))).to(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242)
    step = decode_step(dev, gen, code2, args.batch, args.model)
    us = step["time"](reps=1, m=args.steps)
    gbs = step["weight_bytes"] / us / 1e3
    step["close"]()
    cfg = DECODERS[args.model]
    return {"metric": f"decode step us ({args.model}-shaped, {cfg['layers']} layers x 7 fused GEMVs)",
            "value": round(us, 1), "unit": "us/step", "higher_is_better": False,
            "batch": args.batch, "steps": args.steps, "launches_per_step": step["launches"],
            "us_per_linear": round(us / step["linears"], 3),
            "weight_bytes": step["weight_bytes"], "gbs": round(gbs, 1),
            "frac_of_measured_hbm": round(gbs / peak, 4), "peak_kind": peak_kind,
            "data": f"synthetic random codes and scales; weights {step['weight_bytes'] / 1e6:.0f} MB > L2 "
                    "(no flush needed)"}


def run_sweep(args):
    """Times nf4_dequant on configs 0, 1, 2 (standalone dequant of each Qwen
    layer) and 4, nf4_gemv on configs 2 and 3 at batch 1/4/8, nf4_gemv_ex
    (bf16 y + bias), batches 16/32/64 on config 3, and the recorded decode
    step of a Qwen2.5-1.5B-shaped decoder at batch 1 and 4. Inputs are
    synthetic random codes and scales (timing does not depend on the values);
    each case rotates over enough input sets to exceed 4x the L2."""
    import numpy as np
    import torch

    import w4a16_gemv_gb300 as nf4
    lib = nf4._lib
    dev = torch.device("cuda:0")
    peak, peak_kind = load_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    code2 = torch.from_numpy((((np.arange(256) - 127.5) / 127.5).astype(np.float16))).to(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(12345)
    out = []

    def quant_set(n):
        nb = (n + BS - 1) // BS
        ng = (nb + S2 - 1) // S2
        return dict(packed=torch.randint(0, 256, ((n + 1) // 2,), dtype=torch.uint8, device=dev, generator=gen),
                    absmax_q=torch.randint(0, 256, (nb,), dtype=torch.uint8, device=dev, generator=gen),
                    absmax2=(torch.rand(ng, device=dev, generator=gen) * 0.04 + 0.01).half())

    def nsets_for(bytes_each, cap=8 << 30):
        return max(1, min(int(math.ceil(4 * l2 / bytes_each)), max(1, cap // bytes_each)))

    dq_cases = [("cfg0 1024x1024", 1024 * 1024, 0), ("cfg1 4096x4096", 4096 * 4096, 0),
                ("cfg1 4096x4096", 4096 * 4096, 1)]
    dq_cases += [(f"cfg2 dequant {nm}", n * k, 0) for nm, n, k in
                 (("q/o 1536x1536", 1536, 1536), ("k/v 256x1536", 256, 1536),
                  ("gate/up 8960x1536", 8960, 1536), ("down 1536x8960", 1536, 8960))]
    dq_cases += [("cfg4 28672x8192", 28672 * 8192, 0)]
    dq_cases += [(f"cfg4 flat 2^{e}", 1 << e, 0) for e in (20, 22, 24, 26, 28, 30)]
    dq_cases += [("cfg4 ragged 64*256*1000+64*37", 64 * 256 * 1000 + 64 * 37, 0)]
    for name, n, dtype in dq_cases:
        nb = (n + BS - 1) // BS
        ng = (nb + S2 - 1) // S2
        bytes_ = (n + 1) // 2 + nb + 2 * ng + 512 + 2 * n
        r = nsets_for(bytes_)
        sets = []
        for _ in range(r):
            st = quant_set(n)
            st["out"] = torch.empty(n, dtype=torch.bfloat16 if dtype == 0 else torch.float16, device=dev)
            sets.append(st)

        def launch(i, sp, n=n, dtype=dtype, sets=sets):
            st = sets[i]
            rc = lib.nf4_dequant(st["packed"].data_ptr(), st["absmax_q"].data_ptr(), st["absmax2"].data_ptr(),
                                 code2.data_ptr(), 0.01, n, BS, S2, st["out"].data_ptr(), dtype, sp)
            if rc != 0:
                raise RuntimeError(f"nf4_dequant: {nf4.nf4_status_string(rc)}")
        us = _sweep_time(launch, r)
        gbs = bytes_ / us / 1e3
        out.append({"kind": "dequant", "case": name, "out": "bf16" if dtype == 0 else "fp16", "n": n,
                    "bytes": bytes_, "us": round(us, 3), "gbs": round(gbs, 1),
                    "gelem_per_s": round(n / us / 1e3, 2),
                    "frac_of_measured_hbm": round(gbs / peak, 4), "frac_of_8000": round(gbs / 8000.0, 4),
                    "sets": r})
        del sets
        torch.cuda.empty_cache()

    for d in gemv_layer_times(dev, GEMV_LAYER_CASES, peak, gen, l2):
        d["kind"] = "gemv"
        out.append(d)
    # Output stage fused (bf16 y + bias) and batches above 8 (slabs of eight).
    ex_cases = [("cfg2 q/o bf16+bias", 1536, 1536, 1), ("cfg2 k/v bf16+bias", 256, 1536, 1),
                ("cfg3 attn bf16+bias", 4096, 4096, 1)]
    ex_cases += [(f"cfg3 {nm} wide", N, K, b) for nm, N, K in
                 (("attn", 4096, 4096), ("gate/up", 11008, 4096), ("down", 4096, 11008))
                 for b in (16, 32, 64)]
    for name, N, K, batch in ex_cases:
        n = N * K
        nb = (n + BS - 1) // BS
        ng = (nb + S2 - 1) // S2
        ex = "bias" in name
        bytes_ = n // 2 + nb + 2 * ng + 512 + 2 * batch * K + (2 if ex else 4) * batch * N + (2 * N if ex else 0)
        r = max(2, nsets_for(bytes_))
        sets = []
        for _ in range(r):
            st = quant_set(n)
            st["x"] = torch.randn(batch, K, device=dev, generator=gen).to(torch.bfloat16)
            st["y"] = torch.empty(batch, N, device=dev, dtype=torch.bfloat16 if ex else torch.float32)
            st["b"] = torch.randn(N, device=dev, generator=gen).to(torch.bfloat16)
            sets.append(st)

        def launch(i, sp, N=N, K=K, batch=batch, sets=sets, ex=ex):
            st = sets[i]
            if ex:
                rc = lib.nf4_gemv_ex(st["packed"].data_ptr(), st["absmax_q"].data_ptr(),
                                     st["absmax2"].data_ptr(), code2.data_ptr(), 0.01, N, K, BS, S2,
                                     st["x"].data_ptr(), batch, st["b"].data_ptr(), st["y"].data_ptr(),
                                     0, sp)
            else:
                rc = lib.nf4_gemv(st["packed"].data_ptr(), st["absmax_q"].data_ptr(),
                                  st["absmax2"].data_ptr(), code2.data_ptr(), 0.01, N, K, BS, S2,
                                  st["x"].data_ptr(), batch, st["y"].data_ptr(), sp)
            if rc != 0:
                raise RuntimeError(f"nf4_gemv: {nf4.nf4_status_string(rc)}")
        us = _sweep_time(launch, r)
        gbs = bytes_ / us / 1e3
        out.append({"kind": "gemv", "case": name, "N": N, "K": K, "batch": batch, "bytes": bytes_,
                    "us_per_layer": round(us, 3), "gbs": round(gbs, 1),
                    "frac_of_measured_hbm": round(gbs / peak, 4), "frac_of_8000": round(gbs / 8000.0, 4),
                    "sets": r})
        del sets
        torch.cuda.empty_cache()

    for model, label in (("qwen2.5-1.5b", "Qwen2.5-1.5B-shaped step, 28 layers x 7 GEMVs"),
                         ("llama-7b", "Llama-7B-shaped step, 32 layers x 7 GEMVs")):
        for batch in (1, 4):
            step = decode_step(dev, gen, code2, batch, model)
            us, wbytes = step["time"](), step["weight_bytes"]
            gbs = wbytes / us / 1e3
            out.append({"kind": "decode_step", "case": label, "batch": batch,
                        "launches": step["launches"], "weight_bytes": wbytes,
                        "us_per_step": round(us, 1), "us_per_linear": round(us / step["linears"], 3),
                        "gbs": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak, 4)})
            step["close"]()
            del step
            torch.cuda.empty_cache()

    for d in out:
        if d["kind"] == "decode_step":
            print(f"{'step':8s} {d['case'] + ' B=' + str(d['batch']):44s} {d['us_per_step']:10.1f} us "
                  f"{d['gbs']:9.1f} GB/s {100 * d['frac_of_measured_hbm']:5.1f}% of {peak:.0f} ({peak_kind})",
                  file=sys.stderr)
            continue
        what = d["case"] + (f" {d['out']}" if d["kind"] == "dequant" else f" B={d['batch']}")
        t = d["us"] if d["kind"] == "dequant" else d["us_per_layer"]
        print(f"{d['kind']:8s} {what:44s} {t:10.3f} us {d['gbs']:9.1f} GB/s "
              f"{100 * d['frac_of_measured_hbm']:5.1f}% of {peak:.0f} ({peak_kind}) "
              f"{100 * d['frac_of_8000']:5.1f}% of 8000", file=sys.stderr)
    return {"sweep": out, "peak_gbs": peak, "peak_kind": peak_kind,
            "timing": "CUDA graph of back-to-back launches over rotating input sets (> 4x L2), "
                      "events at the graph's ends, best of 5 replays",
            "data": "synthetic random codes and scales"}


def main():
    faulthandler.enable()
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=500)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-step", action="store_true", help="skip the decode-step detail")
    ap.add_argument("--no-layers", action="store_true", help="skip the per-layer GEMV detail")
    ap.add_argument("--sweep", action="store_true",
                    help="time every dequant and GEMV configuration instead of the step")
    ap.add_argument("--decode-step", action="store_true",
                    help="time the recorded decode step of a Qwen2.5-1.5B-shaped decoder instead")
    ap.add_argument("--batch", type=int, default=1, help="batch of --decode-step")
    ap.add_argument("--model", choices=sorted(DECODERS), default="qwen2.5-1.5b",
                    help="decoder shape of --decode-step")
    ap.add_argument("--dequant", type=int, default=None, metavar="N",
                    help="--steps launches of one bf16 dequant of N elements (for profilers)")
    ap.add_argument("--gemv", type=str, default=None, metavar="N,K,B",
                    help="run --steps launches of one N x K fused GEMV at batch B (for profilers)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.steps < 1:
        raise SystemExit("--steps must be >= 1")

    world, rank, local_rank = replica_env()

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return
    if args.sweep:
        if rank == 0:
            print(json.dumps(run_sweep(args)), flush=True)
        return
    if args.decode_step:
        if rank == 0:
            print(json.dumps(run_decode_step(args)), flush=True)
        return
    if args.gemv:
        if rank == 0:
            print(json.dumps(run_one_gemv(args)), flush=True)
        return
    if args.dequant:
        if rank == 0:
            print(json.dumps(run_one_dequant(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        result = run_native(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


if __name__ == "__main__":
    main()
