"""Benchmark of the QLoRA NF4 hot path on B300.

Headline (one JSON line on rank 0): the fused QLoRA forward at M = 1 over the
Llama-7B-shaped decode set -- 32 layers x {q, k, v, o: 4096x4096;
gate, up: 11008x4096; down: 4096x11008}, NF4 with double quantisation, LoRA
r = 64, alpha = 16 -- reported as GB/s of 4-bit weight bytes (codes + int8
constants + scales + mean).  One step = one forward of every one of the 224
matrices (the whole weight set is 3.34 GB, far above the 126 MB L2, so no
flush is needed between steps).

Secondary numbers measured in the same run: the same set at M = 16, the
prefill-shaped layer (M = 4096, 11008 x 4096, r = 16) forward and backward
dX in TFLOP/s, bulk NF4 quantise / dequantise of the 6.48 B-parameter bf16
set in GB/s, and LoftQ (4096 x 4096, r = 16, T = 5) seconds per alternation.

--impl reference times the CPU oracle on the same metric (bounded sample).
Under torchrun every rank runs its own replica of the decode set (weak
scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "QLoRA NF4 linear GB/s (M=1) & TFLOP/s (M=4096); NF4 quantize GB/s"
WORKLOAD = "llama7b-decode-set M=1: 32 layers x 7 NF4+DQ matrices (q,k,v,o 4096x4096; gate,up 11008x4096; down 4096x11008), LoRA r=64 alpha=16"
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a timed region."""

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- workloads

def build_decode_set(qn, device, layers: int, r: int, seed: int):
    """Quantise the decode set on the device (inputs drawn on the device)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    mats = []
    for layer in range(layers):
        for name, d, k in synth.DECODE_SHAPES:
            W = torch.empty((d, k), dtype=torch.float32, device=device)
            synth.device_normal_(W, 0.02, gen)
            synth.device_outliers_exact_(W, 0.001, 0.2, gen)
            q = qn.nf4_quantize(W, dq=True)
            del W
            A = torch.empty((r, k), device=device).normal_(0, 1 / math.sqrt(k), generator=gen).to(torch.bfloat16)
            B = torch.empty((d, r), device=device).normal_(0, 0.01, generator=gen).to(torch.bfloat16)
            mats.append((name, q, A, B))
    torch.cuda.synchronize()
    return mats


def time_decode(qn, mats, M, steps, warmup, ws, device, alpha=16.0):
    """Timed region: `steps` replays of a CUDA graph holding one pass over all
    matrices (two kernel launches per matrix).  Also times, per matrix shape,
    a graph of that shape's calls alone to get the mean duration of one call."""
    gen = torch.Generator(device=device)
    gen.manual_seed(101)
    xs = {}
    for _, q, _, _ in mats:
        if q.k not in xs:
            xs[q.k] = torch.randn((M, q.k), device=device, generator=gen).to(torch.bfloat16)
    outs = [torch.empty((M, q.d), dtype=torch.bfloat16, device=device) for _, q, _, _ in mats]

    def calls(sel):
        for i in sel:
            _, q, A, B = mats[i]
            qn.qlora_linear_fwd(q, xs[q.k], A, B, alpha, out=outs[i])

    def capture(sel):
        s = torch.cuda.Stream(device)
        s.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(s):
            calls(sel)                      # warm-up outside the graph
        torch.cuda.current_stream(device).wait_stream(s)
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            calls(sel)
        return g

    def timed(g, reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1)

    g_all = capture(range(len(mats)))
    for _ in range(warmup):
        g_all.replay()
    torch.cuda.synchronize(device)
    barrier(ws)
    total_ms = timed(g_all, steps)
    call_ms = {}
    by_shape = {}
    for i, (_, q, _, _) in enumerate(mats):
        by_shape.setdefault((q.d, q.k), []).append(i)
    for shp, sel in by_shape.items():
        g = capture(sel)
        g.replay()
        reps = max(2, steps // 2)
        call_ms[shp] = (timed(g, reps) / (reps * len(sel)), len(sel))
        del g
    return {"total_ms": total_ms, "call_ms": call_ms}


def decode_bytes(mats, M, r):
    w4 = sum(q.nbytes() for _, q, _, _ in mats)
    lora = sum(2 * r * (q.d + q.k) for _, q, _, _ in mats)
    act = sum(2 * M * (q.d + q.k) for _, q, _, _ in mats)
    return w4, lora, act


def time_e2e_decode(qn, mats, M, steps, warmup, device, alpha=16.0):
    """The same step through the public API with HOST buffers: X is copied
    from pinned host memory and Y read back to the host for every matrix."""
    xs = {}
    for _, q, _, _ in mats:
        if q.k not in xs:
            xs[q.k] = torch.randn((M, q.k)).to(torch.bfloat16).pin_memory()
    youts = [torch.empty((M, q.d), dtype=torch.bfloat16).pin_memory() for _, q, _, _ in mats]

    def one_step():
        for i, (_, q, A, B) in enumerate(mats):
            qn.qlora_linear_fwd(q, xs[q.k], A, B, alpha, out=youts[i])

    for _ in range(warmup):
        one_step()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        one_step()
    t1.record()
    torch.cuda.synchronize()
    h2d = sum(2 * M * q.k for _, q, _, _ in mats)
    d2h = sum(2 * M * q.d for _, q, _, _ in mats)
    return t0.elapsed_time(t1), h2d, d2h


def secondary(qn, device, pk, quick: bool):
    """Prefill TFLOP/s, bulk quantise/dequantise GB/s, LoftQ s/alternation."""
    out = {}
    # prefill layer: forward and backward dX
    c_d, c_k, M, r, alpha = 11008, 4096, 4096, 16, 32.0
    gen = torch.Generator(device=device)
    gen.manual_seed(2)
    W = torch.empty((c_d, c_k), device=device).normal_(0, 0.02, generator=gen)
    q = qn.nf4_quantize(W, dq=True)
    del W
    X = torch.randn((M, c_k), device=device, generator=gen).to(torch.bfloat16)
    dY = torch.randn((M, c_d), device=device, generator=gen).to(torch.bfloat16)
    A = torch.empty((r, c_k), device=device).normal_(0, 1 / math.sqrt(c_k), generator=gen).to(torch.bfloat16)
    B = torch.empty((c_d, r), device=device).normal_(0, 0.01, generator=gen).to(torch.bfloat16)
    flops = 2 * M * c_d * c_k + 2 * M * r * (c_k + c_d)
    for name, fn in (("prefill_fwd", lambda: qn.qlora_linear_fwd(q, X, A, B, alpha)),
                     ("prefill_bwd_dx", lambda: qn.qlora_linear_bwd_dx(q, dY, A, B, alpha))):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        reps = 3 if quick else 10
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        tf = flops / (ms * 1e-3) / 1e12
        out[name] = {"ms": ms, "tflops": tf, "frac_of_bf16_peak": tf / pk["bf16_tflops"],
                     "workload": "M=4096, d=11008, k=4096, r=16, alpha=32"}
    del X, dY, q

    # bulk quantise / dequantise of the 32-layer bf16 set (one tensor per call)
    layers = 4 if quick else 32
    gen.manual_seed(3)
    srcs = []
    for _ in range(layers):
        for _, d, k in synth.DECODE_SHAPES:
            t = torch.empty((d, k), dtype=torch.bfloat16, device=device)
            synth.device_normal_(t, 0.02, gen)
            synth.device_outliers_bernoulli_(t, 0.001, 0.2, gen)
            srcs.append(t)
    qs = [qn.NF4Tensor.empty(t.shape[0], t.shape[1], True, device) for t in srcs]
    deq = [torch.empty_like(t) for t in srcs]
    n_params = sum(t.numel() for t in srcs)
    qbytes = sum(2 * t.numel() + qq.nbytes() for t, qq in zip(srcs, qs))
    for name, fn, nbytes in (
            ("quantize", lambda: [qn.nf4_quantize(t, True, out=qq) for t, qq in zip(srcs, qs)], qbytes),
            ("dequantize", lambda: [qn.nf4_dequantize(qq, torch.bfloat16, out=o) for qq, o in zip(qs, deq)], qbytes)):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 2
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": ms, "gbs": gbs, "frac_of_hbm": gbs / pk["hbm_gbs"], "params": n_params,
                     "bytes": nbytes, "workload": f"{layers} layers x 7 bf16 matrices, NF4+DQ"}
    del srcs, qs, deq

    # LoftQ
    Wl = torch.from_numpy(synth.loftq_case(seed=4)).to(device)
    T = 2 if quick else 5
    qn.loftq_init(Wl, r=16, alpha=16.0, T=1)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    _, _, _, resid = qn.loftq_init(Wl, r=16, alpha=16.0, T=T, seed=0, oversample=8, power_iters=4)
    dt = time.perf_counter() - t0
    out["loftq"] = {"s_per_alternation": dt / T, "T": T, "resid": resid,
                    "workload": "4096x4096 Student-t, r=16, oversample 8, 4 power iterations"}
    return out


# ------------------------------------------------------------ oracle timing

def oracle_decode_sample(seconds_budget: float = 15.0):
    """Oracle (CPU, float64) forward of sampled decode matrices at M=1:
    dequantise from its own NF4 state + the float64 product.  Returns the
    metric (GB/s of 4-bit weight bytes) and a description."""
    from oracle import layer, nf4
    m = synth.decode_matrix(seed=1, d=4096, k=4096, r=64, M=1)
    t = nf4.quantize(m["W"], 64, dq=True)                  # setup, untimed
    nbytes = nf4.storage_bytes(4096 * 4096)
    X = m["X"].float().numpy()
    A = m["A"].float().numpy()
    B = m["B"].float().numpy()
    reps, el = 0, 0.0
    while el < seconds_budget and reps < 50:
        t0 = time.perf_counter()
        Wd = nf4.dequantize(t).reshape(4096, 4096)
        layer.linear_fwd(X, Wd, A, B, 16.0, 64)
        el += time.perf_counter() - t0
        reps += 1
    return nbytes * reps / el / 1e9, reps, el


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# --------------------------------------------------------------------- main

def run_reference(args, ws, rank):
    if rank != 0:
        return
    from oracle import layer, nf4
    m = synth.decode_matrix(seed=1, d=4096, k=4096, r=64, M=1)
    t = nf4.quantize(m["W"], 64, dq=True)
    X, A, B = (m[n].float().numpy() for n in ("X", "A", "B"))
    nbytes = nf4.storage_bytes(4096 * 4096)

    def step():
        Wd = nf4.dequantize(t).reshape(4096, 4096)
        layer.linear_fwd(X, Wd, A, B, 16.0, 64)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = nbytes * args.steps / el / 1e9
    sample = "one 4096x4096 decode matrix per step (M=1, r=64): oracle dequantise + float64 product"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--quick", action="store_true", help="shorter secondary loops")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    ws, rank, local = dist_env()

    if args.impl == "reference":
        run_reference(args, ws, rank)
        return

    if ws > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import bit_nf4_quantized_39_b300 as qn
    pk = peaks()
    r = 64
    mats = build_decode_set(qn, device, args.layers, r, seed=1 + rank)

    with ClockSampler(local) as clk:
        res = time_decode(qn, mats, 1, args.steps, args.warmup, ws, device)
    clocks = clk.summary()
    total_ms = max_over_ranks(res["total_ms"], ws)
    w4, lora, act = decode_bytes(mats, 1, r)
    value = w4 * args.steps * ws / (total_ms * 1e-3) / 1e9

    # roofline of the dominant call (the fused M=1 forward of one matrix),
    # per shape: algorithmic bytes / mean CUDA-event duration of one call
    # (from graphs of that shape's calls back to back).
    shapes, tot_bytes, tot_ms = {}, 0.0, 0.0
    for (d, k), (ms, cnt) in res["call_ms"].items():
        q0 = next(q for _, q, _, _ in mats if (q.d, q.k) == (d, k))
        byt = q0.nbytes() + 2 * r * (d + k) + 2 * (d + k) + 4 * r
        shapes[f"{d}x{k}"] = {"us": ms * 1e3, "bytes": byt, "gbs": byt / (ms * 1e-3) / 1e9, "calls": cnt}
        tot_bytes += byt * cnt
        tot_ms += ms * cnt
    achieved = tot_bytes / (tot_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "traffic": None,
                "kernel": "qlora_linear_fwd at M=1 (lora_proj + fused NF4 GEMV), per call",
                "peak_source": pk["source"], "per_shape": shapes}

    e2e_ms, h2d, d2h = time_e2e_decode(qn, mats, 1, max(2, args.steps // 2), 2, device)
    e2e_steps = max(2, args.steps // 2)
    e2e = {"value": w4 * e2e_steps / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h}

    extra = {}
    if rank == 0:
        r16 = time_decode(qn, mats, 16, max(3, args.steps // 2), 2, 1, device)
        extra["decode_M16"] = {"gbs": w4 * max(3, args.steps // 2) / (r16["total_ms"] * 1e-3) / 1e9,
                               "unit": "GB/s of 4-bit weight bytes"}
    del mats
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_secondary:
        extra.update(secondary(qn, device, pk, args.quick))

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, reps, el = oracle_decode_sample()
        cpu = {"value": v, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{reps} forward(s) of one 4096x4096 decode matrix at M=1 ({el:.1f} s): "
                         "oracle dequantise + float64 product", "blas_threads": torch.get_num_threads()}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded device draws: N(0,0.02^2) weights with 0.1% N(0,0.2^2) outliers)",
                "config": {"workload": WORKLOAD, "M": 1, "layers": args.layers, "matrices": 7 * args.layers,
                           "weight_bytes_per_step": w4, "lora_bytes_per_step": lora,
                           "l2": "no flush: 3.34 GB weight set per step >> 126 MB L2",
                           "parallelism": f"replica x{ws}"},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": 2 * 7 * args.layers * args.steps, "clocks": clocks, "secondary": extra}
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
