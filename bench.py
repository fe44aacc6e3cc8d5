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
dX in TFLOP/s, the adapter gradients dA, dB of that layer in GB/s, the
fp32-compute forward, merge of the adapter into the NF4 weight, bulk NF4
quantise / dequantise of the 6.48 B-parameter bf16 set in GB/s, and LoftQ
(4096 x 4096, r = 16, T = 5) seconds per alternation plus its one-step
variant.

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
WORKLOAD = ("llama7b-decode-set M=1: 32 layers x 7 NF4+DQ matrices (q,k,v,o 4096x4096; gate,up 11008x4096; "
            "down 4096x11008), LoRA r=64 alpha=16; per layer 4 calls: grouped q/k/v, o, grouped gate/up, down")
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


# DRAM bytes (read + write) per launch of qlora_gemv_kernel for each kind of
# decode call, from one ncu capture (`ncu --set full --clock-control none -k
# regex:qlora_gemv -s 4 -c 4 python bench.py --profile decode`).  They hold
# for the kernel source they were taken on (its sha256); for any other source
# the bench reports traffic as null.
GEMV_TRAFFIC_SHA256 = "27ae316811226d4aa612fe6ba3790093755e205b5cb5c181514abc29149d2729"
GEMV_TRAFFIC = {"qkv": 29197056, "o": 9789696, "gate_up": 50473728 + 69120, "down": 25294080}


def gemv_traffic(per_kind):
    """Launch-weighted DRAM bytes per launch, or None if the kernel changed."""
    import hashlib
    src = os.path.join(ROOT, "bit_nf4_quantized_39_b300", "csrc", "qlora_gemv.cuh")
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != GEMV_TRAFFIC_SHA256:
            return None
    n = sum(v["launches"] for v in per_kind.values())
    return sum(GEMV_TRAFFIC[k] * v["launches"] for k, v in per_kind.items()) / n


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
    """Largest x over the ranks (the timed region ends when the slowest rank does)."""
    if ws == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(bytes_per_step_per_rank: float, steps: int, ws: int, total_ms: float) -> float:
    """Whole-job GB/s: the bytes every rank processed over the slowest rank's time."""
    return bytes_per_step_per_rank * steps * ws / (total_ms * 1e-3) / 1e9


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


GROUPS = [("qkv", ["q_proj", "k_proj", "v_proj"]), ("o", ["o_proj"]), ("gate_up", ["gate_proj", "up_proj"]),
          ("down", ["down_proj"])]


def decode_plan(mats, layers, M, device, seed=101):
    """Calls of one decode step: per layer, the projections that share an
    input run as one grouped call (q/k/v, gate/up), o and down alone.  Every
    call reads its input from one packed X buffer and writes into one packed
    Y buffer, so a step's host<->device traffic is one copy each way."""
    by = {}
    for i, (name, q, A, B) in enumerate(mats):
        by.setdefault(i // 7, {})[name] = (q, A, B)
    calls, xoff, yoff = [], 0, 0
    for layer in range(layers):
        for gname, names in GROUPS:
            members = [by[layer][n] for n in names]
            k = members[0][0].k
            calls.append(dict(kind=gname, qs=[m[0] for m in members], As=[m[1] for m in members],
                              Bs=[m[2] for m in members], k=k, xoff=xoff,
                              youts=[(yoff + sum(mm[0].d for mm in members[:j]), m[0].d) for j, m in enumerate(members)]))
            xoff += M * k
            yoff += sum(m[0].d for m in members)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    Xall = torch.randn(xoff, device=device, generator=gen).to(torch.bfloat16)
    Yall = torch.empty(yoff * M, dtype=torch.bfloat16, device=device)
    return calls, Xall, Yall


def run_calls(qn, calls, Xall, Yall, M, alpha=16.0, sel=None):
    for c in (calls if sel is None else [calls[i] for i in sel]):
        X = Xall[c["xoff"]:c["xoff"] + M * c["k"]].view(M, c["k"])
        outs = [Yall[o * M:(o + d) * M].view(M, d) for o, d in c["youts"]]
        qn.qlora_linear_fwd_group(c["qs"], X, c["As"], c["Bs"], [alpha] * len(c["qs"]), outs=outs)


def capture(device, fn):
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        fn()                      # warm-up outside the graph
    torch.cuda.current_stream(device).wait_stream(s)
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def timed_replays(device, g, reps, pre=None, post=None):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e0.record()
    for _ in range(reps):
        if pre is not None:
            pre()
        g.replay()
        if post is not None:
            post()
    e1.record()
    torch.cuda.synchronize(device)
    return e0.elapsed_time(e1)


def time_decode(qn, mats, layers, M, steps, warmup, ws, device):
    """Timed region: `steps` replays of a CUDA graph holding one decode step.
    Also times, per kind of call, a graph of that kind's calls alone to get
    the mean duration of one launch."""
    calls, Xall, Yall = decode_plan(mats, layers, M, device)
    g_all = capture(device, lambda: run_calls(qn, calls, Xall, Yall, M))
    for _ in range(warmup):
        g_all.replay()
    torch.cuda.synchronize(device)
    barrier(ws)
    total_ms = timed_replays(device, g_all, steps)
    per_kind = {}
    for kind, _ in GROUPS:
        sel = [i for i, c in enumerate(calls) if c["kind"] == kind]
        g = capture(device, lambda: run_calls(qn, calls, Xall, Yall, M, sel=sel))
        g.replay()
        reps = max(2, steps // 2)
        ms = timed_replays(device, g, reps) / (reps * len(sel))
        c0 = calls[sel[0]]
        w4 = sum(q.nbytes() for q in c0["qs"])
        byt = w4 + sum(2 * A.shape[0] * (q.d + q.k) for q, A in zip(c0["qs"], c0["As"])) \
            + 2 * M * c0["k"] + sum(2 * M * q.d for q in c0["qs"])
        per_kind[kind] = {"us": ms * 1e3, "bytes": byt, "weight_bytes": w4, "gbs": byt / (ms * 1e-3) / 1e9,
                          "launches": len(sel)}
        del g
    # end to end: host inputs in, host outputs out, every step
    Xh = torch.empty(Xall.shape, dtype=Xall.dtype, pin_memory=True).copy_(Xall.cpu())
    Yh = torch.empty(Yall.shape, dtype=Yall.dtype, pin_memory=True)
    e2e_steps = max(2, steps // 2)
    e2e_ms = timed_replays(device, g_all, e2e_steps, pre=lambda: Xall.copy_(Xh, non_blocking=True),
                           post=lambda: Yh.copy_(Yall, non_blocking=True))
    h2d, d2h = Xall.numel() * 2, Yall.numel() * 2
    return {"total_ms": total_ms, "per_kind": per_kind, "e2e_ms": e2e_ms, "e2e_steps": e2e_steps, "h2d": h2d,
            "d2h": d2h, "launches_per_step": len(calls)}


def decode_bytes(mats, M, r):
    w4 = sum(q.nbytes() for _, q, _, _ in mats)
    lora = sum(2 * r * (q.d + q.k) for _, q, _, _ in mats)
    act = sum(2 * M * (q.d + q.k) for _, q, _, _ in mats)
    return w4, lora, act


# fp32 FMA peak of the CUDA cores: 148 SMs x 128 lanes x 2 flops x 2.032 GHz
FP32_FMA_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


def _time_call(fn, reps):
    """Mean CUDA-event time of `reps` back-to-back calls after two warm-up calls."""
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return {"ms": e0.elapsed_time(e1) / reps}


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
    # adapter gradients at the prefill shape: HBM bound (X and dY read once)
    reps = 3 if quick else 10
    grad_bytes = 2 * M * (c_k + c_d) + 2 * r * (c_k + c_d) + 4 * r * (c_k + c_d)
    out["lora_grads"] = _time_call(lambda: qn.qlora_linear_bwd_lora(X, dY, A, B, alpha), reps)
    out["lora_grads"].update(gbs=grad_bytes / (out["lora_grads"]["ms"] * 1e-3) / 1e9, bytes=grad_bytes,
                             workload="dA, dB at M=4096, d=11008, k=4096, r=16 (algorithmic bytes: X, dY, A, B "
                                      "read, dA, dB written)")
    out["lora_grads"]["frac_of_hbm"] = out["lora_grads"]["gbs"] / pk["hbm_gbs"]
    # fp32 compute dtype: prefill-shaped forward (CUDA-core fp32 FMA) and one decode matrix
    Xf, Af, Bf = X.float(), A.float(), B.float()
    out["fp32_fwd"] = _time_call(lambda: qn.qlora_linear_fwd_f32(q, Xf, Af, Bf, alpha), max(2, reps // 2))
    tf = flops / (out["fp32_fwd"]["ms"] * 1e-3) / 1e12
    out["fp32_fwd"].update(tflops=tf, frac_of_fp32_peak=tf / FP32_FMA_TFLOPS,
                           workload="fp32 compute dtype, M=4096, d=11008, k=4096, r=16; CUDA-core FMA")
    del Xf
    x1 = torch.randn((1, c_k), device=device, generator=gen)
    out["fp32_fwd_m1"] = _time_call(lambda: qn.qlora_linear_fwd_f32(q, x1, Af, Bf, alpha), reps)
    out["fp32_fwd_m1"]["gbs"] = q.nbytes() / (out["fp32_fwd_m1"]["ms"] * 1e-3) / 1e9
    out["fp32_fwd_m1"]["workload"] = "fp32 compute dtype, M=1, 11008 x 4096 (GB/s of 4-bit weight bytes)"
    # merge / unmerge of the adapter into the quantised weight
    qo = qn.NF4Tensor.empty(c_d, c_k, True, device)
    merge_bytes = 2 * q.nbytes() + 2 * r * (c_k + c_d)
    out["merge"] = _time_call(lambda: qn.nf4_merge_lora(q, A, B, alpha, 1, out=qo), reps)
    out["merge"].update(gbs=merge_bytes / (out["merge"]["ms"] * 1e-3) / 1e9, bytes=merge_bytes,
                        workload="NF4+DQ 11008 x 4096, r=16: deq + s B A + requantise (state read and written)")
    out["merge"]["frac_of_hbm"] = out["merge"]["gbs"] / pk["hbm_gbs"]
    del X, dY, qo

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
    def graph_of(fn):
        st = torch.cuda.Stream(device)
        st.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(st):
            fn()
        torch.cuda.current_stream(device).wait_stream(st)
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    for name, fn, nbytes in (
            ("quantize", lambda: [qn.nf4_quantize(t, True, out=qq) for t, qq in zip(srcs, qs)], qbytes),
            ("dequantize", lambda: [qn.nf4_dequantize(qq, torch.bfloat16, out=o) for qq, o in zip(qs, deq)], qbytes)):
        g = graph_of(fn)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 3
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": ms, "gbs": gbs, "frac_of_hbm": gbs / pk["hbm_gbs"], "params": n_params,
                     "bytes": nbytes, "workload": f"{layers} layers x 7 bf16 matrices, NF4+DQ, one CUDA graph"}
        del g
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
    q0 = qn.nf4_quantize(Wl)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    _, _, res1 = qn.loftq_replace_lora(Wl, q0, 16, 16.0, seed=0)
    out["loftq_one_step"] = {"s": time.perf_counter() - t0, "resid": res1,
                             "workload": "4096x4096 Student-t, r=16, one Delta-step against NF4(W)"}
    return out


# ------------------------------------------------------------ profiling cases

def profile_case(case: str):
    """Untimed runs for ncu: `decode` / `decode16` = one layer of the decode set
    (4 calls: q/k/v, o, gate/up, down) at M = 1 / 16, three times; `prefill` =
    the prefill layer forward and backward, three times; `loftq` = one LoftQ
    alternation (T = 1, r = 16) of a 1024 x 1024 matrix, twice (`loftq4096`: of
    a 4096 x 4096 matrix, once); `quantize` =
    NF4+DQ quantise and dequantise of one 11008 x 4096 bf16 matrix, three times."""
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    import bit_nf4_quantized_39_b300 as qn
    if case in ("decode", "decode16"):
        M = 1 if case == "decode" else 16
        mats = build_decode_set(qn, device, 1, 64, seed=1)
        calls, Xall, Yall = decode_plan(mats, 1, M, device)
        for _ in range(3):
            run_calls(qn, calls, Xall, Yall, M)
    elif case == "prefill":
        gen = torch.Generator(device=device)
        gen.manual_seed(2)
        c_d, c_k, M, r = 11008, 4096, 4096, 16
        W = torch.empty((c_d, c_k), device=device).normal_(0, 0.02, generator=gen)
        q = qn.nf4_quantize(W, dq=True)
        X = torch.randn((M, c_k), device=device, generator=gen).to(torch.bfloat16)
        dY = torch.randn((M, c_d), device=device, generator=gen).to(torch.bfloat16)
        A = torch.empty((r, c_k), device=device).normal_(0, 1 / math.sqrt(c_k), generator=gen).to(torch.bfloat16)
        B = torch.empty((c_d, r), device=device).normal_(0, 0.01, generator=gen).to(torch.bfloat16)
        for _ in range(3):
            qn.qlora_linear_fwd(q, X, A, B, 32.0)
            qn.qlora_linear_bwd_dx(q, dY, A, B, 32.0)
    elif case in ("loftq", "loftq4096"):
        n = 1024 if case == "loftq" else 4096
        W = torch.from_numpy(synth.loftq_case(seed=4, d=n, k=n)).to(device)
        for _ in range(2 if case == "loftq" else 1):
            qn.loftq_init(W, r=16, alpha=16.0, T=1, seed=0, oversample=8, power_iters=4)
    else:
        gen = torch.Generator(device=device)
        gen.manual_seed(3)
        t = torch.empty((11008, 4096), dtype=torch.bfloat16, device=device)
        synth.device_normal_(t, 0.02, gen)
        synth.device_outliers_bernoulli_(t, 0.001, 0.2, gen)
        qq = qn.NF4Tensor.empty(t.shape[0], t.shape[1], True, device)
        out = torch.empty_like(t)
        for _ in range(3):
            qn.nf4_quantize(t, True, out=qq)
            qn.nf4_dequantize(qq, torch.bfloat16, out=out)
    torch.cuda.synchronize()
    qn.device_status()
    print(json.dumps({"profile": case, "ok": True}))


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
    ap.add_argument("--profile", choices=["decode", "decode16", "prefill", "quantize", "loftq", "loftq4096"],
                    help="run one small case of a workload a few times, untimed (for ncu captures)")
    args = ap.parse_args()
    ws, rank, local = dist_env()

    if args.profile:
        profile_case(args.profile)
        return

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
        res = time_decode(qn, mats, args.layers, 1, args.steps, args.warmup, ws, device)
    clocks = clk.summary()
    total_ms = max_over_ranks(res["total_ms"], ws)
    w4, lora, act = decode_bytes(mats, 1, r)
    value = job_value(w4, args.steps, ws, total_ms)

    # roofline of the dominant kernel (qlora_gemv_kernel, one launch per
    # call): algorithmic bytes per launch / mean CUDA-event launch duration,
    # weighted over the four kinds of call of a decode step.
    tot_bytes = sum(v["bytes"] * v["launches"] for v in res["per_kind"].values())
    tot_s = sum(v["us"] * 1e-6 * v["launches"] for v in res["per_kind"].values())
    achieved = tot_bytes / tot_s / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "traffic": gemv_traffic(res["per_kind"]),
                "kernel": "qlora_gemv_kernel (M=1; 4-bit weight + block constants + LoRA A, B + x + y bytes "
                          "per launch)",
                "peak_source": pk["source"], "per_call": res["per_kind"]}
    e2e = {"value": w4 * res["e2e_steps"] / (res["e2e_ms"] * 1e-3) / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
           "how": "per step: one pinned-host->device copy of all inputs, the graph of public-API calls, "
                  "one device->pinned-host copy of all outputs"}

    extra = {}
    if rank == 0:
        r16 = time_decode(qn, mats, args.layers, 16, max(3, args.steps // 2), 2, 1, device)
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
                           "arith": "NF4 levels as bf16 (byte-pair table) x bf16 x on mma.sync, fp32 block "
                                    "sums scaled by fp32 block constants, fp32 accumulation; bf16 y",
                           "parallelism": f"replica x{ws}"},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": res["launches_per_step"] * args.steps, "clocks": clocks, "secondary": extra}
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
