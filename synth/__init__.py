"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers with fixed seeds and rounds them to the
input dtypes; it holds none of the method's arithmetic.  Both the CUDA path
and the oracle consume its outputs.  Host draws use numpy's PCG64
(``numpy.random.default_rng(seed)``); the multi-gigabyte bench sets are drawn
on the device with ``torch.Generator('cuda')`` seeded the same way.

Workloads (shapes and distributions of the single-layer, decode, prefill,
bulk-quantisation and LoftQ cases):

* layer case:   W 1024x1024 fp32 N(0, 0.02^2); X 16x1024 bf16 N(0,1);
                r=8, alpha=16; A 8x1024 N(0, 1/1024); B 1024x8 N(0, 0.01^2).
* decode set:   Llama-7B projections q/k/v/o 4096x4096, gate/up 11008x4096,
                down 4096x11008; W N(0, 0.02^2) with exactly floor(0.001 n)
                entries, chosen without replacement, redrawn from N(0, 0.2^2);
                X bf16 N(0,1) with M in {1, 16}; r=64, alpha=16.
* prefill case: W 11008x4096 N(0, 0.02^2); X 4096x4096 bf16 N(0,1);
                dY 4096x11008 bf16 N(0,1); r=16, alpha=32.
* bulk set:     32 layers x the 7 decode shapes, bf16 N(0, 0.02^2) with
                Bernoulli(0.001) outliers from N(0, 0.2^2).
* LoftQ case:   W 4096x4096 fp32 Student-t(df=4) scaled to std 0.02
                (t_4 has variance 2, so the draw is multiplied by 0.02/sqrt 2);
                T=5, r=16.
"""

from __future__ import annotations

import math

import numpy as np
import torch

DECODE_SHAPES = [  # (name, d, k): W is d x k, Y = X W^T
    ("q_proj", 4096, 4096), ("k_proj", 4096, 4096), ("v_proj", 4096, 4096),
    ("o_proj", 4096, 4096), ("gate_proj", 11008, 4096), ("up_proj", 11008, 4096),
    ("down_proj", 4096, 11008),
]
N_LAYERS = 32


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """Round a float array to a CPU bf16 tensor (input dtype conversion)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def normal(g: np.random.Generator, shape, std: float) -> np.ndarray:
    return (g.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def with_outliers_exact(g: np.random.Generator, W: np.ndarray, frac: float, std: float) -> np.ndarray:
    """Replace exactly floor(frac * n) entries, chosen without replacement, by N(0, std^2)."""
    flat = W.reshape(-1)
    cnt = int(math.floor(frac * flat.size))
    if cnt:
        idx = g.choice(flat.size, size=cnt, replace=False)
        flat[idx] = normal(g, cnt, std)
    return W


def lora_factors(g: np.random.Generator, d: int, k: int, r: int):
    """A (r x k) ~ N(0, 1/k) and B (d x r) ~ N(0, 0.01^2), both rounded to bf16."""
    A = normal(g, (r, k), 1.0 / math.sqrt(k))
    B = normal(g, (d, r), 0.01)
    return to_bf16(A), to_bf16(B)


def layer_case(seed: int = 0, d: int = 1024, k: int = 1024, M: int = 16, r: int = 8,
               alpha: float = 16.0) -> dict:
    """Single-layer case (defaults: the 1024x1024 reference layer, seed 0)."""
    g = rng(seed)
    W = normal(g, (d, k), 0.02)
    X = to_bf16(g.standard_normal((M, k), dtype=np.float32))
    A, B = lora_factors(g, d, k, r)
    dY = to_bf16(g.standard_normal((M, d), dtype=np.float32))
    return dict(W=W, X=X, A=A, B=B, dY=dY, r=r, alpha=alpha, d=d, k=k, M=M)


def decode_matrix(seed: int, d: int, k: int, r: int = 64, M: int = 1) -> dict:
    """One decode-set matrix with its outliers, X (M x k) and LoRA factors, on the host."""
    g = rng(seed)
    W = with_outliers_exact(g, normal(g, (d, k), 0.02), 0.001, 0.2)
    X = to_bf16(g.standard_normal((M, k), dtype=np.float32))
    A, B = lora_factors(g, d, k, r)
    return dict(W=W, X=X, A=A, B=B, r=r, alpha=16.0, d=d, k=k, M=M)


def prefill_case(seed: int = 2, d: int = 11008, k: int = 4096, M: int = 4096,
                 r: int = 16, alpha: float = 32.0) -> dict:
    g = rng(seed)
    W = normal(g, (d, k), 0.02)
    X = to_bf16(g.standard_normal((M, k), dtype=np.float32))
    A, B = lora_factors(g, d, k, r)
    dY = to_bf16(g.standard_normal((M, d), dtype=np.float32))
    return dict(W=W, X=X, A=A, B=B, dY=dY, r=r, alpha=alpha, d=d, k=k, M=M)


def loftq_case(seed: int = 4, d: int = 4096, k: int = 4096) -> np.ndarray:
    """Student-t (df=4) weights scaled to standard deviation 0.02."""
    g = rng(seed)
    t = g.standard_t(4, size=(d, k))
    return (t * (0.02 / math.sqrt(2.0))).astype(np.float32)


def adversarial_block_values(seed: int, cb: np.ndarray, nblocks: int) -> np.ndarray:
    """Blocks built from given levels: exact codebook multiples, near-level
    perturbations by a few ulps, zero blocks, single non-zeros and negative
    absmax.  ``cb`` is whatever 16-level table the caller supplies; no
    quantiser arithmetic happens here."""
    g = rng(seed)
    out = []
    for b in range(nblocks):
        kind = b % 5
        scale = np.float32(10.0 ** g.uniform(-4, 1))
        if kind == 0:
            idx = g.integers(0, 16, 64)
            idx[0] = 15
            out.append((cb[idx] * scale).astype(np.float32))
        elif kind == 1:
            idx = g.integers(0, 16, 64)
            idx[0] = 0
            v = (cb[idx] * scale).astype(np.float32)
            ulps = g.integers(-3, 4, 64).astype(np.int32)
            ulps[v == 0] = 0                      # keep exact zeros (no sign crossing)
            bits = v.view(np.int32) + ulps        # same-sign neighbours of the level multiples
            v = bits.view(np.float32)
            v[0] = -scale
            out.append(v)
        elif kind == 2:
            out.append(np.zeros(64, dtype=np.float32))
        elif kind == 3:
            v = np.zeros(64, dtype=np.float32)
            v[g.integers(0, 64)] = np.float32(g.choice([-1.0, 1.0])) * scale
            out.append(v)
        else:
            out.append(normal(g, 64, float(scale)))
    return np.concatenate(out)


def near_point_blocks(seed: int, points: np.ndarray, nblocks: int, max_ulps: int = 4) -> np.ndarray:
    """Blocks whose normalised values sit on or a few ulps around given points.

    Each 64-element block gets a random scale m; element 0 is +-m (so the
    block absmax is m) and the others are fp32(p * m) moved by up to
    ``max_ulps`` ulps, for points p drawn from ``points`` (the caller passes
    the decision boundaries it wants exercised)."""
    g = rng(seed)
    pts = np.asarray(points, dtype=np.float32)
    out = []
    for _ in range(nblocks):
        m = np.float32(10.0 ** g.uniform(-5, 2))
        p = pts[g.integers(0, pts.size, 64)]
        v = (p * m).astype(np.float32)
        ulps = g.integers(-max_ulps, max_ulps + 1, 64).astype(np.int32)
        ulps[v == 0] = 0
        v = (v.view(np.int32) + ulps).view(np.float32)
        v = np.clip(v, -m, m).astype(np.float32)
        v[0] = m if g.integers(0, 2) else -m
        out.append(v)
    return np.concatenate(out)


# ---- device-side generators for the multi-gigabyte bench sets ----------------

def device_normal_(t: torch.Tensor, std: float, gen: torch.Generator) -> torch.Tensor:
    return t.normal_(0.0, std, generator=gen)


def device_outliers_exact_(t: torch.Tensor, frac: float, std: float, gen: torch.Generator) -> torch.Tensor:
    flat = t.view(-1)
    cnt = int(math.floor(frac * flat.numel()))
    if cnt:
        idx = torch.randperm(flat.numel(), device=t.device, generator=gen)[:cnt]
        flat[idx] = torch.empty(cnt, device=t.device, dtype=t.dtype).normal_(0.0, std, generator=gen)
    return t


def device_outliers_bernoulli_(t: torch.Tensor, p: float, std: float, gen: torch.Generator) -> torch.Tensor:
    flat = t.view(-1)
    mask = torch.empty(flat.numel(), device=t.device, dtype=torch.float32).uniform_(generator=gen) < p
    draws = torch.empty(flat.numel(), device=t.device, dtype=t.dtype).normal_(0.0, std, generator=gen)
    flat.copy_(torch.where(mask, draws, flat))
    return t
