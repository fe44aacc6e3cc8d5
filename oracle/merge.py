"""Merge / unmerge of a LoRA adapter into an NF4 weight (test infrastructure only).

"PEFT quantization guide" (huggingface docs, 量化), section on merging
adapters into quantised weights: merging dequantises the base weight, adds
the adapter weight and quantises the result again; unmerging does the
reverse (dequantise, subtract, requantise), so it does not give back the
original quantised weight, and repeated merge/unmerge cycles can accumulate
rounding error.  "LoftQ explainer" §5.2 uses the same operation to export a
merged model.

With the layer's adapter scale s = alpha / r ("PEFT course notes" §2.2 and
§2.4) and sign = +1 (merge) or -1 (unmerge):

    W'' = NF4( deq(Q) + sign * s * B A )

READINGS (the pages give no precision for the sum):
* A (r x k) and B (d x r) are the layer's bf16 adapter factors.  The product
  of two bf16 values has at most 16 significant bits, so every term
  B[i, q] * A[q, j] is exact in fp32.
* (B A)[i, j] is accumulated in fp32 in ascending q, one rounding per
  addition; then t = fp32(s * (B A)[i, j]) and W''_pre = fp32(deq + sign * t)
  (each step rounded once, no fused multiply-add).
* The requantisation is the same NF4 quantiser as everywhere else, with
  double quantisation when the input Q has it.
"""

from __future__ import annotations

import numpy as np

from . import nf4


def _check_bf16_values(a: np.ndarray, name: str) -> np.ndarray:
    a32 = np.ascontiguousarray(a, dtype=np.float32)
    if np.any(a32.view(np.uint32) & 0xFFFF):
        raise ValueError(f"{name} must hold bf16 values (the layer's adapter dtype)")
    return a32


def adapter_product_f32(A, B) -> np.ndarray:
    """(B A) in fp32: terms exact, summed in ascending rank order."""
    A32 = _check_bf16_values(A, "A")
    B32 = _check_bf16_values(B, "B")
    r = A32.shape[0]
    acc = np.zeros((B32.shape[0], A32.shape[1]), dtype=np.float32)
    for q in range(r):
        term = np.multiply(B32[:, q][:, None], A32[q, :][None, :], dtype=np.float32)  # exact
        acc = np.add(acc, term, dtype=np.float32)
    return acc


def merged_weight(Q: nf4.NF4Tensor, d: int, k: int, A, B, alpha: float, r: int, sign: int = 1) -> np.ndarray:
    """fp32 weight before requantisation: fp32(deq(Q) + sign * fp32(s * (B A)))."""
    if sign not in (1, -1):
        raise ValueError("sign must be +1 (merge) or -1 (unmerge)")
    s = np.float32(np.float32(alpha) / np.float32(r))
    t = np.multiply(s, adapter_product_f32(A, B), dtype=np.float32)
    base = nf4.dequantize(Q).reshape(d, k)
    if sign > 0:
        return np.add(base, t, dtype=np.float32)
    return np.subtract(base, t, dtype=np.float32)


def merge(Q: nf4.NF4Tensor, d: int, k: int, A, B, alpha: float, r: int, sign: int = 1) -> nf4.NF4Tensor:
    """NF4(deq(Q) + sign * s * B A) with the input's block sizes and DQ setting."""
    W = merged_weight(Q, d, k, A, B, alpha, r, sign)
    return nf4.quantize(W, Q.block, Q.dq, Q.dq_block)
