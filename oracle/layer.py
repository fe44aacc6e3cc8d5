"""QLoRA linear layer oracle in float64 (test infrastructure only).

"PEFT course notes" §2.2: the frozen weight W in R^{d x k} plus the low-rank
update BA with B in R^{d x r}, A in R^{r x k}; the output is h = Wx + BAx.
"QLoRA paper summary" (abstract): the frozen weight is the 4-bit quantised
one, and gradients are back-propagated through it into the adapter.
READING: the adapter is scaled by s = alpha / r (lora_alpha is the scaling
factor of "PEFT course notes" §2.4); rows of X are tokens, so for a batch
X in R^{M x k}:

    Y  = X W'^T + s (X A^T) B^T                       (M x d)
    dX = dY W'  + s (dY B) A                          (M x k)
    dB = s dY^T (X A^T)                               (d x r)
    dA = s (dY B)^T X                                 (r x k)

dA and dB are the gradients of a loss L with dL/dY = dY with respect to the
adapter factors, the part of the backward pass that reaches the trainable
weights ("QLoRA paper summary", abstract: gradients are back-propagated
through the frozen 4-bit weight into the low-rank adapters).

where W' is the fp32 dequantised weight.  Every operand is widened exactly
to float64 and each product is one numpy matmul (a library primitive).
"""

from __future__ import annotations

import numpy as np


def lora_param_count(d: int, k: int, r: int) -> int:
    """Trainable adapter parameters: B is d x r, A is r x k ("PEFT course notes" §2.2)."""
    return (d + k) * r


def linear_fwd(X, Wdeq, A, B, alpha: float, r: int) -> np.ndarray:
    """Y = X W'^T + (alpha/r) (X A^T) B^T in float64."""
    X64 = np.asarray(X, dtype=np.float64)
    W64 = np.asarray(Wdeq, dtype=np.float64)
    A64 = np.asarray(A, dtype=np.float64)
    B64 = np.asarray(B, dtype=np.float64)
    s = float(alpha) / float(r)
    return X64 @ W64.T + s * ((X64 @ A64.T) @ B64.T)


def linear_bwd_dx(dY, Wdeq, A, B, alpha: float, r: int) -> np.ndarray:
    """dX = dY W' + (alpha/r) (dY B) A in float64 (gradient of Y w.r.t. X)."""
    dY64 = np.asarray(dY, dtype=np.float64)
    W64 = np.asarray(Wdeq, dtype=np.float64)
    A64 = np.asarray(A, dtype=np.float64)
    B64 = np.asarray(B, dtype=np.float64)
    s = float(alpha) / float(r)
    return dY64 @ W64 + s * ((dY64 @ B64) @ A64)


def lora_grads(X, dY, A, B, alpha: float, r: int):
    """(dA, dB) in float64: dA = s (dY B)^T X  (r x k),  dB = s dY^T (X A^T)  (d x r).

    Y depends on A only through s (X A^T) B^T and on B only through the same
    term, so for L = <dY, Y>: dL/dB[i, q] = s sum_m dY[m, i] (X A^T)[m, q] and
    dL/dA[q, j] = s sum_m (dY B)[m, q] X[m, j].
    """
    X64 = np.asarray(X, dtype=np.float64)
    dY64 = np.asarray(dY, dtype=np.float64)
    A64 = np.asarray(A, dtype=np.float64)
    B64 = np.asarray(B, dtype=np.float64)
    s = float(alpha) / float(r)
    u = X64 @ A64.T          # M x r
    v = dY64 @ B64           # M x r
    dB = s * (dY64.T @ u)
    dA = s * (v.T @ X64)
    return dA, dB


def rel_fro(a, b) -> float:
    """Relative Frobenius error ||a - b||_F / ||b||_F (b is the reference)."""
    a64 = np.asarray(a, dtype=np.float64)
    b64 = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b64)
    num = np.linalg.norm(a64 - b64)
    return float(num / den) if den > 0 else float(num)
