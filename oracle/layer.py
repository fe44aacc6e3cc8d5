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


def rel_fro(a, b) -> float:
    """Relative Frobenius error ||a - b||_F / ||b||_F (b is the reference)."""
    a64 = np.asarray(a, dtype=np.float64)
    b64 = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b64)
    num = np.linalg.norm(a64 - b64)
    return float(num / den) if den > 0 else float(num)
