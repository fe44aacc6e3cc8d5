"""LoftQ initialisation oracle with an exact LAPACK SVD (test infrastructure only).

"LoftQ explainer" (mhpn.cn/news/832204):
  §2.2  objective  min_{Q, Delta} ||W - (Q + Delta)||_F^2,  rank(Delta) <= r;
  §2.3  alternation: Q-step  Q = quantise(W - Delta) by round-to-nearest;
        Delta-step  Delta = U_r Sigma_r V_r^T, the top-r SVD of W - Q;
        a few rounds (5-10); afterwards Q is the frozen weight and Delta
        initialises the adapter.

READINGS: the quantiser is the same NF4 blockwise quantiser (with double
quantisation when ``dq``) as the layer's; the Q-step input W - s B A is
rounded to fp32 because the quantiser consumes fp32; the adapter carries the
layer's scale s = alpha / r, so the factors are split as
B = U_r sqrt(Sigma_r) / sqrt(s), A = sqrt(Sigma_r) V_r^T / sqrt(s), giving
s B A = Delta.  Residuals e_t = ||W - deq(Q_t) - s B_t A_t||_F for
t = 0..T, where e_0 is plain QLoRA (Q_0 = NF4(W), no adapter).

One-step variant ("PEFT quantization guide", section on
replace_lora_weights_loftq): the base weight stays the quantised tensor the
caller already has, and only the adapter is replaced by one Delta-step
against it, B A from the top-r SVD of W - deq(Q).  Nothing is requantised.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import nf4


@dataclass
class LoftQResult:
    Q: nf4.NF4Tensor
    A: np.ndarray            # r x k, float64
    B: np.ndarray            # d x r, float64
    resid: list = field(default_factory=list)   # e_0 .. e_T
    sing: list = field(default_factory=list)    # singular values of W - deq(Q_t), per t


def rank_r(R: np.ndarray, r: int):
    """Best rank-r approximation of R (Eckart-Young) via float64 LAPACK SVD."""
    U, S, Vt = np.linalg.svd(R, full_matrices=False)
    return U[:, :r], S[:r], Vt[:r, :], S


def loftq(W, r: int, alpha: float, T: int, block: int = nf4.BLOCK,
          dq: bool = True, dq_block: int = nf4.DQ_BLOCK) -> LoftQResult:
    """Run T LoftQ alternations on an fp32 matrix W (d x k)."""
    W32 = np.asarray(W, dtype=np.float32)
    d, k = W32.shape
    W64 = W32.astype(np.float64)
    s = float(alpha) / float(r)

    Q = nf4.quantize(W32, block, dq, dq_block)
    R = W64 - nf4.dequantize(Q).reshape(d, k).astype(np.float64)
    B = np.zeros((d, r))
    A = np.zeros((r, k))
    res = LoftQResult(Q=Q, A=A, B=B, resid=[float(np.linalg.norm(R))])
    for _ in range(T):
        target = (W64 - s * (B @ A)).astype(np.float32)      # Q-step input
        Q = nf4.quantize(target, block, dq, dq_block)
        R = W64 - nf4.dequantize(Q).reshape(d, k).astype(np.float64)
        U, S, Vt, S_all = rank_r(R, r)                        # Delta-step
        sq = np.sqrt(S)
        B = (U * sq[None, :]) / np.sqrt(s)
        A = (sq[:, None] * Vt) / np.sqrt(s)
        res.resid.append(float(np.linalg.norm(R - s * (B @ A))))
        res.sing.append(S_all)
    res.Q, res.A, res.B = Q, A, B
    return res


@dataclass
class OneStepResult:
    A: np.ndarray            # r x k, float64
    B: np.ndarray            # d x r, float64
    resid: list              # [||W - deq(Q)||_F, ||W - deq(Q) - s B A||_F]
    sing: np.ndarray         # singular values of W - deq(Q)


def loftq_one_step(W, Q: nf4.NF4Tensor, r: int, alpha: float) -> OneStepResult:
    """One Delta-step against a given quantised weight Q (no Q-step).

    R = W - deq(Q); B = U_r sqrt(Sigma_r) / sqrt(s), A = sqrt(Sigma_r) V_r^T / sqrt(s),
    so s B A is the best rank-r approximation of R.
    """
    W64 = np.asarray(W, dtype=np.float32).astype(np.float64)
    d, k = W64.shape
    s = float(alpha) / float(r)
    R = W64 - nf4.dequantize(Q).reshape(d, k).astype(np.float64)
    U, S, Vt, S_all = rank_r(R, r)
    sq = np.sqrt(S)
    B = (U * sq[None, :]) / np.sqrt(s)
    A = (sq[:, None] * Vt) / np.sqrt(s)
    return OneStepResult(A=A, B=B, resid=[float(np.linalg.norm(R)), float(np.linalg.norm(R - s * (B @ A)))],
                         sing=S_all)
