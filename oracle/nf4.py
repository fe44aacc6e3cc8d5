"""NF4 blockwise quantisation oracle (test infrastructure only).

Plain numpy, step by step in the order the pages give them:

1. codebook: 16 normal-quantile levels normalised to [-1, 1] with an exact
   zero ("QLoRA paper summary", NF4 bullet: a data type that is
   information-theoretically optimal for normally distributed weights, built
   from the quantile function of the standard normal);
2. normalise each block by its absmax ("QLoRA technical analysis" §2.1 shows
   ``abs_max = max(abs(x)); normalized = x / abs_max``; the block of 64
   elements replaces the page's whole tensor);
3. nearest codebook level per element by brute force (the same page's
   ``argmin |codebook - v|`` loop; argmin returns the first minimum, so ties
   go to the lower code index);
4. pack two 4-bit codes per byte (the 4x memory reduction of "PEFT course
   notes" §4.2); READING: the even element goes to the low nibble;
5. double quantisation: the absmax constants are quantised again ("PEFT
   course notes" §4.2, "QLoRA paper summary" double-quant bullet); READING:
   int8 codes in groups of 256 constants after subtracting their mean;
6. dequantisation ``w = c[code] * absmax'`` in fp32, optionally rounded to
   bf16, the compute dtype of "PEFT quantization guide".

Readings for silent points: IEEE fp32 division ``x / absmax`` (no reciprocal
multiply); a block whose absmax is 0 gets code 7 (the exact zero) everywhere;
the DQ mean is the exact mean of the constants rounded once to fp32; int8
codes round half-to-even and clamp to [-127, 127]; a group whose largest
deviation is 0 gets scale 0 and codes 0; the dequantised constant is
``fp32(fp32(q * sigma) + mu)`` (two roundings, no fused multiply-add); when
the element count is odd the unused high nibble of the last byte is 0.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
from scipy.stats import norm

from . import exact

BLOCK = 64
DQ_BLOCK = 256


def codebook() -> np.ndarray:
    """The 16 NF4 levels, ascending, as fp32.

    Construction of the QLoRA normal-quantile table: with the tail offset
    delta = (1/30 + 1/32) / 2, take 8 positive levels Phi^-1(p) for the first
    8 of 9 equally spaced probabilities from 1 - delta down to 1/2, and 7
    negative levels -Phi^-1(p) for the first 7 of 8 equally spaced
    probabilities over the same range; add an exact 0, sort, divide by the
    largest level (so the span is [-1, 1]) and round to fp32.
    """
    delta = 0.5 * (1.0 / 30.0 + 1.0 / 32.0)
    p_hi = 1.0 - delta
    pos = norm.ppf(np.linspace(p_hi, 0.5, 9)[:-1])
    neg = -norm.ppf(np.linspace(p_hi, 0.5, 8)[:-1])
    levels = np.sort(np.concatenate([pos, [0.0], neg]))
    levels = levels / levels.max()
    return levels.astype(np.float32)


def nearest_code(v: np.ndarray, cb: np.ndarray | None = None) -> np.ndarray:
    """Index of the nearest codebook level for each fp32 value, ties to lower.

    Brute force over all 16 levels with float64 distances (the difference of
    two fp32 values near a decision point is exact in float64).
    ``np.argmin`` returns the first minimum, i.e. the lower index on a tie.
    """
    cb = codebook() if cb is None else cb
    v64 = np.asarray(v, dtype=np.float32).astype(np.float64).reshape(-1)
    out = np.empty(v64.shape, dtype=np.uint8)
    step = 1 << 20
    c64 = cb.astype(np.float64)
    for s in range(0, v64.size, step):
        d = np.abs(v64[s:s + step, None] - c64[None, :])
        out[s:s + step] = np.argmin(d, axis=1).astype(np.uint8)
    return out.reshape(np.shape(v))


def block_absmax(x32: np.ndarray, block: int = BLOCK) -> np.ndarray:
    """max |x| over consecutive blocks of ``block`` elements (last block may be short)."""
    flat = np.asarray(x32, dtype=np.float32).reshape(-1)
    n = flat.size
    nblk = -(-n // block)
    pad = np.zeros(nblk * block, dtype=np.float32)
    pad[:n] = np.abs(flat)
    return pad.reshape(nblk, block).max(axis=1).astype(np.float32)


def quantize_codes(x32: np.ndarray, block: int = BLOCK):
    """Per-element 4-bit codes (unpacked, uint8) and the fp32 block absmax."""
    flat = np.asarray(x32, dtype=np.float32).reshape(-1)
    n = flat.size
    absmax = block_absmax(flat, block)
    m_el = np.repeat(absmax, block)[:n]
    v = np.zeros(n, dtype=np.float32)
    nz = m_el != 0
    v[nz] = np.divide(flat[nz], m_el[nz], dtype=np.float32)  # IEEE fp32 RN
    return nearest_code(v), absmax


def pack(codes: np.ndarray) -> np.ndarray:
    """Two codes per byte: element 2q in the low nibble, 2q+1 in the high nibble."""
    c = np.asarray(codes, dtype=np.uint8).reshape(-1)
    if c.size % 2:
        c = np.concatenate([c, np.zeros(1, dtype=np.uint8)])
    return (c[0::2] | (c[1::2] << 4)).astype(np.uint8)


def unpack(packed: np.ndarray, n: int) -> np.ndarray:
    """Inverse of :func:`pack`, returning the first ``n`` codes."""
    p = np.asarray(packed, dtype=np.uint8).reshape(-1)
    out = np.empty(p.size * 2, dtype=np.uint8)
    out[0::2] = p & 0x0F
    out[1::2] = p >> 4
    return out[:n]


def double_quant(absmax: np.ndarray, dq_block: int = DQ_BLOCK):
    """Quantise the fp32 absmax constants to int8 in groups of ``dq_block``.

    mu = exact mean of all constants rounded to fp32; per group g:
    c_j = fp32(m_j - mu), S_g = max |c_j|, sigma_g = fp32(S_g / 127),
    q_j = clamp(rint_half_even(fp32(c_j / sigma_g)), -127, 127), 0 when sigma_g = 0.
    Returns (q int8[nblk], sigma fp32[ngrp], mu fp32).
    """
    m = np.asarray(absmax, dtype=np.float32).reshape(-1)
    nblk = m.size
    mu = exact.exact_mean_f32(m)
    c = np.subtract(m, mu, dtype=np.float32)
    ngrp = -(-nblk // dq_block)
    q = np.zeros(nblk, dtype=np.int8)
    sigma = np.zeros(ngrp, dtype=np.float32)
    for g in range(ngrp):
        cg = c[g * dq_block:(g + 1) * dq_block]
        S = np.float32(np.max(np.abs(cg)))
        sg = np.divide(S, np.float32(127.0), dtype=np.float32)
        sigma[g] = sg
        if sg == 0:
            continue
        r = np.rint(np.divide(cg, sg, dtype=np.float32))
        q[g * dq_block:(g + 1) * dq_block] = np.clip(r, -127, 127).astype(np.int8)
    return q, sigma, np.float32(mu)


def dequant_absmax(q: np.ndarray, sigma: np.ndarray, mu, dq_block: int = DQ_BLOCK) -> np.ndarray:
    """m'_j = fp32(fp32(q_j * sigma_g) + mu), two separate fp32 roundings."""
    q = np.asarray(q, dtype=np.int8).reshape(-1)
    g = np.arange(q.size) // dq_block
    prod = np.multiply(q.astype(np.float32), sigma[g], dtype=np.float32)
    return np.add(prod, np.float32(mu), dtype=np.float32)


@dataclass
class NF4Tensor:
    """Quantised state of one tensor of ``n`` elements."""
    n: int
    block: int
    packed: np.ndarray           # uint8[ceil(n/2)]
    absmax: np.ndarray           # fp32[nblk], exact block absmax
    dq: bool
    dq_block: int
    absmax_q: np.ndarray | None = None   # int8[nblk]
    absmax_scale: np.ndarray | None = None  # fp32[ngrp]
    absmax_mean: np.float32 | None = None

    def effective_absmax(self) -> np.ndarray:
        """Constants the dequantiser uses: exact absmax, or its DQ decode."""
        if not self.dq:
            return self.absmax
        return dequant_absmax(self.absmax_q, self.absmax_scale, self.absmax_mean, self.dq_block)


def quantize(x, block: int = BLOCK, dq: bool = True, dq_block: int = DQ_BLOCK) -> NF4Tensor:
    """Blockwise NF4 quantisation of an fp32 (or exactly widened bf16) tensor."""
    x32 = np.asarray(x, dtype=np.float32).reshape(-1)
    codes, absmax = quantize_codes(x32, block)
    t = NF4Tensor(n=x32.size, block=block, packed=pack(codes), absmax=absmax,
                  dq=dq, dq_block=dq_block)
    if dq:
        t.absmax_q, t.absmax_scale, t.absmax_mean = double_quant(absmax, dq_block)
    return t


def dequantize(t: NF4Tensor) -> np.ndarray:
    """fp32 weights w_e = fp32(c[code_e] * absmax'_block(e))."""
    cb = codebook()
    codes = unpack(t.packed, t.n)
    m = t.effective_absmax()
    m_el = np.repeat(m, t.block)[:t.n]
    return np.multiply(cb[codes], m_el, dtype=np.float32)


def dequantize_bf16_bits(t: NF4Tensor) -> np.ndarray:
    """bf16 bit patterns of the dequantised weights (fp32 result rounded RNE)."""
    return exact.f32_to_bf16_bits(dequantize(t))


def storage_bytes(n: int, block: int = BLOCK, dq: bool = True, dq_block: int = DQ_BLOCK) -> int:
    """Bytes of quantised state: packed codes + constants (+ DQ scales and mean)."""
    nblk = -(-n // block)
    codes = -(-n // 2)
    if not dq:
        return codes + 4 * nblk
    ngrp = -(-nblk // dq_block)
    return codes + nblk + 4 * ngrp + 4
