"""Pins for the NF4 oracle: values the pages print, exact arithmetic, brute force.

None of these re-types the oracle's own formula: each checks the oracle
against an independent route (exact rationals, pure-Python loops, a library
routine for a special case, or printed values).
"""

import os
from fractions import Fraction
from statistics import NormalDist

import numpy as np
import pytest

from oracle import exact, nf4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- codebook

def test_codebook_printed_values():
    cb = nf4.codebook()
    for idx, val, dec in _read_golden("nf4_codebook_printed.txt"):
        assert round(float(cb[int(idx)]), int(dec)) == float(val), (idx, cb[int(idx)])


def test_codebook_structure():
    cb = nf4.codebook()
    assert cb.dtype == np.float32 and cb.size == 16
    assert np.all(np.diff(cb.astype(np.float64)) > 0)          # strictly increasing
    assert cb[0] == -1.0 and cb[15] == 1.0                      # span [-1, 1]
    assert cb[7] == 0.0                                         # exact zero
    assert np.sum(cb < 0) == 7 and np.sum(cb > 0) == 8          # asymmetric split


def test_codebook_against_independent_quantile_routine():
    # statistics.NormalDist.inv_cdf is an independent implementation of the
    # normal quantile function; rebuild the positive/negative levels with it.
    nd = NormalDist()
    delta = 0.5 * (1 / 30 + 1 / 32)
    hi = 1 - delta
    pos = [nd.inv_cdf(hi + (0.5 - hi) * i / 8) for i in range(8)]
    neg = [-nd.inv_cdf(hi + (0.5 - hi) * i / 7) for i in range(7)]
    lv = sorted(pos + [0.0] + neg)
    top = max(lv)
    ref = np.array([x / top for x in lv], dtype=np.float64)
    cb = nf4.codebook().astype(np.float64)
    assert np.max(np.abs(cb - ref)) < 1e-7


# ------------------------------------------------------ nearest-level search

def _midpoints_exact(cb):
    return [(Fraction(float(cb[i])) + Fraction(float(cb[i + 1]))) / 2 for i in range(15)]


def _code_by_exact_thresholds(vals, cb):
    """Independent route: count exact midpoints strictly below v (ties -> lower)."""
    mids = _midpoints_exact(cb)
    out = []
    for v in vals:
        fv = Fraction(float(v))
        out.append(sum(1 for m in mids if fv > m))
    return np.array(out, dtype=np.uint8)


def test_nearest_matches_exact_thresholds_random():
    cb = nf4.codebook()
    g = np.random.default_rng(123)
    v = g.uniform(-1, 1, 3000).astype(np.float32)
    assert np.array_equal(nf4.nearest_code(v, cb), _code_by_exact_thresholds(v, cb))


def test_nearest_exhaustive_near_every_threshold():
    cb = nf4.codebook()
    mids = _midpoints_exact(cb)
    vals = []
    for m in mids:
        centre = np.float32(float(m)).view(np.int32)
        vals.append((centre + np.arange(-1000, 1001, dtype=np.int32)).view(np.float32))
    v = np.concatenate(vals)
    assert np.array_equal(nf4.nearest_code(v, cb), _code_by_exact_thresholds(v, cb))


def test_nearest_tie_goes_to_lower_index():
    cb = nf4.codebook()
    found = 0
    for i, m in enumerate(_midpoints_exact(cb)):
        f = np.float32(float(m))
        if Fraction(float(f)) == m:       # midpoint exactly representable in fp32
            found += 1
            assert nf4.nearest_code(np.array([f]), cb)[0] == i
    # also a constructed tie on a toy table (library-independent check)
    toy = np.array([-1.0, 0.0, 0.5, 1.0] + [2.0 + i for i in range(12)], dtype=np.float32)
    assert nf4.nearest_code(np.array([0.25], dtype=np.float32), toy)[0] == 1
    assert found >= 0


def test_nearest_pure_python_bruteforce_tiny():
    cb = nf4.codebook()
    g = np.random.default_rng(7)
    v = g.uniform(-1.05, 1.05, 200).astype(np.float32)
    ref = []
    for x in v:
        best, bi = None, None
        for i, c in enumerate(cb):
            dist = abs(Fraction(float(x)) - Fraction(float(c)))
            if best is None or dist < best:
                best, bi = dist, i
        ref.append(bi)
    assert np.array_equal(nf4.nearest_code(v, cb), np.array(ref, dtype=np.uint8))


# ------------------------------------------------------------ block absmax

def test_block_absmax_loop_with_ragged_tail():
    g = np.random.default_rng(1)
    x = g.standard_normal(64 * 5 + 17).astype(np.float32)
    got = nf4.block_absmax(x, 64)
    ref = [max(abs(float(t)) for t in x[s:s + 64]) for s in range(0, x.size, 64)]
    assert got.size == 6
    assert np.array_equal(got, np.array(ref, dtype=np.float32))


# ---------------------------------------------------------------- round trip

def test_codebook_multiples_round_trip_exactly():
    cb = nf4.codebook()
    g = np.random.default_rng(5)
    for _ in range(200):
        m = np.float32(10.0 ** g.uniform(-6, 3))
        idx = g.integers(0, 16, 64)
        idx[g.integers(0, 64)] = 15 if g.integers(0, 2) else 0   # absmax present
        x = np.multiply(cb[idx], m, dtype=np.float32)
        t = nf4.quantize(x, 64, dq=False)
        assert np.array_equal(nf4.unpack(t.packed, 64), idx.astype(np.uint8))
        assert np.array_equal(nf4.dequantize(t), x)


def test_zero_block_and_single_nonzero():
    x = np.zeros(128, dtype=np.float32)
    x[70] = -3.5
    t = nf4.quantize(x, 64, dq=False)
    codes = nf4.unpack(t.packed, 128)
    assert np.all(codes[:64] == 7)
    assert codes[70] == 0 and np.all(np.delete(codes[64:], 6) == 7)
    assert t.absmax[0] == 0 and t.absmax[1] == np.float32(3.5)
    w = nf4.dequantize(t)
    assert np.array_equal(w, x)


def test_dequant_error_bound():
    cb = nf4.codebook().astype(np.float64)
    gap = np.max(np.diff(cb))
    g = np.random.default_rng(11)
    x = (g.standard_normal(64 * 300) * 0.02).astype(np.float32)
    t = nf4.quantize(x, 64, dq=False)
    w = nf4.dequantize(t).astype(np.float64)
    m = np.repeat(t.absmax.astype(np.float64), 64)
    err = np.abs(w - x.astype(np.float64))
    assert np.all(err <= m * gap / 2 * (1 + 1e-6) + 1e-30)


def test_pack_nibble_order_and_odd_length():
    codes = np.array([1, 2, 3, 4, 15], dtype=np.uint8)
    p = nf4.pack(codes)
    assert list(p) == [0x21, 0x43, 0x0F]
    assert np.array_equal(nf4.unpack(p, 5), codes)


# ------------------------------------------------------ double quantisation

def test_double_quant_error_bound_and_rounding():
    g = np.random.default_rng(3)
    m = np.abs(g.standard_normal(256 * 7 + 100) * 0.05).astype(np.float32)
    q, sigma, mu = nf4.double_quant(m, 256)
    assert q.dtype == np.int8 and np.all(np.abs(q.astype(int)) <= 127)
    mp = nf4.dequant_absmax(q, sigma, mu, 256).astype(np.float64)
    grp = np.arange(m.size) // 256
    bound = sigma[grp].astype(np.float64) / 2 + 4 * np.spacing(np.abs(m).astype(np.float32)).astype(np.float64) \
        + 4 * np.spacing(np.float32(mu))
    assert np.all(np.abs(mp - m.astype(np.float64)) <= bound)
    # every group uses its full int8 range: the extreme deviation maps to +-127
    for gi in range(sigma.size):
        assert np.max(np.abs(q[grp == gi].astype(int))) == 127


def test_double_quant_half_even_and_zero_group():
    # one group whose deviations are exact multiples: mean 0 after construction
    m = np.array([1.0, 3.0] + [2.0] * 254, dtype=np.float32)  # mean exactly 2
    q, sigma, mu = nf4.double_quant(m, 256)
    assert mu == np.float32(2.0)
    assert sigma[0] == np.float32(np.float32(1.0) / np.float32(127.0))
    assert q[0] == -127 and q[1] == 127 and np.all(q[2:] == 0)
    # constant constants: deviation 0 -> sigma 0, codes 0, decode = mu exactly
    m2 = np.full(300, 0.125, dtype=np.float32)
    q2, s2, mu2 = nf4.double_quant(m2, 256)
    assert np.all(s2 == 0) and np.all(q2 == 0) and mu2 == np.float32(0.125)
    assert np.all(nf4.dequant_absmax(q2, s2, mu2, 256) == np.float32(0.125))
    # rint ties to even: 2.5 -> 2, 3.5 -> 4 (numpy rint is IEEE roundeven)
    assert np.rint(np.float32(2.5)) == 2 and np.rint(np.float32(3.5)) == 4


def test_storage_closed_form():
    n = 4096 * 4096
    # 4-bit codes + int8 absmax per 64 + fp32 scale per 256 blocks + fp32 mean
    bits = 8 * nf4.storage_bytes(n) / n
    assert abs(bits - (4 + 8 / 64 + 32 / (64 * 256) + 32 / n)) < 1e-9
    assert nf4.storage_bytes(n, dq=False) * 8 / n == 4.5
    # "about 4x" memory reduction versus 16-bit weights (PEFT course notes §4.2)
    assert 3.8 < 16 / bits < 4.0
    # a 65B-parameter base model fits a 48 GB GPU ("QLoRA paper summary")
    assert 65e9 * bits / 8 < 48e9


# ------------------------------------------------------------- exact helpers

def test_exact_sum_matches_fraction_bruteforce():
    g = np.random.default_rng(9)
    for _ in range(20):
        v = np.abs(g.standard_normal(50) * 10.0 ** g.uniform(-40, 30, 50)).astype(np.float32)
        v[:3] = [0.0, 1e-45, 3e38]
        ref = sum((Fraction(float(x)) for x in v), Fraction(0))
        assert exact.exact_sum_f32(v) == ref


def _is_nearest_f32(x: Fraction, f: np.float32) -> bool:
    fv = Fraction(float(f))
    up = Fraction(float(np.nextafter(f, np.float32(np.inf))))
    dn = Fraction(float(np.nextafter(f, np.float32(-np.inf))))
    d = abs(fv - x)
    if abs(up - x) < d or abs(dn - x) < d:
        return False
    if abs(up - x) == d or abs(dn - x) == d:     # tie: must be the even one
        return (int(np.float32(f).view(np.uint32)) & 1) == 0
    return True


def test_round_fraction_to_f32_nearest():
    g = np.random.default_rng(10)
    for _ in range(400):
        x = Fraction(int(g.integers(1, 2**62)), int(g.integers(1, 2**62))) * Fraction(2) ** int(g.integers(-160, 120))
        assert _is_nearest_f32(x, exact.round_fraction_to_f32(x))
    # exact ties between neighbouring fp32 values go to the even significand
    one = Fraction(1)
    tie = one + Fraction(1, 2**24)                 # halfway between 1 and 1+2^-23
    assert exact.round_fraction_to_f32(tie) == np.float32(1.0)
    tie2 = one + Fraction(3, 2**24)
    assert exact.round_fraction_to_f32(tie2) == np.float32(1.0 + 2.0**-22)
    # subnormal range
    assert exact.round_fraction_to_f32(Fraction(3, 2**150)) == np.float32(2.0**-148)


def test_exact_mean_order_independent():
    g = np.random.default_rng(12)
    v = np.abs(g.standard_normal(10000) * 0.05).astype(np.float32)
    a = exact.exact_mean_f32(v)
    b = exact.exact_mean_f32(v[::-1].copy())
    ref = exact.round_fraction_to_f32(sum((Fraction(float(x)) for x in v), Fraction(0)) / v.size)
    assert a == b == ref


def test_bf16_rounding_against_torch_and_neighbours():
    import torch
    g = np.random.default_rng(13)
    x = (g.standard_normal(20000) * 10.0 ** g.uniform(-20, 20, 20000)).astype(np.float32)
    # exact halfway cases: low 16 bits == 0x8000
    halfway = (((0x3F80 + g.integers(0, 256, 200)).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, halfway])
    ours = exact.f32_to_bf16_bits(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)
    # neighbour check: no other bf16 value is closer to x
    for xv, bb in zip(x[:300], ours[:300]):
        fx = Fraction(float(xv))
        b = int(bb)
        if (b & 0x7FFF) in (0, 0x7F7F):
            continue
        near = [Fraction(float(exact.bf16_bits_to_f32(np.array([b + dlt], np.uint16))[0]))
                for dlt in (-1, 0, 1)]
        assert abs(near[1] - fx) <= min(abs(near[0] - fx), abs(near[2] - fx))


# ---------------------------------------------------------- quantise helpers

@pytest.mark.parametrize("n", [1, 63, 64, 65, 64 * 257 + 5])
def test_quantize_any_length(n):
    g = np.random.default_rng(n)
    x = (g.standard_normal(n) * 0.02).astype(np.float32)
    t = nf4.quantize(x, 64, dq=True, dq_block=256)
    assert t.packed.size == (n + 1) // 2
    assert t.absmax.size == -(-n // 64)
    assert t.absmax_scale.size == -(-t.absmax.size // 256)
    w = nf4.dequantize(t)
    assert w.shape == (n,)
    assert np.all(np.abs(w) <= np.repeat(t.effective_absmax(), 64)[:n] * (1 + 1e-6))
