"""Pins of the oracle's adapter gradients, one-step LoftQ, merge / unmerge and
the double-quantisation rounding rules, each against something other than the
function under test: brute-force loops, the exact adjoint identity of a
bilinear map, Eckart-Young through an independent eigensolver, exactly
low-rank residuals, the quantiser's idempotence, the NF4 error bound, and
hand-derived rational arithmetic.  CPU only."""

from fractions import Fraction

import numpy as np
import pytest

import synth
from oracle import layer, loftq, merge, nf4


def _bf16_vals(a):
    return synth.to_bf16(a).float().numpy()


# ----------------------------------------------------------- adapter gradients

def test_lora_grads_brute_force_loops():
    g = np.random.default_rng(1)
    M, d, k, r, alpha = 3, 4, 5, 2, 6.0
    X, dY = g.standard_normal((M, k)), g.standard_normal((M, d))
    A, B = g.standard_normal((r, k)), g.standard_normal((d, r))
    dA, dB = layer.lora_grads(X, dY, A, B, alpha, r)
    s = alpha / r
    for q in range(r):
        for j in range(k):
            acc = 0.0
            for m in range(M):
                v = sum(dY[m, i] * B[i, q] for i in range(d))
                acc += v * X[m, j]
            assert abs(dA[q, j] - s * acc) < 1e-12
    for i in range(d):
        for q in range(r):
            acc = 0.0
            for m in range(M):
                u = sum(X[m, j] * A[q, j] for j in range(k))
                acc += dY[m, i] * u
            assert abs(dB[i, q] - s * acc) < 1e-12


def test_lora_grads_adjoint_identity():
    """L(A, B) = <dY, X W^T + s X A^T B^T> is linear in A and in B, so a step E
    changes L by exactly <dA, E> (resp. <dB, F>)."""
    g = np.random.default_rng(2)
    M, d, k, r, alpha = 7, 11, 9, 3, 12.0
    s = alpha / r
    X, dY, W = g.standard_normal((M, k)), g.standard_normal((M, d)), g.standard_normal((d, k))
    A, B = g.standard_normal((r, k)), g.standard_normal((d, r))
    E, F = g.standard_normal((r, k)), g.standard_normal((d, r))

    def loss(Am, Bm):
        Y = X @ W.T + s * (X @ Am.T) @ Bm.T
        return float(np.sum(dY * Y))

    dA, dB = layer.lora_grads(X, dY, A, B, alpha, r)
    assert dA.shape == (r, k) and dB.shape == (d, r)
    base = loss(A, B)
    assert abs((loss(A + E, B) - base) - float(np.sum(dA * E))) < 1e-9 * max(1.0, abs(base))
    assert abs((loss(A, B + F) - base) - float(np.sum(dB * F))) < 1e-9 * max(1.0, abs(base))


# --------------------------------------------------------------- one-step LoftQ

def test_one_step_recovers_an_exactly_low_rank_residual():
    g = np.random.default_rng(3)
    d, k, r, alpha = 96, 128, 4, 8.0
    s = alpha / r
    Q = nf4.quantize((g.standard_normal((d, k)) * 0.02).astype(np.float32), 64, dq=True)
    L = (g.standard_normal((d, r)) @ g.standard_normal((r, k))) * 1e-3
    W = (nf4.dequantize(Q).reshape(d, k).astype(np.float64) + L).astype(np.float32)
    res = loftq.loftq_one_step(W, Q, r, alpha)
    R = W.astype(np.float64) - nf4.dequantize(Q).reshape(d, k)
    assert abs(res.resid[0] - np.linalg.norm(R)) < 1e-12 * np.linalg.norm(R)
    # only the fp32 rounding of W is left over
    assert res.resid[1] < 1e-6 * res.resid[0]
    assert np.max(np.abs(s * (res.B @ res.A) - L)) < 1e-8
    assert res.A.shape == (r, k) and res.B.shape == (d, r)


def test_one_step_eckart_young_independent_eigensolver():
    g = np.random.default_rng(4)
    d, k, r, alpha = 80, 64, 6, 6.0
    W = (g.standard_normal((d, k)) * 0.02).astype(np.float32)
    Q = nf4.quantize((W * 1.1).astype(np.float32), 64, dq=False)    # any given Q, not NF4(W)
    res = loftq.loftq_one_step(W, Q, r, alpha)
    R = W.astype(np.float64) - nf4.dequantize(Q).reshape(d, k)
    ev = np.sort(np.linalg.eigvalsh(R.T @ R))[::-1]                 # sigma_i^2, another LAPACK routine
    expect = np.sqrt(max(float(np.sum(R * R) - np.sum(ev[:r])), 0.0))
    assert abs(res.resid[1] - expect) < 1e-7 * res.resid[0]
    assert res.resid[1] < res.resid[0]


def test_one_step_keeps_q_and_matches_first_alternation_when_q_is_nf4_of_w():
    """With Q = NF4(W) the first LoftQ alternation quantises W - 0 = W again, so
    its adapter is the one-step adapter (consistency of two oracle paths)."""
    W = synth.loftq_case(seed=5, d=128, k=192)
    Q = nf4.quantize(W, 64, dq=True)
    one = loftq.loftq_one_step(W, Q, 8, 8.0)
    full = loftq.loftq(W, 8, 8.0, T=1)
    assert np.array_equal(full.Q.packed, Q.packed)
    assert abs(one.resid[1] - full.resid[1]) < 1e-12
    assert np.allclose(one.B @ one.A, full.B @ full.A, atol=1e-12)


# ------------------------------------------------------------------ merge

def _adapter(g, d, k, r):
    A = _bf16_vals(g.standard_normal((r, k)) / np.sqrt(k))
    B = _bf16_vals(g.standard_normal((d, r)) * 0.01)
    return A, B


def test_adapter_product_order_and_exact_terms():
    # terms 1, 2^-24, 2^-24: ascending rank order rounds 1 + 2^-24 to 1 twice
    # (ties to even); any other order, or a wider accumulator, gives 1 + 2^-23
    B = np.array([[1.0, 2.0 ** -12, 2.0 ** -12]], np.float32)
    A = np.array([[1.0], [2.0 ** -12], [2.0 ** -12]], np.float32)
    assert merge.adapter_product_f32(A, B)[0, 0] == np.float32(1.0)
    assert merge.adapter_product_f32(A[::-1].copy(), B[:, ::-1].copy())[0, 0] == np.float32(1.0 + 2.0 ** -23)
    # r = 1: the single product is exact
    g = np.random.default_rng(5)
    A1, B1 = _adapter(g, 8, 16, 1)
    exact = [[Fraction(float(B1[i, 0])) * Fraction(float(A1[0, j])) for j in range(16)] for i in range(8)]
    got = merge.adapter_product_f32(A1, B1)
    assert all(Fraction(float(got[i, j])) == exact[i][j] for i in range(8) for j in range(16))
    with pytest.raises(ValueError):
        merge.adapter_product_f32(np.full((1, 4), 1.0 + 2.0 ** -20, np.float32), B1[:4])


def test_adapter_product_recursive_summation_bound():
    g = np.random.default_rng(6)
    d, k, r = 24, 40, 16
    A, B = _adapter(g, d, k, r)
    got = merge.adapter_product_f32(A, B).astype(np.float64)
    u = 2.0 ** -24
    gamma = (r * u) / (1 - r * u)
    for i in range(0, d, 5):
        for j in range(0, k, 7):
            terms = [Fraction(float(B[i, q])) * Fraction(float(A[q, j])) for q in range(r)]
            ex = sum(terms, Fraction(0))
            assert abs(Fraction(float(got[i, j])) - ex) <= Fraction(gamma) * sum(abs(t) for t in terms)


def test_merge_with_zero_adapter_is_idempotent():
    g = np.random.default_rng(7)
    d, k, r = 64, 192, 4
    W = (g.standard_normal((d, k)) * 0.02).astype(np.float32)
    A, B = _adapter(g, d, k, r)
    for dq in (False, True):
        Q = nf4.quantize(W, 64, dq=dq)
        Qm = merge.merge(Q, d, k, A, np.zeros_like(B), 8.0, r)
        assert np.array_equal(Qm.packed, Q.packed)              # codes come back unchanged
        if not dq:
            assert np.array_equal(Qm.absmax, Q.absmax)          # and so do exact constants


def test_merge_within_nf4_error_bound_and_sign():
    g = np.random.default_rng(8)
    d, k, r, alpha = 64, 256, 8, 16.0
    s = alpha / r
    W = (g.standard_normal((d, k)) * 0.02).astype(np.float32)
    A, B = _adapter(g, d, k, r)
    B = B * 4
    Q = nf4.quantize(W, 64, dq=False)
    gap = float(np.max(np.diff(nf4.codebook().astype(np.float64))))
    base = nf4.dequantize(Q).reshape(d, k).astype(np.float64)
    for sign in (1, -1):
        target = base + sign * s * (B.astype(np.float64) @ A.astype(np.float64))   # library matmul
        Qm = merge.merge(Q, d, k, A, B, alpha, r, sign)
        w = nf4.dequantize(Qm).reshape(d, k).astype(np.float64)
        m = np.repeat(Qm.absmax.astype(np.float64), 64).reshape(d, k)
        assert np.all(np.abs(w - target) <= m * gap / 2 * (1 + 1e-5) + 1e-9)
        other = base - sign * s * (B.astype(np.float64) @ A.astype(np.float64))
        assert np.linalg.norm(w - target) < 0.5 * np.linalg.norm(w - other)


def test_unmerge_after_merge_drifts_within_two_error_bounds():
    g = np.random.default_rng(9)
    d, k, r, alpha = 64, 128, 8, 8.0
    W = (g.standard_normal((d, k)) * 0.02).astype(np.float32)
    A, B = _adapter(g, d, k, r)
    Q = nf4.quantize(W, 64, dq=False)
    Qm = merge.merge(Q, d, k, A, B * 4, alpha, r, 1)
    Qu = merge.merge(Qm, d, k, A, B * 4, alpha, r, -1)
    gap = float(np.max(np.diff(nf4.codebook().astype(np.float64))))
    w0 = nf4.dequantize(Q).reshape(d, k).astype(np.float64)
    wu = nf4.dequantize(Qu).reshape(d, k).astype(np.float64)
    mm = np.repeat(np.maximum(Qm.absmax, Qu.absmax).astype(np.float64), 64).reshape(d, k)
    assert np.all(np.abs(wu - w0) <= mm * gap * (1 + 1e-5) + 1e-9)
    assert not np.array_equal(Qu.packed, Q.packed)     # the round trip does not restore Q


# ------------------------------------------------- double-quantisation rounding

def test_dq_codes_round_half_to_even_on_exact_ties():
    """A group with mean exactly 2, largest deviation 127/128 (sigma = 2^-7
    exactly) and deviations (j + 1/2)/128, so fp32(c_j / sigma) = j + 1/2
    exactly; every step below is checked to be exact with Fractions."""
    half = [0.5, 1.5, 2.5, 3.5, 126.5]
    dev = [127.0] + half
    m = []
    for v in dev:
        m += [2.0 + v / 128.0, 2.0 - v / 128.0]
    m += [2.0] * (256 - len(m))
    m = np.array(m, np.float32)
    assert all(Fraction(float(x)) == Fraction(2) + Fraction(s) * Fraction(v) / 128
               for x, (s, v) in zip(m, [(sg, v) for v in dev for sg in (1, -1)]))
    assert sum(Fraction(float(x)) for x in m) / 256 == 2
    q, sigma, mu = nf4.double_quant(m, 256)
    assert mu == np.float32(2.0) and sigma[0] == np.float32(2.0 ** -7)
    # hand-derived: ties go to the even integer, symmetric for negatives
    want = {127.0: 127, 0.5: 0, 1.5: 2, 2.5: 2, 3.5: 4, 126.5: 126}
    for i, v in enumerate(dev):
        assert q[2 * i] == want[v], (v, q[2 * i])
        assert q[2 * i + 1] == -want[v], (v, q[2 * i + 1])
    assert np.all(q[2 * len(dev):] == 0)


def test_dq_decode_rounds_product_then_sum():
    """m' = fp32(fp32(q sigma) + mu): a case (found with exact rationals) where
    one rounding of q sigma + mu gives a different fp32."""
    q = np.array([-50], np.int8)
    sigma = np.array([0x3A033898], np.uint32).view(np.float32)
    mu = np.array([0x3D2495CF], np.uint32).view(np.float32)[0]
    fq, fs, fm = Fraction(-50), Fraction(float(sigma[0])), Fraction(float(mu))
    prod64 = np.float64(-50) * np.float64(sigma[0])
    assert Fraction(prod64) == fq * fs                        # exact in float64
    p32 = np.float32(prod64)                                  # first rounding
    s64 = np.float64(p32) + np.float64(mu)
    assert Fraction(s64) == Fraction(float(p32)) + fm         # exact in float64
    two = np.float32(s64)                                     # second rounding
    one64 = prod64 + np.float64(mu)
    assert Fraction(one64) == fq * fs + fm
    one = np.float32(one64)                                   # single rounding
    assert two != one
    got = nf4.dequant_absmax(q, sigma, mu, 256)
    assert got.view(np.uint32)[0] == np.float32(two).view(np.uint32)
