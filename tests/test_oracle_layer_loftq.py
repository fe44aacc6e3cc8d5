"""Pins for the layer and LoftQ oracles: printed counts, brute force, adjoint
identity, special cases, Eckart-Young through an independent eigen-solver."""

import os

import numpy as np

import synth
from oracle import layer, loftq, nf4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_lora_param_count_printed():
    with open(os.path.join(GOLDEN, "lora_param_count.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    d, k, r, full, lora, ratio, tol = rows[0]
    d, k, r = int(d), int(k), int(r)
    n_lora = layer.lora_param_count(d, k, r)
    assert n_lora == 131072
    assert abs(n_lora - float(lora)) / float(lora) < float(tol)
    assert abs(d * k - float(full)) / float(full) < float(tol)
    assert abs(d * k / n_lora - float(ratio)) / float(ratio) < float(tol)
    # shapes the oracle uses: B is d x r, A is r x k
    A = np.zeros((r, k)); B = np.zeros((d, r))
    assert A.size + B.size == n_lora


def _loops_fwd(X, W, A, B, s):
    M, k = X.shape
    d = W.shape[0]
    r = A.shape[0]
    Y = np.zeros((M, d))
    for t in range(M):
        u = [sum(X[t, j] * A[q, j] for j in range(k)) for q in range(r)]
        for i in range(d):
            Y[t, i] = sum(X[t, j] * W[i, j] for j in range(k)) + s * sum(u[q] * B[i, q] for q in range(r))
    return Y


def _loops_bwd(dY, W, A, B, s):
    M, d = dY.shape
    k = W.shape[1]
    r = A.shape[0]
    dX = np.zeros((M, k))
    for t in range(M):
        v = [sum(dY[t, i] * B[i, q] for i in range(d)) for q in range(r)]
        for j in range(k):
            dX[t, j] = sum(dY[t, i] * W[i, j] for i in range(d)) + s * sum(v[q] * A[q, j] for q in range(r))
    return dX


def test_layer_bruteforce_tiny():
    g = np.random.default_rng(0)
    M, d, k, r = 3, 5, 7, 2
    X = g.standard_normal((M, k)); W = g.standard_normal((d, k))
    A = g.standard_normal((r, k)); B = g.standard_normal((d, r))
    dY = g.standard_normal((M, d))
    alpha = 6.0
    assert np.allclose(layer.linear_fwd(X, W, A, B, alpha, r), _loops_fwd(X, W, A, B, alpha / r), rtol=1e-12, atol=1e-12)
    assert np.allclose(layer.linear_bwd_dx(dY, W, A, B, alpha, r), _loops_bwd(dY, W, A, B, alpha / r), rtol=1e-12, atol=1e-12)


def test_layer_adjoint_identity():
    # dX is the adjoint of the linear map X -> Y:  <dY, Y(X)> == <dX(dY), X>
    g = np.random.default_rng(1)
    M, d, k, r = 6, 40, 24, 4
    X = g.standard_normal((M, k)); W = g.standard_normal((d, k))
    A = g.standard_normal((r, k)); B = g.standard_normal((d, r)); dY = g.standard_normal((M, d))
    lhs = np.sum(dY * layer.linear_fwd(X, W, A, B, 8.0, r))
    rhs = np.sum(layer.linear_bwd_dx(dY, W, A, B, 8.0, r) * X)
    assert abs(lhs - rhs) <= 1e-10 * (abs(lhs) + 1)


def test_layer_unit_rows_and_pure_lora():
    c = synth.layer_case(seed=0, d=128, k=128, M=4, r=8)
    t = nf4.quantize(c["W"], 64, dq=True)
    Wd = nf4.dequantize(t).reshape(128, 128)
    A = c["A"].float().numpy(); B = c["B"].float().numpy()
    X = np.zeros((3, 128)); X[0, 5] = 1; X[1, 0] = 1; X[2, 127] = 1
    Y = layer.linear_fwd(X, Wd, A, 0 * B, 16.0, 8)
    assert np.array_equal(Y[0], Wd[:, 5].astype(np.float64))
    assert np.array_equal(Y[2], Wd[:, 127].astype(np.float64))
    # all codes at the exact zero: the layer is the adapter alone
    zero = nf4.quantize(np.zeros((128, 128), np.float32), 64, dq=True)
    Wz = nf4.dequantize(zero).reshape(128, 128)
    assert not np.any(Wz)
    Xr = c["X"].float().numpy().astype(np.float64)
    A = A.astype(np.float64); B = B.astype(np.float64)
    Y2 = layer.linear_fwd(Xr, Wz, A, B, 16.0, 8)
    small = _loops_fwd(Xr[:1, :16], np.zeros((4, 16)), A[:, :16], B[:4], 16.0 / 8)
    Ys = layer.linear_fwd(Xr[:1, :16], np.zeros((4, 16)), A[:, :16], B[:4], 16.0, 8)
    assert np.allclose(Ys, small, rtol=1e-12, atol=1e-14)
    assert np.allclose(Y2, layer.linear_fwd(Xr, np.zeros((128, 128)), A, B, 16.0, 8), rtol=0, atol=0)


def test_loftq_T0_is_plain_qlora():
    W = synth.loftq_case(seed=4, d=64, k=128)
    res = loftq.loftq(W, r=4, alpha=4.0, T=0)
    t = nf4.quantize(W, 64, dq=True)
    e0 = np.linalg.norm(W.astype(np.float64) - nf4.dequantize(t).reshape(W.shape))
    assert res.resid == [e0]
    assert np.array_equal(res.Q.packed, t.packed)
    assert not np.any(res.A) and not np.any(res.B)


def test_loftq_eckart_young_independent_eigensolver():
    W = synth.loftq_case(seed=4, d=96, k=64)
    r, alpha = 5, 10.0
    res = loftq.loftq(W, r=r, alpha=alpha, T=2)
    R = W.astype(np.float64) - nf4.dequantize(res.Q).reshape(W.shape)
    # eigenvalues of R^T R are the squared singular values (independent of SVD)
    ev = np.sort(np.linalg.eigvalsh(R.T @ R))[::-1]
    tail = np.sum(np.clip(ev[r:], 0, None))
    assert abs(res.resid[-1] ** 2 - tail) <= 1e-9 * np.sum(ev)
    s = alpha / r
    D = s * res.B @ res.A
    assert np.linalg.matrix_rank(D, tol=1e-12 * np.linalg.norm(D)) <= r
    assert abs(np.linalg.norm(R - D) - res.resid[-1]) < 1e-12 * res.resid[0]


def test_loftq_first_step_never_worse_and_trend():
    W = synth.loftq_case(seed=4, d=128, k=128)
    res = loftq.loftq(W, r=8, alpha=8.0, T=5)
    e = res.resid
    assert len(e) == 6
    assert e[1] <= e[0]                 # Q_1 = Q_0 and a rank-r fit can only help
    assert e[-1] < e[0]
    # the exact alternation is close to monotone; allow tiny NF4 boundary noise
    for a, b in zip(e[1:], e[2:]):
        assert b <= a * (1 + 1e-3)
