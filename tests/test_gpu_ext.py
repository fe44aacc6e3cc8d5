"""GPU parity of the adapter gradients, the fp32-compute layer, merge /
unmerge and one-step LoftQ against the float64 oracle.

Tolerances:
* dA, dB: relative Frobenius error <= 5e-3 (the layer's bound), also per
  tile.  The CUDA path keeps X A^T and dY B as bf16 hi + lo (about 16 bits)
  and accumulates in fp32; measured errors are near 1e-5.
* fp32-compute layer: relative Frobenius error <= 1e-5.  Every operand is
  exact in fp32 (the weight is its exact fp32 dequantisation) and each
  output is a sum of K <= 11008 fp32 products accumulated in fp32: the
  rounding error grows like sqrt(K) * 2^-24 ~ 6e-6 relative for random data.
* merge / unmerge: codes, block constants and DQ state bit-exact (the merge
  arithmetic is fixed operation for operation, and the quantiser is exact).
* one-step LoftQ: both residuals within 1 % of the oracle's (exact SVD), the
  first one within 1e-6 (same quantised weight, different summation order).
"""

import numpy as np
import pytest
import torch

import synth
from oracle import layer, loftq, merge, nf4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qn():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import bit_nf4_quantized_39_b300 as mod
    return mod


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def tile_max_rel(Y, Yref, rows, cols):
    worst = 0.0
    for i in range(0, Y.shape[0], rows):
        for j in range(0, Y.shape[1], cols):
            worst = max(worst, layer.rel_fro(Y[i:i + rows, j:j + cols], Yref[i:i + rows, j:j + cols]))
    return worst


# ------------------------------------------------------------ adapter gradients

@pytest.mark.parametrize("M,d,k,r", [
    (16, 1024, 1024, 8), (37, 200, 192, 3), (300, 520, 1024, 64), (65, 128, 64, 100), (1, 256, 512, 16),
    (4096, 11008, 4096, 16),
])
def test_lora_grads(qn, M, d, k, r):
    c = synth.layer_case(seed=M + d + k + r, d=d, k=k, M=M, r=r, alpha=2.0 * r)
    dA, dB = qn.qlora_linear_bwd_lora(c["X"].cuda(), c["dY"].cuda(), c["A"].cuda(), c["B"].cuda(), c["alpha"])
    qn.device_status()
    rA, rB = layer.lora_grads(_f64(c["X"]), _f64(c["dY"]), _f64(c["A"]), _f64(c["B"]), c["alpha"], r)
    gA, gB = _f64(dA), _f64(dB)
    assert dA.shape == (r, k) and dB.shape == (d, r)
    assert layer.rel_fro(gA, rA) < 5e-3, layer.rel_fro(gA, rA)
    assert layer.rel_fro(gB, rB) < 5e-3, layer.rel_fro(gB, rB)
    assert tile_max_rel(gA, rA, 16, 128) < 5e-3
    assert tile_max_rel(gB, rB, 128, 16) < 5e-3


def test_lora_grads_repeat_bitwise(qn):
    c = synth.layer_case(seed=3, d=512, k=384, M=200, r=16)
    a = qn.qlora_linear_bwd_lora(c["X"].cuda(), c["dY"].cuda(), c["A"].cuda(), c["B"].cuda(), 8.0)
    b = qn.qlora_linear_bwd_lora(c["X"].cuda(), c["dY"].cuda(), c["A"].cuda(), c["B"].cuda(), 8.0)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# --------------------------------------------------------- fp32-compute layer

@pytest.mark.parametrize("M,d,k,r", [
    (1, 256, 512, 8), (7, 200, 192, 3), (16, 1024, 1024, 8), (300, 330, 256, 24), (129, 1000, 128, 64),
])
def test_fp32_layer(qn, M, d, k, r):
    c = synth.layer_case(seed=11 * M + d, d=d, k=k, M=M, r=r, alpha=2.0 * r)
    g = np.random.default_rng(M + 5)
    X = torch.from_numpy(g.standard_normal((M, k)).astype(np.float32))
    dY = torch.from_numpy(g.standard_normal((M, d)).astype(np.float32))
    A = torch.from_numpy((g.standard_normal((r, k)) / np.sqrt(k)).astype(np.float32))
    B = torch.from_numpy((g.standard_normal((d, r)) * 0.01).astype(np.float32))
    q = qn.nf4_quantize(torch.from_numpy(c["W"]).cuda())
    Y = qn.qlora_linear_fwd_f32(q, X.cuda(), A.cuda(), B.cuda(), c["alpha"])
    dX = qn.qlora_linear_bwd_dx_f32(q, dY.cuda(), A.cuda(), B.cuda(), c["alpha"])
    qn.device_status()
    Wd = nf4.dequantize(nf4.quantize(c["W"], 64, dq=True)).reshape(d, k)
    Yref = layer.linear_fwd(X.numpy(), Wd, A.numpy(), B.numpy(), c["alpha"], r)
    dXref = layer.linear_bwd_dx(dY.numpy(), Wd, A.numpy(), B.numpy(), c["alpha"], r)
    assert Y.dtype == torch.float32 and dX.dtype == torch.float32
    assert layer.rel_fro(_f64(Y), Yref) < 1e-5, layer.rel_fro(_f64(Y), Yref)
    assert layer.rel_fro(_f64(dX), dXref) < 1e-5, layer.rel_fro(_f64(dX), dXref)


def test_fp32_layer_decode_shape(qn):
    m = synth.decode_matrix(seed=2, d=4096, k=11008, r=64, M=1)
    g = np.random.default_rng(1)
    X = torch.from_numpy(g.standard_normal((1, 11008)).astype(np.float32))
    A, B = m["A"].float(), m["B"].float()
    q = qn.nf4_quantize(torch.from_numpy(m["W"]).cuda())
    Y = qn.qlora_linear_fwd_f32(q, X.cuda(), A.cuda(), B.cuda(), m["alpha"])
    qn.device_status()
    Wd = nf4.dequantize(nf4.quantize(m["W"], 64, dq=True)).reshape(4096, 11008)
    Yref = layer.linear_fwd(X.numpy(), Wd, A.numpy(), B.numpy(), m["alpha"], 64)
    assert layer.rel_fro(_f64(Y), Yref) < 1e-5


# ---------------------------------------------------------------- merge

def _bits_equal(qt, ref, dq):
    assert np.array_equal(qt.codes.cpu().numpy(), ref.packed)
    assert np.array_equal(qt.absmax.cpu().numpy().view(np.uint32), ref.absmax.view(np.uint32))
    if dq:
        assert np.array_equal(qt.absmax_q.cpu().numpy(), ref.absmax_q)
        assert np.array_equal(qt.absmax_scale.cpu().numpy().view(np.uint32), ref.absmax_scale.view(np.uint32))
        assert qt.absmax_mean.cpu().numpy().view(np.uint32)[0] == np.float32(ref.absmax_mean).view(np.uint32)


@pytest.mark.parametrize("d,k,r,dq,sign", [
    (256, 512, 8, True, 1), (256, 512, 8, True, -1), (200, 320, 40, False, 1), (77, 64, 1, True, 1),
    (1024, 1024, 64, True, 1), (4096, 4096, 16, True, -1),
])
def test_merge_bit_exact(qn, d, k, r, dq, sign):
    c = synth.layer_case(seed=d + k + r, d=d, k=k, M=1, r=r, alpha=2.0 * r)
    B = (c["B"].float() * 8).to(torch.bfloat16)  # an adapter large enough to move many codes
    q = qn.nf4_quantize(torch.from_numpy(c["W"]).cuda(), dq=dq)
    qm = qn.nf4_merge_lora(q, c["A"].cuda(), B.cuda(), c["alpha"], sign)
    qn.device_status()
    ref = merge.merge(nf4.quantize(c["W"], 64, dq=dq), d, k, c["A"].float().numpy(), B.float().numpy(),
                      c["alpha"], r, sign)
    _bits_equal(qm, ref, dq)


def test_merge_in_place_and_round_trip(qn):
    d, k, r = 512, 768, 16
    c = synth.layer_case(seed=21, d=d, k=k, M=1, r=r, alpha=32.0)
    A, B = c["A"].cuda(), (c["B"].float() * 8).to(torch.bfloat16).cuda()
    q = qn.nf4_quantize(torch.from_numpy(c["W"]).cuda())
    codes0 = q.codes.clone()
    qn.nf4_merge_lora(q, A, B, c["alpha"], 1, out=q)      # in place
    qn.nf4_merge_lora(q, A, B, c["alpha"], -1, out=q)     # unmerge in place
    qn.device_status()
    ref = nf4.quantize(c["W"], 64, dq=True)
    ref = merge.merge(ref, d, k, c["A"].float().numpy(), B.float().cpu().numpy(), c["alpha"], r, 1)
    ref = merge.merge(ref, d, k, c["A"].float().numpy(), B.float().cpu().numpy(), c["alpha"], r, -1)
    _bits_equal(q, ref, True)
    assert not torch.equal(q.codes, codes0)               # the round trip drifts, as the pages say


# ---------------------------------------------------------- one-step LoftQ

@pytest.mark.parametrize("d,k,r,scale", [(256, 320, 8, 1.0), (1024, 1024, 16, 1.0), (512, 768, 4, 1.1)])
def test_loftq_replace_lora(qn, d, k, r, scale):
    W = synth.loftq_case(seed=7 + d, d=d, k=k)
    Wq = (W * np.float32(scale)).astype(np.float32)       # scale != 1: Q is not NF4(W)
    q = qn.nf4_quantize(torch.from_numpy(Wq).cuda())
    codes0 = q.codes.clone()
    A, B, res = qn.loftq_replace_lora(torch.from_numpy(W).cuda(), q, r, float(r), seed=3)
    qn.device_status()
    assert torch.equal(q.codes, codes0)                   # Q is kept as it is
    ref = loftq.loftq_one_step(W, nf4.quantize(Wq, 64, dq=True), r, float(r))
    assert abs(res[0] - ref.resid[0]) <= 1e-6 * ref.resid[0]
    assert abs(res[1] - ref.resid[1]) <= 1e-2 * ref.resid[1], (res, ref.resid)
    assert res[1] < res[0]
    # the returned factors reproduce the reported residual
    R = W.astype(np.float64) - nf4.dequantize(nf4.quantize(Wq, 64, dq=True)).reshape(d, k)
    s = 1.0
    e = np.linalg.norm(R - s * (B.cpu().double().numpy() @ A.cpu().double().numpy()))
    assert abs(e - res[1]) <= 1e-4 * res[1]
