"""GPU parity of the tensor-core forward and backward (M > 16, r <= 64, the tcgen05 kernels)
against the float64 oracle, relative Frobenius error <= 5e-3.

The shapes put ragged edges on every tile boundary of that kernel: weight
rows not a multiple of 128, token counts below, at and above one 256-token
tile, a single 64-column stage, padded adapter ranks (r = 1, 33, 40) and the
largest rank it takes (64), and forward grids of several waves of tiles
(more tiles than SMs); r = 65 checks the CUDA-core kernel that takes over
above that rank."""

import numpy as np
import pytest
import torch

import synth
from oracle import layer, nf4

pytestmark = pytest.mark.gpu

TOL = 5e-3


@pytest.fixture(scope="module")
def qn():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import bit_nf4_quantized_39_b300 as mod
    return mod


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _fwd(qn, W, X, A, B, alpha, dq=True):
    q = qn.nf4_quantize(torch.from_numpy(W).cuda(), dq=dq)
    Wd = nf4.dequantize(nf4.quantize(W, 64, dq=dq)).reshape(W.shape)
    Y = qn.qlora_linear_fwd(q, X.cuda(), A.cuda(), B.cuda(), alpha)
    qn.device_status()
    return _f64(Y), layer.linear_fwd(_f64(X), Wd, _f64(A), _f64(B), alpha, A.shape[0])


@pytest.mark.parametrize("M,d,k,r", [
    (17, 128, 64, 8), (256, 256, 128, 16), (257, 384, 192, 1), (300, 200, 576, 33),
    (600, 1000, 256, 64), (1024, 512, 1024, 40), (40, 130, 64, 65),
    # more tiles than SMs: the grid runs in several waves; ragged rows and tokens
    (1300, 6500, 128, 24), (2100, 2600, 320, 64),
])
def test_tc_forward_shapes(qn, M, d, k, r):
    c = synth.layer_case(seed=M + 3 * d + k, d=d, k=k, M=M, r=r, alpha=2.0 * r)
    Y, ref = _fwd(qn, c["W"], c["X"], c["A"], c["B"], c["alpha"])
    assert layer.rel_fro(Y, ref) < TOL, (M, d, k, r)


def test_tc_forward_exact_absmax(qn):
    c = synth.layer_case(seed=5, d=384, k=320, M=200, r=16)
    Y, ref = _fwd(qn, c["W"], c["X"], c["A"], c["B"], c["alpha"], dq=False)
    assert layer.rel_fro(Y, ref) < TOL


def test_tc_forward_degenerate_terms(qn):
    c = synth.layer_case(seed=6, d=256, k=256, M=300, r=8)
    Y, ref = _fwd(qn, c["W"], c["X"], c["A"], torch.zeros_like(c["B"]), c["alpha"])  # no adapter
    assert layer.rel_fro(Y, ref) < TOL
    Y, ref = _fwd(qn, np.zeros((256, 256), np.float32), c["X"], c["A"], c["B"], c["alpha"])  # adapter only
    assert layer.rel_fro(Y, ref) < TOL


# W = 0 isolates the adapter term s (X A^T) B^T; ranks up to 16 take the
# single-pass projection (one CTA per 16 tokens over all of K), including a
# ragged last token block, K shorter than one 256-column stage, and odd ranks.
@pytest.mark.parametrize("M,d,k,r", [(1000, 512, 1024, 16), (33, 128, 4096, 3), (129, 256, 64, 11)])
def test_tc_forward_adapter_only(qn, M, d, k, r):
    c = synth.layer_case(seed=M + d + k + r, d=d, k=k, M=M, r=r, alpha=2.0 * r)
    Y, ref = _fwd(qn, np.zeros((d, k), np.float32), c["X"], c["A"], c["B"], c["alpha"])
    assert layer.rel_fro(Y, ref) < TOL, (M, d, k, r)


def _bwd(qn, W, dY, A, B, alpha, dq=True):
    q = qn.nf4_quantize(torch.from_numpy(W).cuda(), dq=dq)
    Wd = nf4.dequantize(nf4.quantize(W, 64, dq=dq)).reshape(W.shape)
    dX = qn.qlora_linear_bwd_dx(q, dY.cuda(), A.cuda(), B.cuda(), alpha)
    qn.device_status()
    return _f64(dX), layer.linear_bwd_dx(_f64(dY), Wd, _f64(A), _f64(B), alpha, A.shape[0])


# The backward runs on the tensor cores for M > 16, r <= 64 and d a multiple
# of 8 (dequantised W^T in the workspace, then a tcgen05 GEMM); the shapes put
# ragged edges on its 128-column and 256-token tiles and on the K = d loop.
@pytest.mark.parametrize("M,d,k,r", [
    (17, 128, 64, 8), (256, 256, 128, 16), (257, 384, 192, 1), (300, 200, 576, 33),
    (600, 1000, 256, 64), (1024, 520, 1024, 40), (40, 130, 64, 65),
])
def test_tc_backward_shapes(qn, M, d, k, r):
    c = synth.layer_case(seed=M + 5 * d + k, d=d, k=k, M=M, r=r, alpha=2.0 * r)
    dX, ref = _bwd(qn, c["W"], c["dY"], c["A"], c["B"], c["alpha"])
    assert layer.rel_fro(dX, ref) < TOL, (M, d, k, r)


def test_tc_backward_exact_absmax_and_degenerate(qn):
    c = synth.layer_case(seed=7, d=384, k=320, M=200, r=16)
    dX, ref = _bwd(qn, c["W"], c["dY"], c["A"], c["B"], c["alpha"], dq=False)
    assert layer.rel_fro(dX, ref) < TOL
    dX, ref = _bwd(qn, c["W"], c["dY"], torch.zeros_like(c["A"]), c["B"], c["alpha"])   # no adapter
    assert layer.rel_fro(dX, ref) < TOL
    dX, ref = _bwd(qn, np.zeros((384, 320), np.float32), c["dY"], c["A"], c["B"], c["alpha"])  # adapter only
    assert layer.rel_fro(dX, ref) < TOL


def test_prefill_calls_in_a_graph_match_eager(qn):
    """The large-M forward, backward dX and adapter gradients run part of
    their work on a second stream (event fork / join).  Captured in a CUDA
    graph and replayed, they must give the same bits as the eager calls."""
    c = synth.layer_case(seed=11, d=1000, k=256, M=600, r=16, alpha=32.0)
    q = qn.nf4_quantize(torch.from_numpy(c["W"]).cuda())
    X, dY = c["X"].cuda(), c["dY"].cuda()
    A, B = c["A"].cuda(), c["B"].cuda()
    Y0 = qn.qlora_linear_fwd(q, X, A, B, c["alpha"])
    dX0 = qn.qlora_linear_bwd_dx(q, dY, A, B, c["alpha"])
    dA0, dB0 = qn.qlora_linear_bwd_lora(X, dY, A, B, c["alpha"])
    torch.cuda.synchronize()
    Y1, dX1 = torch.empty_like(Y0), torch.empty_like(dX0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up on the capture stream (workspace allocation)
        qn.qlora_linear_fwd(q, X, A, B, c["alpha"], out=Y1)
        qn.qlora_linear_bwd_dx(q, dY, A, B, c["alpha"], out=dX1)
        qn.qlora_linear_bwd_lora(X, dY, A, B, c["alpha"])
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        qn.qlora_linear_fwd(q, X, A, B, c["alpha"], out=Y1)
        qn.qlora_linear_bwd_dx(q, dY, A, B, c["alpha"], out=dX1)
        dA1, dB1 = qn.qlora_linear_bwd_lora(X, dY, A, B, c["alpha"])
    Y1.zero_(); dX1.zero_()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    qn.device_status()
    assert torch.equal(Y1, Y0)
    assert torch.equal(dX1, dX0)
    assert torch.equal(dA1, dA0) and torch.equal(dB1, dB0)
