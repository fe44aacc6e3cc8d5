"""GPU parity of the fused QLoRA layer (forward Y and backward dX) against the
float64 oracle.  Tolerance: relative Frobenius error <= 5e-3, the bound the
method's target fixes for layer outputs; the CUDA path rounds the dequantised
weight and the outputs to bf16 and accumulates in fp32, which stays well
inside it (typically ~2e-3)."""

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


def tile_max_rel(Y, Yref, rows=256, cols=128):
    """Largest relative Frobenius error over rows x cols tiles of the output
    (token tiles x weight-row tiles), so that one wrong tile cannot hide in
    the global norm."""
    Y = np.asarray(Y, np.float64)
    Yref = np.asarray(Yref, np.float64)
    worst = 0.0
    for i in range(0, Y.shape[0], rows):
        for j in range(0, Y.shape[1], cols):
            worst = max(worst, layer.rel_fro(Y[i:i + rows, j:j + cols], Yref[i:i + rows, j:j + cols]))
    return worst


def _run(qn, W, X, A, B, alpha, dY=None):
    q = qn.nf4_quantize(torch.from_numpy(W).cuda(), dq=True)
    ref = nf4.quantize(W, 64, dq=True)
    Wd = nf4.dequantize(ref).reshape(W.shape)
    Y = qn.qlora_linear_fwd(q, X.cuda(), A.cuda(), B.cuda(), alpha)
    out = {"Y": Y, "Yref": layer.linear_fwd(_f64(X), Wd, _f64(A), _f64(B), alpha, A.shape[0])}
    if dY is not None:
        dX = qn.qlora_linear_bwd_dx(q, dY.cuda(), A.cuda(), B.cuda(), alpha)
        out["dX"] = dX
        out["dXref"] = layer.linear_bwd_dx(_f64(dY), Wd, _f64(A), _f64(B), alpha, A.shape[0])
    qn.device_status()
    return out


def test_layer_case(qn):
    c = synth.layer_case(seed=0)
    o = _run(qn, c["W"], c["X"], c["A"], c["B"], c["alpha"], c["dY"])
    assert layer.rel_fro(_f64(o["Y"]), o["Yref"]) < TOL
    assert layer.rel_fro(_f64(o["dX"]), o["dXref"]) < TOL
    assert tile_max_rel(_f64(o["Y"]), o["Yref"], 16, 16) < TOL
    assert tile_max_rel(_f64(o["dX"]), o["dXref"], 16, 16) < TOL


@pytest.mark.parametrize("M,d,k,r", [
    (1, 256, 512, 8), (2, 200, 192, 3), (5, 384, 1024, 64), (16, 320, 256, 16),
    (17, 192, 320, 8), (100, 330, 256, 24), (300, 128, 640, 64), (129, 1000, 128, 1),
    # 8 < M <= 16: the K-slice kernel (k a multiple of 256, ragged rows and
    # tokens, one and several tiles per CTA, a second batch of tiles per CTA)
    # and the row-group kernel (k not)
    (12, 1000, 512, 8), (9, 3000, 768, 24), (12, 200, 320, 8), (12, 30000, 256, 8), (12, 1000, 1024, 8),
    # M <= 8 with x too large for the few-token kernel: the row-group kernel
    (6, 256, 4096, 16),
])
def test_shapes_with_ragged_tails(qn, M, d, k, r):
    c = synth.layer_case(seed=M * 7 + d, d=d, k=k, M=M, r=r, alpha=2.0 * r)
    o = _run(qn, c["W"], c["X"], c["A"], c["B"], c["alpha"], c["dY"])
    assert layer.rel_fro(_f64(o["Y"]), o["Yref"]) < TOL, (M, d, k, r)
    assert layer.rel_fro(_f64(o["dX"]), o["dXref"]) < TOL, (M, d, k, r)
    assert tile_max_rel(_f64(o["Y"]), o["Yref"], 64, 16) < TOL, (M, d, k, r)
    assert tile_max_rel(_f64(o["dX"]), o["dXref"], 64, 64) < TOL, (M, d, k, r)


def test_degenerate_adapter_and_weight(qn):
    c = synth.layer_case(seed=9, d=256, k=256, M=24, r=8)
    zB = torch.zeros_like(c["B"])
    o = _run(qn, c["W"], c["X"], c["A"], zB, c["alpha"], c["dY"])          # B = 0: plain GEMM
    assert layer.rel_fro(_f64(o["Y"]), o["Yref"]) < TOL
    Wz = np.zeros((256, 256), np.float32)                                    # deq(Q) = 0: pure adapter
    o = _run(qn, Wz, c["X"], c["A"], c["B"], c["alpha"], c["dY"])
    assert layer.rel_fro(_f64(o["Y"]), o["Yref"]) < TOL
    assert layer.rel_fro(_f64(o["dX"]), o["dXref"]) < TOL


@pytest.mark.parametrize("shape", [(4096, 4096), (11008, 4096), (4096, 11008)])
@pytest.mark.parametrize("M", [1, 16])
def test_decode_shapes(qn, shape, M):
    d, k = shape
    m = synth.decode_matrix(seed=1, d=d, k=k, r=64, M=M)
    o = _run(qn, m["W"], m["X"], m["A"], m["B"], m["alpha"])
    assert layer.rel_fro(_f64(o["Y"]), o["Yref"]) < TOL
    assert tile_max_rel(_f64(o["Y"]), o["Yref"], 16, 16) < TOL   # every 16-row tile of W


def test_prefill_full_size_sampled_rows(qn):
    """M=4096, d=11008, k=4096, r=16: full Y and dX on the GPU; the oracle
    checks 48 sampled token rows of each (the full float64 product is 0.7
    TFLOP), three from every 256-token tile, and every 128-column tile of
    those rows on its own."""
    c = synth.prefill_case(seed=2)
    W = c["W"]
    q = qn.nf4_quantize(torch.from_numpy(W).cuda(), dq=True)
    Y = qn.qlora_linear_fwd(q, c["X"].cuda(), c["A"].cuda(), c["B"].cuda(), c["alpha"])
    dX = qn.qlora_linear_bwd_dx(q, c["dY"].cuda(), c["A"].cuda(), c["B"].cuda(), c["alpha"])
    qn.device_status()
    ref = nf4.quantize(W, 64, dq=True)
    Wd = nf4.dequantize(ref).reshape(W.shape)
    g = np.random.default_rng(2)
    rows = np.sort(np.concatenate([t0 + g.choice(256, 3, replace=False) for t0 in range(0, c["M"], 256)]))
    A, B = _f64(c["A"]), _f64(c["B"])
    Yref = layer.linear_fwd(_f64(c["X"])[rows], Wd, A, B, c["alpha"], c["r"])
    dXref = layer.linear_bwd_dx(_f64(c["dY"])[rows], Wd, A, B, c["alpha"], c["r"])
    assert layer.rel_fro(_f64(Y)[rows], Yref) < TOL
    assert layer.rel_fro(_f64(dX)[rows], dXref) < TOL
    assert tile_max_rel(_f64(Y)[rows], Yref, 3, 128) < TOL      # 3 rows of one token tile x 128 weight rows
    assert tile_max_rel(_f64(dX)[rows], dXref, 3, 128) < TOL
    # every output finite and of the right scale
    assert torch.isfinite(Y.float()).all() and torch.isfinite(dX.float()).all()


def test_host_buffers_round_trip(qn):
    """The host-buffer path copies X in and Y out around the same kernels."""
    c = synth.layer_case(seed=4, d=512, k=512, M=1, r=8)
    q = qn.nf4_quantize(torch.from_numpy(c["W"]).cuda())
    Xh = c["X"].pin_memory()
    Yh = qn.qlora_linear_fwd(q, Xh, c["A"].cuda(), c["B"].cuda(), c["alpha"])
    torch.cuda.synchronize()
    Yd = qn.qlora_linear_fwd(q, c["X"].cuda(), c["A"].cuda(), c["B"].cuda(), c["alpha"])
    assert not Yh.is_cuda
    assert torch.equal(Yh, Yd.cpu())


def test_decode_repeated_and_graph_replay(qn):
    """The single-token kernel hands off through workspace semaphores that it
    returns to zero: repeated calls and CUDA-graph replays must give the same
    bits and raise no device timeout."""
    m = synth.decode_matrix(seed=3, d=4096, k=4096, r=64, M=1)
    q = qn.nf4_quantize(torch.from_numpy(m["W"]).cuda())
    X, A, B = m["X"].cuda(), m["A"].cuda(), m["B"].cuda()
    Y1 = qn.qlora_linear_fwd(q, X, A, B, m["alpha"]).clone()
    Y2 = qn.qlora_linear_fwd(q, X, A, B, m["alpha"]).clone()
    out = torch.empty_like(Y1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        qn.qlora_linear_fwd(q, X, A, B, m["alpha"], out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        qn.qlora_linear_fwd(q, X, A, B, m["alpha"], out=out)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, Y1)
    qn.device_status()
    assert torch.equal(Y1, Y2)


@pytest.mark.parametrize("M", [1, 4])
def test_chain_reads_previous_output(qn, M):
    """Each call's input is the previous call's output.  The few-token kernels
    are launched as programmatic dependents (start early, read x only after
    griddepcontrol.wait) and the single-token kernel in plain stream order;
    either way x must be read only once the call before has written it.  The
    outputs start as NaN, so a read that comes too early shows; every link
    must equal that link recomputed alone after a synchronise, eagerly and
    replayed in one CUDA graph."""
    d = k = 4096
    n = 6
    m = synth.decode_matrix(seed=5, d=d, k=k, r=16, M=M)
    q = qn.nf4_quantize(torch.from_numpy(m["W"]).cuda())
    A, B, X0 = m["A"].cuda(), m["B"].cuda(), m["X"].cuda()
    ys = [torch.empty((M, d), dtype=torch.bfloat16, device="cuda") for _ in range(n)]

    def chain():
        x = X0
        for y in ys:
            qn.qlora_linear_fwd(q, x, A, B, m["alpha"], out=y)
            x = y

    def check():
        prev = X0
        for i, y in enumerate(ys):
            ref = qn.qlora_linear_fwd(q, prev, A, B, m["alpha"])
            torch.cuda.synchronize()
            assert torch.isfinite(y.float()).all(), i
            assert torch.equal(y, ref), i
            prev = y

    for y in ys:
        y.fill_(float("nan"))
    chain()
    torch.cuda.synchronize()
    check()
    eager = [y.clone() for y in ys]

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        chain()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    for rep in range(2):
        for y in ys:
            y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for i, (y, e) in enumerate(zip(ys, eager)):
            assert torch.equal(y, e), (rep, i)
    qn.device_status()


@pytest.mark.parametrize("M", [1, 3, 12])
def test_group_of_projections(qn, M):
    """Projections of one input in one call (query/key/value style), with
    different d and r per member, against the oracle one by one."""
    g = np.random.default_rng(40 + M)
    k = 1536
    shapes = [(512, 8), (768, 16), (320, 4)]
    X = synth.to_bf16(g.standard_normal((M, k), dtype=np.float32))
    qs, As, Bs, alphas, refs = [], [], [], [], []
    for i, (d, r) in enumerate(shapes):
        c = synth.layer_case(seed=100 + i, d=d, k=k, M=M, r=r, alpha=2.0 * r)
        qs.append(qn.nf4_quantize(torch.from_numpy(c["W"]).cuda()))
        As.append(c["A"].cuda()); Bs.append(c["B"].cuda()); alphas.append(c["alpha"])
        Wd = nf4.dequantize(nf4.quantize(c["W"], 64, dq=True)).reshape(d, k)
        refs.append(layer.linear_fwd(_f64(X), Wd, _f64(c["A"]), _f64(c["B"]), c["alpha"], r))
    Ys = qn.qlora_linear_fwd_group(qs, X.cuda(), As, Bs, alphas)
    qn.device_status()
    for Y, ref in zip(Ys, refs):
        assert layer.rel_fro(_f64(Y), ref) < TOL
    # same bits as the single-projection calls
    for q, A, B, a, Y in zip(qs, As, Bs, alphas, Ys):
        assert torch.equal(qn.qlora_linear_fwd(q, X.cuda(), A, B, a), Y)


@pytest.mark.parametrize("M", [1, 4])
def test_forward_right_after_its_inputs_are_written(qn, M):
    """The forward starts as a programmatic dependent of the kernel before it.
    Here that kernel writes the forward's own operands: nf4_quantize writes Q
    (its last kernel writes the DQ codes and scales) and a torch copy writes
    A and B, each immediately before the call.  Q starts as garbage (codes
    0xFF, scales NaN) and A, B as NaN, so a read that comes too early shows.
    Checked eagerly and in a CUDA graph replay against the same call made
    after a synchronise."""
    d = k = 4096
    m = synth.decode_matrix(seed=6, d=d, k=k, r=16, M=M)
    W = torch.from_numpy(m["W"]).cuda()
    A0, B0, X = m["A"].cuda(), m["B"].cuda(), m["X"].cuda()
    q = qn.NF4Tensor.empty(d, k, True, "cuda")
    A = torch.empty_like(A0)
    B = torch.empty_like(B0)
    Y = torch.empty((M, d), dtype=torch.bfloat16, device="cuda")
    qref = qn.nf4_quantize(W)
    ref = qn.qlora_linear_fwd(qref, X, A0, B0, m["alpha"])
    torch.cuda.synchronize()

    def poison():
        q.codes.fill_(0xFF)
        q.absmax_q.fill_(127)
        q.absmax_scale.fill_(float("nan"))
        A.fill_(float("nan"))
        B.fill_(float("nan"))
        Y.fill_(float("nan"))

    def step():
        qn.nf4_quantize(W, out=q)
        A.copy_(A0)
        B.copy_(B0)
        qn.qlora_linear_fwd(q, X, A, B, m["alpha"], out=Y)

    for _ in range(2):
        poison()
        torch.cuda.synchronize()
        step()
        torch.cuda.synchronize()
        assert torch.equal(Y, ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        poison()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(Y, ref)
    qn.device_status()


@pytest.mark.parametrize("M", [1, 4])
def test_small_m_adapter_term_on_its_own(qn, M):
    """The single-kernel path for M <= 8 forms the adapter term u . B[row] in a
    separate warp and hands it to the epilogue.  With W = 0 (every code is the
    exact zero) Y is that term alone, so a missing or stale hand-off shows in
    every tile; a large adapter on a grouped call checks it next to X W^T."""
    k = 4096
    g = np.random.default_rng(70 + M)
    X = synth.to_bf16(g.standard_normal((M, k), dtype=np.float32))
    qs, As, Bs, refs = [], [], [], []
    for i, d in enumerate((4096, 4096, 1024)):
        W = np.zeros((d, k), np.float32) if i == 0 else (g.standard_normal((d, k)) * 0.02).astype(np.float32)
        A = synth.to_bf16((g.standard_normal((64, k)) / np.sqrt(k)).astype(np.float32))
        B = synth.to_bf16((g.standard_normal((d, 64)) * (1.0 if i else 0.05)).astype(np.float32))
        qs.append(qn.nf4_quantize(torch.from_numpy(W).cuda()))
        As.append(A.cuda()); Bs.append(B.cuda())
        Wd = nf4.dequantize(nf4.quantize(W, 64, dq=True)).reshape(d, k)
        refs.append(layer.linear_fwd(_f64(X), Wd, _f64(A), _f64(B), 16.0, 64))
    Ys = qn.qlora_linear_fwd_group(qs, X.cuda(), As, Bs, [16.0] * 3)
    qn.device_status()
    for Y, ref in zip(Ys, refs):
        assert layer.rel_fro(_f64(Y), ref) < TOL
        assert tile_max_rel(_f64(Y), ref, 16, 16) < TOL
    # the same projections one at a time
    for q, A, B, ref in zip(qs, As, Bs, refs):
        Y = qn.qlora_linear_fwd(q, X.cuda(), A, B, 16.0)
        qn.device_status()
        assert tile_max_rel(_f64(Y), ref, 16, 16) < TOL


@pytest.mark.parametrize("M", [1, 3])
def test_few_token_exact_and_mixed_block_constants(qn, M):
    """The M <= 8 kernel decodes the block constants straight from global
    memory: fp32 absmax (dq = False) four blocks at a time when the number of
    blocks per row is a multiple of 4 and one at a time otherwise, and a
    grouped call whose projections mix fp32 and double-quantised constants."""
    g = np.random.default_rng(90 + M)

    def proj(d, k, dq, r):
        W = (g.standard_normal((d, k)) * 0.02).astype(np.float32)
        A = synth.to_bf16((g.standard_normal((r, k)) / np.sqrt(k)).astype(np.float32))
        B = synth.to_bf16((g.standard_normal((d, r)) * 0.05).astype(np.float32))
        q = qn.nf4_quantize(torch.from_numpy(W).cuda(), dq=dq)
        Wd = nf4.dequantize(nf4.quantize(W, 64, dq=dq)).reshape(d, k)
        return q, A, B, Wd

    for d, k in ((300, 512), (200, 192)):  # 8 and 3 blocks per row
        X = synth.to_bf16(g.standard_normal((M, k), dtype=np.float32))
        q, A, B, Wd = proj(d, k, False, 8)
        Y = qn.qlora_linear_fwd(q, X.cuda(), A.cuda(), B.cuda(), 16.0)
        qn.device_status()
        ref = layer.linear_fwd(_f64(X), Wd, _f64(A), _f64(B), 16.0, 8)
        assert tile_max_rel(_f64(Y), ref, 16, 16) < TOL, (d, k)
    k = 512
    X = synth.to_bf16(g.standard_normal((M, k), dtype=np.float32))
    parts = [proj(256, k, True, 16), proj(130, k, False, 8), proj(70, k, True, 4)]
    Ys = qn.qlora_linear_fwd_group([p[0] for p in parts], X.cuda(), [p[1].cuda() for p in parts],
                                   [p[2].cuda() for p in parts], [16.0] * 3)
    qn.device_status()
    for Y, (q, A, B, Wd) in zip(Ys, parts):
        ref = layer.linear_fwd(_f64(X), Wd, _f64(A), _f64(B), 16.0, A.shape[0])
        assert tile_max_rel(_f64(Y), ref, 16, 16) < TOL

