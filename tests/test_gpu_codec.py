"""GPU parity of the NF4 codec against the CPU oracle: bit-exact codes, block
absmax, double-quantisation bytes, and bit-exact fp32 / bf16 dequantisation.
Every call goes through the C ABI (via the ctypes binding)."""

import numpy as np
import pytest
import torch

import synth
from oracle import exact, nf4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qn():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import bit_nf4_quantized_39_b300 as mod
    return mod


def _check_state(q, ref, sample_blocks=None):
    codes = q.codes.cpu().numpy()
    if sample_blocks is None:
        assert np.array_equal(codes[:ref.packed.size], ref.packed)
    else:
        for b in sample_blocks:
            assert np.array_equal(codes[b * 32:(b + 1) * 32], ref.packed[b * 32:(b + 1) * 32]), b
    nblk = ref.absmax.size
    assert np.array_equal(q.absmax.cpu().numpy()[:nblk].view(np.uint32), ref.absmax.view(np.uint32))
    if ref.dq:
        assert np.array_equal(q.absmax_q.cpu().numpy()[:nblk], ref.absmax_q)
        assert np.array_equal(q.absmax_scale.cpu().numpy()[:ref.absmax_scale.size].view(np.uint32),
                              ref.absmax_scale.view(np.uint32))
        assert q.absmax_mean.cpu().numpy()[0].view(np.uint32) == np.float32(ref.absmax_mean).view(np.uint32)


def _quant_both(qn, W_host, dq=True, bf16=False):
    if bf16:
        Wt = torch.from_numpy(W_host).to(torch.bfloat16)
        W32 = Wt.float().numpy()
        Wd = Wt.cuda()
    else:
        W32 = W_host
        Wd = torch.from_numpy(W_host).cuda()
    q = qn.nf4_quantize(Wd, dq=dq)
    torch.cuda.synchronize()
    return q, nf4.quantize(W32, 64, dq=dq), W32


def test_layer_case_quantize_dequantize_bitexact(qn):
    c = synth.layer_case(seed=0)
    q, ref, _ = _quant_both(qn, c["W"])
    _check_state(q, ref)
    w32 = qn.nf4_dequantize(q, torch.float32).cpu().numpy().reshape(-1)
    assert np.array_equal(w32.view(np.uint32), nf4.dequantize(ref).view(np.uint32))
    w16 = qn.nf4_dequantize(q, torch.bfloat16).view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)
    assert np.array_equal(w16, nf4.dequantize_bf16_bits(ref))
    qn.device_status()


@pytest.mark.parametrize("dq", [True, False])
def test_adversarial_blocks(qn, dq):
    v = synth.adversarial_block_values(seed=3, cb=nf4.codebook(), nblocks=640)
    q, ref, _ = _quant_both(qn, v.reshape(64, -1), dq=dq)
    _check_state(q, ref)
    w = qn.nf4_dequantize(q, torch.float32).cpu().numpy().reshape(-1)
    assert np.array_equal(w.view(np.uint32), nf4.dequantize(ref).view(np.uint32))


def _oracle_thresholds():
    """Decision points of the oracle's codebook: exact midpoints, rounded to
    fp32 both ways (the values a division lands on or next to)."""
    from fractions import Fraction
    cb = nf4.codebook()
    pts = []
    for i in range(15):
        mid = (Fraction(float(cb[i])) + Fraction(float(cb[i + 1]))) / 2
        f = np.float32(float(mid))
        pts += [f, np.nextafter(f, np.float32(-1)), np.nextafter(f, np.float32(1))]
    return np.array(pts + list(cb), dtype=np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_near_threshold_values(qn, dtype):
    """Quotients x/m on and around every decision threshold: the GPU's
    division and nearest-level decision must agree with IEEE division and the
    brute-force argmin bit for bit."""
    v = synth.near_point_blocks(seed=17, points=_oracle_thresholds(), nblocks=4000)
    q, ref, _ = _quant_both(qn, v.reshape(250, -1), bf16=(dtype == "bf16"))
    _check_state(q, ref)


@pytest.mark.parametrize("n", [1, 2, 63, 64, 65, 127, 64 * 257 + 5, 1_000_003])
def test_ragged_lengths(qn, n):
    g = np.random.default_rng(n)
    x = (g.standard_normal(n) * 0.02).astype(np.float32).reshape(1, n)
    q, ref, _ = _quant_both(qn, x)
    _check_state(q, ref)
    for dt, conv in ((torch.float32, lambda a: a.view(np.uint32)),
                     (torch.bfloat16, None)):
        out = qn.nf4_dequantize(q, dt)
        if dt == torch.float32:
            assert np.array_equal(out.cpu().numpy().reshape(-1).view(np.uint32), nf4.dequantize(ref).view(np.uint32))
        else:
            got = out.view(torch.int16).cpu().numpy().reshape(-1).view(np.uint16)
            assert np.array_equal(got, nf4.dequantize_bf16_bits(ref))


@pytest.mark.parametrize("n", [1, 63, 64, 65, 64 * 8 - 1, 64 * 9, 64 * 257 + 5, 1_000_003])
def test_ragged_lengths_bf16_input(qn, n):
    """bf16 input: stages of 8 blocks, so a partial last stage for n/64 not a
    multiple of 8, and fewer stages than warps for the small cases."""
    g = np.random.default_rng(n + 7)
    x = (g.standard_normal(n) * 0.02).astype(np.float32).reshape(1, n)
    q, ref, _ = _quant_both(qn, x, bf16=True)
    _check_state(q, ref)


def test_bf16_input(qn):
    g = synth.rng(11)
    W = synth.with_outliers_exact(g, synth.normal(g, (512, 768), 0.02), 0.001, 0.2)
    q, ref, _ = _quant_both(qn, W, bf16=True)
    _check_state(q, ref)


def test_special_values(qn):
    x = np.zeros((4, 64 * 4), dtype=np.float32)
    x[0, :64] = 0.0                                   # all-zero block
    x[0, 64] = -1e-40                                 # subnormal absmax
    x[0, 65] = 5e-41
    x[1, :64] = np.float32(3e38) * np.linspace(-1, 1, 64, dtype=np.float32)   # near FLT_MAX
    x[2, :] = np.float32(1.0)                         # constant blocks -> code 15
    x[3, :] = -np.float32(2.0) ** -126                # smallest normal, negative
    q, ref, _ = _quant_both(qn, x)
    _check_state(q, ref)


def test_repeat_calls_identical(qn):
    """Launch-shape independence and no state carried between calls."""
    c = synth.layer_case(seed=5, d=1536, k=1024)
    Wd = torch.from_numpy(c["W"]).cuda()
    a = qn.nf4_quantize(Wd)
    b = qn.nf4_quantize(Wd)
    torch.cuda.synchronize()
    for f in ("codes", "absmax", "absmax_q", "absmax_scale", "absmax_mean"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f


def test_full_size_decode_matrix_sampled(qn):
    """11008 x 4096 with outliers (a gate/up projection of the decode set):
    all constants bit-exact, codes bit-exact on 512 sampled blocks, dequant
    bit-exact on the same blocks."""
    m = synth.decode_matrix(seed=1, d=11008, k=4096)
    W = m["W"]
    Wd = torch.from_numpy(W).to(torch.bfloat16).cuda()
    W32 = Wd.float().cpu().numpy()
    q = qn.nf4_quantize(Wd, dq=True)
    torch.cuda.synchronize()
    flat = W32.reshape(-1)
    absmax = nf4.block_absmax(flat, 64)
    qd, sig, mu = nf4.double_quant(absmax, 256)
    assert np.array_equal(q.absmax.cpu().numpy().view(np.uint32), absmax.view(np.uint32))
    assert np.array_equal(q.absmax_q.cpu().numpy(), qd)
    assert np.array_equal(q.absmax_scale.cpu().numpy().view(np.uint32), sig.view(np.uint32))
    assert q.absmax_mean.cpu().numpy()[0] == mu
    g = np.random.default_rng(0)
    blocks = np.sort(g.choice(absmax.size, 512, replace=False))
    codes = q.codes.cpu().numpy()
    cb = nf4.codebook()
    w16 = qn.nf4_dequantize(q, torch.bfloat16).view(torch.int16).cpu().numpy().reshape(-1).view(np.uint16)
    mprime = nf4.dequant_absmax(qd, sig, mu, 256)
    for b in blocks:
        seg = flat[b * 64:(b + 1) * 64]
        v = np.divide(seg, absmax[b], dtype=np.float32) if absmax[b] != 0 else np.zeros(64, np.float32)
        want = nf4.pack(nf4.nearest_code(v, cb))
        assert np.array_equal(codes[b * 32:(b + 1) * 32], want), b
        wv = np.multiply(cb[nf4.unpack(want, 64)], mprime[b], dtype=np.float32)
        assert np.array_equal(w16[b * 64:(b + 1) * 64], exact.f32_to_bf16_bits(wv)), b
