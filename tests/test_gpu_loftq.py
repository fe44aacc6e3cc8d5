"""GPU parity of LoftQ: residuals ||W - deq(Q_t) - s B_t A_t||_F within 1% of
the oracle's (exact SVD) at every alternation, plus structural checks.  The
GPU path takes the rank-r step by randomised subspace iteration, so only the
residuals (not the factors) are compared."""

import json
import os

import numpy as np
import pytest
import torch

import synth
from oracle import loftq, nf4

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "loftq_4096_r16_T5.json")


@pytest.fixture(scope="module")
def qn():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import bit_nf4_quantized_39_b300 as mod
    return mod


# Panels of 32, 64 and 96 columns: r + oversample = 12, 16, 24 (32); 40 (64); 72 and 96 (96).
@pytest.mark.parametrize("d,k,r,T", [(256, 256, 8, 3), (512, 384, 16, 5), (192, 640, 4, 2), (1024, 1024, 64, 3),
                                     (384, 512, 32, 2), (320, 448, 88, 2)])
def test_small_against_oracle(qn, d, k, r, T):
    W = synth.loftq_case(seed=4, d=d, k=k)
    q, A, B, resid = qn.loftq_init(torch.from_numpy(W).cuda(), r=r, alpha=float(r), T=T, seed=1,
                                   oversample=8, power_iters=4)
    qn.device_status()
    ref = loftq.loftq(W, r=r, alpha=float(r), T=T)
    assert len(resid) == T + 1
    # t = 0 is plain QLoRA: identical quantiser, so equal up to fp64 summation order
    assert abs(resid[0] - ref.resid[0]) <= 1e-6 * ref.resid[0]
    for t in range(1, T + 1):
        assert abs(resid[t] - ref.resid[t]) <= 0.01 * ref.resid[t], (t, resid[t], ref.resid[t])
    # returned state: Q is NF4 of W - s B_{T-1} A_{T-1}; residual with returned A, B matches resid[T]
    Wd = qn.nf4_dequantize(q, torch.float32).double()
    R = torch.from_numpy(W).cuda().double() - Wd - (B.double() @ A.double())
    assert abs(torch.linalg.norm(R).item() - resid[T]) <= 1e-4 * resid[T]


def test_rank_above_the_panel_limit_is_rejected(qn):
    W = torch.from_numpy(synth.loftq_case(seed=4, d=256, k=256)).cuda()
    with pytest.raises(qn.QnError):
        qn.loftq_init(W, r=90, alpha=90.0, T=1, oversample=8)      # 98 > 96


def test_T0_equals_plain_quantizer(qn):
    W = synth.loftq_case(seed=4, d=128, k=256)
    q, A, B, resid = qn.loftq_init(torch.from_numpy(W).cuda(), r=4, alpha=4.0, T=0)
    ref = nf4.quantize(W, 64, dq=True)
    assert np.array_equal(q.codes.cpu().numpy(), ref.packed)
    assert not A.any() and not B.any()
    assert len(resid) == 1


def test_full_size_against_stored_oracle(qn):
    """4096 x 4096 Student-t weights, r=16, T=5, oversample 8, 4 power
    iterations; stored oracle residuals from tests/golden/make_loftq_golden.py."""
    with open(GOLDEN) as f:
        gold = json.load(f)["resid"]
    W = synth.loftq_case(seed=4)
    _, _, _, resid = qn.loftq_init(torch.from_numpy(W).cuda(), r=16, alpha=16.0, T=5, seed=0,
                                   oversample=8, power_iters=4)
    qn.device_status()
    for t, (a, b) in enumerate(zip(resid, gold)):
        assert abs(a - b) <= 0.01 * b, (t, a, b)
