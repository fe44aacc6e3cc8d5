"""nf4_quantize_noalloc: the quantiser entry point that allocates nothing.

It serves callers that cannot call cudaMalloc (another allocator owns the
free device memory, or the caller's loop cannot take the device-wide
synchronisation an allocation implies): its 2.25 KiB of scratch is a static
device array inside the library.  This test calls it through the C ABI and
checks every output against the allocating entry point nf4_quantize (the
codec's tolerance: bit-exact), on two calls in a row with different inputs,
so a stale scratch from the first call would show up in the second.  The
file sorts last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

FIELDS = ("codes", "absmax", "absmax_q", "absmax_scale", "absmax_mean")


def _noalloc(qn, W, q):
    st = q.c_struct()
    dt = qn.QN_F32 if W.dtype == torch.float32 else qn.QN_BF16
    status = qn.lib.nf4_quantize_noalloc(W.data_ptr(), dt, ctypes.byref(st),
                                         torch.cuda.current_stream().cuda_stream)
    assert status == qn.QN_OK, qn.lib.qn_last_error().decode()


def test_noalloc_quantize_matches_allocating_entry_point():
    assert torch.cuda.is_available(), "GPU test needs CUDA"
    import bit_nf4_quantized_39_b300 as qn

    cases = [synth.layer_case(seed=21, d=768, k=1024)["W"],
             synth.decode_matrix(seed=22, d=1000, k=448)["W"] * np.float32(7.0)]
    for W_host in cases:                       # two calls in a row
        W = torch.from_numpy(W_host).cuda()
        want = qn.nf4_quantize(W, dq=True)
        got = qn.NF4Tensor.empty(W.shape[0], W.shape[1], True, W.device)
        _noalloc(qn, W, got)
        qn.device_status()
        for f in FIELDS:
            a = getattr(got, f).cpu().numpy()
            b = getattr(want, f).cpu().numpy()
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), f
    # bf16 input through the same scratch
    Wb = torch.from_numpy(cases[0]).to(torch.bfloat16).cuda()
    want = qn.nf4_quantize(Wb, dq=True)
    got = qn.NF4Tensor.empty(Wb.shape[0], Wb.shape[1], True, Wb.device)
    _noalloc(qn, Wb, got)
    torch.cuda.synchronize()
    for f in FIELDS:
        assert torch.equal(getattr(got, f), getattr(want, f)), f
