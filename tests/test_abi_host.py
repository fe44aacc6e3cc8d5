"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function include/qlora_nf4.h declares, its constant tables match the
oracle's independent construction, and argument errors come back as status
codes before anything is launched."""

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qlora_nf4.h")


@pytest.fixture(scope="module")
def qn():
    import __graft_entry__ as ge
    ge._build_module().build()      # no-op when the library is up to date
    import bit_nf4_quantized_39_b300 as mod
    return mod


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return")))


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ("nf4_quantize", "nf4_dequantize", "qlora_linear_fwd", "qlora_linear_bwd_dx", "loftq_init",
              "qlora_linear_bwd_lora", "qlora_linear_fwd_f32", "qlora_linear_bwd_dx_f32", "loftq_replace_lora",
              "nf4_merge_lora"):
        assert n in names


def test_library_exports_every_declared_symbol(qn):
    raw = ctypes.CDLL(qn.LIB_PATH)
    for n in header_functions():
        assert hasattr(raw, n), n
    assert set(header_functions()) <= set(qn.EXPORTS)
    assert qn.lib.qn_abi_version() == 2


def test_tables_match_oracle_codebook_and_thresholds(qn):
    from fractions import Fraction
    from oracle import nf4
    cb, th = qn.tables()
    ocb = nf4.codebook()
    assert np.array_equal(np.array(cb, dtype=np.float32).view(np.uint32), ocb.view(np.uint32))
    for i, t in enumerate(th):
        mid = (Fraction(float(ocb[i])) + Fraction(float(ocb[i + 1]))) / 2
        t32 = np.float32(t)
        assert Fraction(float(t32)) <= mid
        assert Fraction(float(np.nextafter(t32, np.float32(np.inf)))) > mid


def test_workspace_queries(qn):
    assert qn.workspace_bytes(qn.QN_OP_QUANTIZE, 0, 1024, 1024, 0) == 256 * 1024 + 2048
    assert qn.workspace_bytes(qn.QN_OP_DEQUANTIZE, 0, 1024, 1024, 0) == 0
    assert qn.workspace_bytes(qn.QN_OP_LINEAR_FWD, 1, 4096, 4096, 64) >= 4 * 64
    assert qn.workspace_bytes(qn.QN_OP_LINEAR_FWD, 0, 4096, 4096, 64) == 0
    lq = qn.workspace_bytes(qn.QN_OP_LOFTQ, 0, 4096, 4096, 16)
    assert lq >= 4096 * 4096 * 4


def _struct(qn, d=128, k=128, block=64, dq=1, dq_block=256, ptr=0x10000):
    return qn.qn_nf4(d, k, block, dq, dq_block, 0, ptr, ptr, ptr, ptr, ptr)


def _err(qn, status):
    return status, qn.lib.qn_last_error().decode()


def test_argument_errors_return_before_launch(qn):
    L = qn.lib
    P = 0x10000  # never dereferenced: every call below fails validation first
    st = _struct(qn)
    assert L.nf4_quantize(P, 0, None, P, 4096, None) == qn.QN_EINVAL
    bad_block = _struct(qn, block=32)
    assert L.nf4_quantize(P, 0, ctypes.byref(bad_block), P, 4096, None) == qn.QN_EUNSUPPORTED
    bad_dq = _struct(qn, dq_block=128)
    assert L.nf4_quantize(P, 0, ctypes.byref(bad_dq), P, 4096, None) == qn.QN_EUNSUPPORTED
    assert L.nf4_quantize(P, 7, ctypes.byref(st), P, 4096, None) == qn.QN_EINVAL
    assert L.nf4_quantize(P + 4, 0, ctypes.byref(st), P, 4096, None) == qn.QN_EALIGN
    assert L.nf4_quantize(P, 0, ctypes.byref(st), P, 16, None) == qn.QN_ENOMEM
    neg = _struct(qn, d=-1)
    assert L.nf4_quantize(P, 0, ctypes.byref(neg), P, 4096, None) == qn.QN_ESHAPE
    assert L.nf4_dequantize(ctypes.byref(st), None, 0, None) == qn.QN_EINVAL
    # layer: k % 64, r range, M range, alignment, workspace size
    odd_k = _struct(qn, k=100)
    assert L.qlora_linear_fwd(ctypes.byref(odd_k), P, 1, P, P, 8, 16.0, P, P, 1 << 20, None) == qn.QN_ESHAPE
    assert L.qlora_linear_fwd(ctypes.byref(st), P, 1, P, P, 0, 16.0, P, P, 1 << 20, None) == qn.QN_ESHAPE
    assert L.qlora_linear_fwd(ctypes.byref(st), P, 1, P, P, 300, 16.0, P, P, 1 << 20, None) == qn.QN_ESHAPE
    assert L.qlora_linear_fwd(ctypes.byref(st), P, 0, P, P, 8, 16.0, P, P, 1 << 20, None) == qn.QN_ESHAPE
    assert L.qlora_linear_fwd(ctypes.byref(st), P + 2, 1, P, P, 8, 16.0, P, P, 1 << 20, None) == qn.QN_EALIGN
    assert L.qlora_linear_fwd(ctypes.byref(st), P, 1, P, P, 8, float("nan"), P, P, 1 << 20, None) == qn.QN_EINVAL
    assert L.qlora_linear_fwd(ctypes.byref(st), P, 1, P, P, 8, 16.0, P, P, 4, None) == qn.QN_ENOMEM
    assert L.qlora_linear_bwd_dx(ctypes.byref(st), P, 1, P, P, 8, 16.0, P, None, 1 << 20, None) == qn.QN_EINVAL
    msg = _err(qn, L.qlora_linear_bwd_dx(ctypes.byref(st), P, 1, P, P, 8, 16.0, P, P, 4, None))[1]
    assert "workspace" in msg
    # LoftQ: rank + oversample bound, T bound, shape agreement
    res = (ctypes.c_double * 8)()
    assert L.loftq_init(P, 128, 128, 90, 16.0, 5, 0, 8, 4, ctypes.byref(st), P, P, ctypes.addressof(res), P,
                        1 << 30, None) == qn.QN_ESHAPE      # r + oversample = 98 > 96
    assert L.loftq_init(P, 128, 128, 8, 16.0, 99, 0, 8, 4, ctypes.byref(st), P, P, ctypes.addressof(res), P,
                        1 << 30, None) == qn.QN_ESHAPE
    assert L.loftq_init(P, 64, 128, 8, 16.0, 5, 0, 8, 4, ctypes.byref(st), P, P, ctypes.addressof(res), P,
                        1 << 30, None) == qn.QN_ESHAPE


def test_noalloc_quantize_argument_errors(qn):
    L = qn.lib
    P = 0x10000
    assert L.nf4_quantize_noalloc(P, 0, None, None) == qn.QN_EINVAL
    st = _struct(qn)
    assert L.nf4_quantize_noalloc(P, 9, ctypes.byref(st), None) == qn.QN_EINVAL
    assert L.nf4_quantize_noalloc(P + 8, 0, ctypes.byref(st), None) == qn.QN_EALIGN
    # 2^41 elements: QN_ESHAPE comes from the shape check every entry point
    # shares (d*k <= 2^40), which also bounds what the static scratch covers
    huge = _struct(qn, d=1 << 21, k=1 << 20)
    assert L.nf4_quantize_noalloc(P, 0, ctypes.byref(huge), None) == qn.QN_ESHAPE
    assert "too large" in qn.lib.qn_last_error().decode()


def test_new_entry_points_reject_bad_arguments(qn):
    L = qn.lib
    P = 0x10000
    st = _struct(qn)
    res = (ctypes.c_double * 2)()
    # adapter gradients: rank bound, NULL, alignment, workspace
    assert L.qlora_linear_bwd_lora(P, P, 4, 64, 64, P, P, 0, 16.0, P, P, P, 1 << 30, None) == qn.QN_ESHAPE
    assert L.qlora_linear_bwd_lora(P, None, 4, 64, 64, P, P, 8, 16.0, P, P, P, 1 << 30, None) == qn.QN_EINVAL
    assert L.qlora_linear_bwd_lora(P + 4, P, 4, 64, 64, P, P, 8, 16.0, P, P, P, 1 << 30, None) == qn.QN_EALIGN
    assert L.qlora_linear_bwd_lora(P, P, 4, 64, 64, P, P, 8, 16.0, P, P, P, 16, None) == qn.QN_ENOMEM
    # fp32 layer: k % 64, r range, workspace
    odd_k = _struct(qn, k=100)
    assert L.qlora_linear_fwd_f32(ctypes.byref(odd_k), P, 1, P, P, 8, 16.0, P, P, 1 << 20, None) == qn.QN_ESHAPE
    assert L.qlora_linear_bwd_dx_f32(ctypes.byref(st), P, 1, P, P, 300, 16.0, P, P, 1 << 20, None) == qn.QN_ESHAPE
    assert L.qlora_linear_fwd_f32(ctypes.byref(st), P, 1, P, P, 8, 16.0, P, P, 4, None) == qn.QN_ENOMEM
    # merge: sign, rank, shape agreement
    assert L.nf4_merge_lora(ctypes.byref(st), P, P, 8, 16.0, 0, ctypes.byref(st), P, 1 << 20, None) == qn.QN_EINVAL
    assert L.nf4_merge_lora(ctypes.byref(st), P, P, 0, 16.0, 1, ctypes.byref(st), P, 1 << 20, None) == qn.QN_ESHAPE
    other = _struct(qn, d=st.d * 2)
    assert L.nf4_merge_lora(ctypes.byref(st), P, P, 8, 16.0, 1, ctypes.byref(other), P, 1 << 20, None) == qn.QN_ESHAPE
    # one-step LoftQ: rank + oversample bound
    assert L.loftq_replace_lora(P, ctypes.byref(st), 90, 16.0, 0, 8, 4, P, P, ctypes.addressof(res), P, 1 << 30,
                                None) == qn.QN_ESHAPE      # r + oversample = 98 > 96
    # workspace queries of the new operations
    assert qn.workspace_bytes(qn.QN_OP_LINEAR_BWD_LORA, 4096, 11008, 4096, 16) > 256 * 1024
    assert qn.workspace_bytes(qn.QN_OP_LINEAR_F32, 16, 1024, 1024, 8) >= 256 * 1024 + 16 * 8 * 4
    assert qn.workspace_bytes(qn.QN_OP_MERGE, 0, 1024, 1024, 8) == qn.workspace_bytes(qn.QN_OP_QUANTIZE, 0, 1024, 1024, 0)
