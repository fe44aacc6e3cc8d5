"""Python binding of libqlora_nf4 (the B300 QLoRA NF4 hot path).

Argument marshalling only: every step of the path runs in the CUDA kernels of
``libqlora_nf4.so`` (built by :func:`bit_nf4_quantized_39_b300.build.build`).
PyTorch provides device memory, streams and the host<->device copies of the
host-buffer entry points; it computes nothing of the method.

The functions carry the names of the C ABI (``include/qlora_nf4.h``):

* :func:`nf4_quantize`        W (d x k, fp32/bf16, CUDA) -> :class:`NF4Tensor`
* :func:`nf4_dequantize`      NF4Tensor -> fp32 / bf16 weights
* :func:`qlora_linear_fwd`    Y  = X deq(Q)^T + (alpha/r) (X A^T) B^T
* :func:`qlora_linear_bwd_dx` dX = dY deq(Q) + (alpha/r) (dY B) A
* :func:`qlora_linear_bwd_lora`  dA = s (dY B)^T X, dB = s dY^T (X A^T)
* :func:`qlora_linear_fwd_f32` / :func:`qlora_linear_bwd_dx_f32`  fp32 compute dtype
* :func:`loftq_init`          LoftQ alternation -> (Q, A, B, residuals)
* :func:`loftq_replace_lora`  one LoftQ step against a given Q -> (A, B, residuals)
* :func:`nf4_merge_lora`      NF4(deq(Q) +- s B A) (merge / unmerge)

If the shared library is missing, importing this package raises ImportError:
there is no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqlora_nf4.so")

QN_OK, QN_EINVAL, QN_ESHAPE, QN_EALIGN, QN_ENOMEM, QN_ECUDA, QN_ETIMEOUT, QN_EUNSUPPORTED = range(8)
QN_F32, QN_BF16 = 0, 1
(QN_OP_QUANTIZE, QN_OP_DEQUANTIZE, QN_OP_LINEAR_FWD, QN_OP_LINEAR_BWD_DX, QN_OP_LOFTQ, QN_OP_LINEAR_BWD_LORA,
 QN_OP_LINEAR_F32, QN_OP_MERGE) = range(8)

_STATUS_NAMES = {0: "QN_OK", 1: "QN_EINVAL", 2: "QN_ESHAPE", 3: "QN_EALIGN", 4: "QN_ENOMEM",
                 5: "QN_ECUDA", 6: "QN_ETIMEOUT", 7: "QN_EUNSUPPORTED"}


class QnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class qn_nf4(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int64), ("k", ctypes.c_int64), ("block", ctypes.c_int32),
                ("dq", ctypes.c_int32), ("dq_block", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("codes", ctypes.c_void_p), ("absmax", ctypes.c_void_p), ("absmax_q", ctypes.c_void_p),
                ("absmax_scale", ctypes.c_void_p), ("absmax_mean", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "qn_abi_version": (ctypes.c_int, []),
        "qn_last_error": (ctypes.c_char_p, []),
        "qn_nf4_tables": (None, [vp, vp]),
        "qn_workspace_bytes": (sz, [ctypes.c_int, i64, i64, i64, i32]),
        "nf4_quantize": (ctypes.c_int, [vp, ctypes.c_int, P(qn_nf4), vp, sz, vp]),
        "nf4_dequantize": (ctypes.c_int, [P(qn_nf4), vp, ctypes.c_int, vp]),
        "qlora_linear_fwd": (ctypes.c_int, [P(qn_nf4), vp, i64, vp, vp, i32, f32, vp, vp, sz, vp]),
        "qlora_linear_bwd_dx": (ctypes.c_int, [P(qn_nf4), vp, i64, vp, vp, i32, f32, vp, vp, sz, vp]),
        "loftq_init": (ctypes.c_int, [vp, i64, i64, i32, f32, i32, ctypes.c_uint64, i32, i32,
                                      P(qn_nf4), vp, vp, vp, vp, sz, vp]),
        "qn_device_status": (ctypes.c_int, [vp]),
        "nf4_quantize_noalloc": (ctypes.c_int, [vp, ctypes.c_int, P(qn_nf4), vp]),
        "qlora_linear_fwd_group": (ctypes.c_int, [i32, P(P(qn_nf4)), vp, i64, P(vp), P(vp), P(i32), P(f32), P(vp),
                                                  vp, sz, vp]),
        "qlora_linear_bwd_lora": (ctypes.c_int, [vp, vp, i64, i64, i64, vp, vp, i32, f32, vp, vp, vp, sz, vp]),
        "qlora_linear_fwd_f32": (ctypes.c_int, [P(qn_nf4), vp, i64, vp, vp, i32, f32, vp, vp, sz, vp]),
        "qlora_linear_bwd_dx_f32": (ctypes.c_int, [P(qn_nf4), vp, i64, vp, vp, i32, f32, vp, vp, sz, vp]),
        "loftq_replace_lora": (ctypes.c_int, [vp, P(qn_nf4), i32, f32, ctypes.c_uint64, i32, i32, vp, vp, vp,
                                              vp, sz, vp]),
        "nf4_merge_lora": (ctypes.c_int, [P(qn_nf4), vp, vp, i32, f32, i32, P(qn_nf4), vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()
EXPORTS = ("qn_abi_version", "qn_last_error", "qn_nf4_tables", "qn_workspace_bytes", "nf4_quantize",
           "nf4_dequantize", "qlora_linear_fwd", "qlora_linear_bwd_dx", "loftq_init", "qn_device_status",
           "nf4_quantize_noalloc", "qlora_linear_fwd_group", "qlora_linear_bwd_lora", "qlora_linear_fwd_f32",
           "qlora_linear_bwd_dx_f32", "loftq_replace_lora", "nf4_merge_lora")


def _check(status: int):
    if status != QN_OK:
        raise QnError(status, lib.qn_last_error().decode())


def _stream_ptr(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _dev_bf16(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bf16 (got {t.dtype})")
    return t.contiguous()


_WS: dict = {}


_ZERO_AREA = 256 * 1024  # leading bytes of every workspace that must start at zero


def _workspace(nbytes: int, device) -> torch.Tensor | None:
    """A cached device workspace of at least ``nbytes`` bytes (256-byte aligned)."""
    if nbytes == 0:
        return None
    key = (str(device), torch.cuda.current_stream(device).cuda_stream)
    ws = _WS.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(nbytes + 512, dtype=torch.uint8, device=device)
        ws[:min(ws.numel(), _ZERO_AREA + 512)].zero_()  # the semaphore area starts at zero
        _WS[key] = ws
    return ws


def _ws_ptr(ws):
    if ws is None:
        return None, 0
    p = ws.data_ptr()
    off = (-p) % 256
    return p + off, ws.numel() - off


def tables():
    """(codebook[16], thresholds[15]) as the library's kernels use them."""
    cb = (ctypes.c_float * 16)()
    th = (ctypes.c_float * 15)()
    lib.qn_nf4_tables(ctypes.addressof(cb), ctypes.addressof(th))
    return list(cb), list(th)


def workspace_bytes(op: int, M: int, d: int, k: int, r: int) -> int:
    return int(lib.qn_workspace_bytes(op, M, d, k, r))


@dataclass
class NF4Tensor:
    """Quantised state of a d x k weight (all tensors on one CUDA device)."""
    d: int
    k: int
    codes: torch.Tensor            # uint8[ceil(n/2)]
    absmax: torch.Tensor           # fp32[nblk]
    dq: bool
    absmax_q: torch.Tensor | None = None      # int8[nblk]
    absmax_scale: torch.Tensor | None = None  # fp32[ngrp]
    absmax_mean: torch.Tensor | None = None   # fp32[1]
    block: int = 64
    dq_block: int = 256

    @staticmethod
    def empty(d: int, k: int, dq: bool = True, device="cuda") -> "NF4Tensor":
        n = d * k
        nblk = -(-n // 64)
        ngrp = -(-nblk // 256)
        mk = lambda cnt, dt: torch.empty(max(cnt, 1), dtype=dt, device=device)
        return NF4Tensor(d=d, k=k, codes=mk(-(-n // 2), torch.uint8), absmax=mk(nblk, torch.float32), dq=dq,
                         absmax_q=mk(nblk, torch.int8) if dq else None,
                         absmax_scale=mk(ngrp, torch.float32) if dq else None,
                         absmax_mean=mk(1, torch.float32) if dq else None)

    def c_struct(self) -> qn_nf4:
        return qn_nf4(self.d, self.k, self.block, 1 if self.dq else 0, self.dq_block, 0,
                      _ptr(self.codes), _ptr(self.absmax), _ptr(self.absmax_q), _ptr(self.absmax_scale),
                      _ptr(self.absmax_mean))

    @property
    def device(self):
        return self.codes.device

    def nbytes(self) -> int:
        """Bytes of the quantised state the dequantiser reads."""
        n = self.d * self.k
        b = -(-n // 2)
        nblk = -(-n // 64)
        if self.dq:
            return b + nblk + 4 * (-(-nblk // 256)) + 4
        return b + 4 * nblk


def nf4_quantize(W: torch.Tensor, dq: bool = True, out: NF4Tensor | None = None, stream=None) -> NF4Tensor:
    """Blockwise NF4 quantisation of a CUDA fp32/bf16 tensor viewed as d x k."""
    if not W.is_cuda:
        raise ValueError("W must be a CUDA tensor")
    if W.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("W must be fp32 or bf16")
    W = W.contiguous()
    d, k = (W.shape[0], W.numel() // W.shape[0]) if W.dim() >= 2 else (1, W.numel())
    q = out if out is not None else NF4Tensor.empty(d, k, dq, W.device)
    st = q.c_struct()
    ws = _workspace(workspace_bytes(QN_OP_QUANTIZE, 0, d, k, 0), W.device)
    wp, wn = _ws_ptr(ws)
    _check(lib.nf4_quantize(W.data_ptr(), QN_F32 if W.dtype == torch.float32 else QN_BF16,
                            ctypes.byref(st), wp, wn, _stream_ptr(stream)))
    return q


def nf4_dequantize(q: NF4Tensor, dtype=torch.float32, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("dtype must be fp32 or bf16")
    o = out if out is not None else torch.empty((q.d, q.k), dtype=dtype, device=q.device)
    st = q.c_struct()
    _check(lib.nf4_dequantize(ctypes.byref(st), o.data_ptr(), QN_F32 if dtype == torch.float32 else QN_BF16,
                              _stream_ptr(stream)))
    return o


def qlora_linear_fwd(q: NF4Tensor, X: torch.Tensor, A: torch.Tensor, B: torch.Tensor, alpha: float,
                     out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = X deq(Q)^T + (alpha/r) (X A^T) B^T.  X may live on the host: then it
    is copied to the device, and Y copied back, around the kernel call."""
    host = not X.is_cuda
    if host:
        Xd = X.to(q.device, non_blocking=True)
    else:
        Xd = X
    Xd = _dev_bf16(Xd, "X").reshape(-1, q.k)
    A = _dev_bf16(A, "A")
    B = _dev_bf16(B, "B")
    r = A.shape[0]
    M = Xd.shape[0]
    Y = out if (out is not None and not host) else torch.empty((M, q.d), dtype=torch.bfloat16, device=q.device)
    ws = _workspace(workspace_bytes(QN_OP_LINEAR_FWD, M, q.d, q.k, r), q.device)
    wp, wn = _ws_ptr(ws)
    st = q.c_struct()
    _check(lib.qlora_linear_fwd(ctypes.byref(st), Xd.data_ptr(), M, A.data_ptr(), B.data_ptr(), r, float(alpha),
                                Y.data_ptr(), wp, wn, _stream_ptr(stream)))
    if host:
        Yh = out if out is not None else torch.empty((M, q.d), dtype=torch.bfloat16, pin_memory=True)
        Yh.copy_(Y, non_blocking=True)
        return Yh
    return Y


def qlora_linear_fwd_group(qs, X: torch.Tensor, As, Bs, alphas, outs=None, stream=None):
    """Several projections of one input: Y[g] = X deq(Q[g])^T + (alpha[g]/r[g]) (X A[g]^T) B[g]^T."""
    n = len(qs)
    k = qs[0].k
    Xd = _dev_bf16(X, "X").reshape(-1, k)
    M = Xd.shape[0]
    As = [_dev_bf16(a, "A") for a in As]
    Bs = [_dev_bf16(b, "B") for b in Bs]
    rs = [a.shape[0] for a in As]
    Ys = list(outs) if outs is not None else [torch.empty((M, q.d), dtype=torch.bfloat16, device=q.device) for q in qs]
    structs = [q.c_struct() for q in qs]
    QP = (ctypes.POINTER(qn_nf4) * n)(*[ctypes.pointer(st) for st in structs])
    AP = (ctypes.c_void_p * n)(*[a.data_ptr() for a in As])
    BP = (ctypes.c_void_p * n)(*[b.data_ptr() for b in Bs])
    YP = (ctypes.c_void_p * n)(*[y.data_ptr() for y in Ys])
    RP = (ctypes.c_int32 * n)(*rs)
    FP = (ctypes.c_float * n)(*[float(a) for a in alphas])
    ws = _workspace(workspace_bytes(QN_OP_LINEAR_FWD, M, sum(q.d for q in qs), k, sum(rs)), qs[0].device)
    wp, wn = _ws_ptr(ws)
    _check(lib.qlora_linear_fwd_group(n, QP, Xd.data_ptr(), M, AP, BP, RP, FP, YP, wp, wn, _stream_ptr(stream)))
    return Ys


def qlora_linear_bwd_dx(q: NF4Tensor, dY: torch.Tensor, A: torch.Tensor, B: torch.Tensor, alpha: float,
                        out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dX = dY deq(Q) + (alpha/r) (dY B) A."""
    dY = _dev_bf16(dY, "dY").reshape(-1, q.d)
    A = _dev_bf16(A, "A")
    B = _dev_bf16(B, "B")
    r = A.shape[0]
    M = dY.shape[0]
    dX = out if out is not None else torch.empty((M, q.k), dtype=torch.bfloat16, device=q.device)
    ws = _workspace(workspace_bytes(QN_OP_LINEAR_BWD_DX, M, q.d, q.k, r), q.device)
    wp, wn = _ws_ptr(ws)
    st = q.c_struct()
    _check(lib.qlora_linear_bwd_dx(ctypes.byref(st), dY.data_ptr(), M, A.data_ptr(), B.data_ptr(), r, float(alpha),
                                   dX.data_ptr(), wp, wn, _stream_ptr(stream)))
    return dX


def loftq_init(W: torch.Tensor, r: int, alpha: float, T: int = 5, seed: int = 0, oversample: int = 8,
               power_iters: int = 4, dq: bool = True, stream=None):
    """LoftQ initialisation of a CUDA fp32 matrix: returns (Q, A fp32 r x k, B fp32 d x r, resid list)."""
    if not W.is_cuda or W.dtype != torch.float32 or W.dim() != 2:
        raise ValueError("W must be a 2-D CUDA fp32 tensor")
    W = W.contiguous()
    d, k = W.shape
    q = NF4Tensor.empty(d, k, dq, W.device)
    A = torch.empty((r, k), dtype=torch.float32, device=W.device)
    B = torch.empty((d, r), dtype=torch.float32, device=W.device)
    resid = (ctypes.c_double * (T + 1))()
    ws = _workspace(workspace_bytes(QN_OP_LOFTQ, 0, d, k, r), W.device)
    wp, wn = _ws_ptr(ws)
    st = q.c_struct()
    _check(lib.loftq_init(W.data_ptr(), d, k, r, float(alpha), T, seed, oversample, power_iters,
                          ctypes.byref(st), A.data_ptr(), B.data_ptr(), ctypes.addressof(resid), wp, wn,
                          _stream_ptr(stream)))
    return q, A, B, list(resid)


def qlora_linear_bwd_lora(X: torch.Tensor, dY: torch.Tensor, A: torch.Tensor, B: torch.Tensor, alpha: float,
                          stream=None):
    """(dA fp32 r x k, dB fp32 d x r): gradients of the adapter factors for dL/dY = dY."""
    A = _dev_bf16(A, "A")
    B = _dev_bf16(B, "B")
    r, k = A.shape
    d = B.shape[0]
    X = _dev_bf16(X, "X").reshape(-1, k)
    dY = _dev_bf16(dY, "dY").reshape(-1, d)
    M = X.shape[0]
    if dY.shape[0] != M:
        raise ValueError("X and dY must have the same number of rows")
    dA = torch.empty((r, k), dtype=torch.float32, device=X.device)
    dB = torch.empty((d, r), dtype=torch.float32, device=X.device)
    ws = _workspace(workspace_bytes(QN_OP_LINEAR_BWD_LORA, M, d, k, r), X.device)
    wp, wn = _ws_ptr(ws)
    _check(lib.qlora_linear_bwd_lora(X.data_ptr(), dY.data_ptr(), M, d, k, A.data_ptr(), B.data_ptr(), r,
                                     float(alpha), dA.data_ptr(), dB.data_ptr(), wp, wn, _stream_ptr(stream)))
    return dA, dB


def _dev_f32(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.float32:
        raise ValueError(f"{name} must be fp32 (got {t.dtype})")
    return t.contiguous()


def qlora_linear_fwd_f32(q: NF4Tensor, X: torch.Tensor, A: torch.Tensor, B: torch.Tensor, alpha: float,
                         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = X deq(Q)^T + (alpha/r) (X A^T) B^T with fp32 X, A, B, Y (fp32 compute dtype)."""
    X = _dev_f32(X, "X").reshape(-1, q.k)
    A = _dev_f32(A, "A")
    B = _dev_f32(B, "B")
    r, M = A.shape[0], X.shape[0]
    Y = out if out is not None else torch.empty((M, q.d), dtype=torch.float32, device=q.device)
    ws = _workspace(workspace_bytes(QN_OP_LINEAR_F32, M, q.d, q.k, r), q.device)
    wp, wn = _ws_ptr(ws)
    st = q.c_struct()
    _check(lib.qlora_linear_fwd_f32(ctypes.byref(st), X.data_ptr(), M, A.data_ptr(), B.data_ptr(), r, float(alpha),
                                    Y.data_ptr(), wp, wn, _stream_ptr(stream)))
    return Y


def qlora_linear_bwd_dx_f32(q: NF4Tensor, dY: torch.Tensor, A: torch.Tensor, B: torch.Tensor, alpha: float,
                            out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dX = dY deq(Q) + (alpha/r) (dY B) A with fp32 operands (fp32 compute dtype)."""
    dY = _dev_f32(dY, "dY").reshape(-1, q.d)
    A = _dev_f32(A, "A")
    B = _dev_f32(B, "B")
    r, M = A.shape[0], dY.shape[0]
    dX = out if out is not None else torch.empty((M, q.k), dtype=torch.float32, device=q.device)
    ws = _workspace(workspace_bytes(QN_OP_LINEAR_F32, M, q.d, q.k, r), q.device)
    wp, wn = _ws_ptr(ws)
    st = q.c_struct()
    _check(lib.qlora_linear_bwd_dx_f32(ctypes.byref(st), dY.data_ptr(), M, A.data_ptr(), B.data_ptr(), r,
                                       float(alpha), dX.data_ptr(), wp, wn, _stream_ptr(stream)))
    return dX


def loftq_replace_lora(W: torch.Tensor, q: NF4Tensor, r: int, alpha: float, seed: int = 0, oversample: int = 8,
                       power_iters: int = 4, stream=None):
    """One LoftQ step against the given quantised weight q (kept as it is):
    returns (A fp32 r x k, B fp32 d x r, [||W - deq(q)||_F, ||W - deq(q) - s B A||_F])."""
    W = _dev_f32(W, "W")
    if W.dim() != 2 or W.shape != (q.d, q.k):
        raise ValueError("W must be a d x k fp32 CUDA tensor matching q")
    A = torch.empty((r, q.k), dtype=torch.float32, device=W.device)
    B = torch.empty((q.d, r), dtype=torch.float32, device=W.device)
    resid = (ctypes.c_double * 2)()
    ws = _workspace(workspace_bytes(QN_OP_LOFTQ, 0, q.d, q.k, r), W.device)
    wp, wn = _ws_ptr(ws)
    st = q.c_struct()
    _check(lib.loftq_replace_lora(W.data_ptr(), ctypes.byref(st), r, float(alpha), seed, oversample, power_iters,
                                  A.data_ptr(), B.data_ptr(), ctypes.addressof(resid), wp, wn, _stream_ptr(stream)))
    return A, B, list(resid)


def nf4_merge_lora(q: NF4Tensor, A: torch.Tensor, B: torch.Tensor, alpha: float, sign: int = 1,
                   out: NF4Tensor | None = None, stream=None) -> NF4Tensor:
    """NF4(deq(q) + sign (alpha/r) B A): sign +1 merges the adapter, -1 unmerges it.
    ``out=q`` merges in place."""
    A = _dev_bf16(A, "A")
    B = _dev_bf16(B, "B")
    r = A.shape[0]
    o = out if out is not None else NF4Tensor.empty(q.d, q.k, q.dq, q.device)
    ws = _workspace(workspace_bytes(QN_OP_MERGE, 0, q.d, q.k, r), q.device)
    wp, wn = _ws_ptr(ws)
    si, so = q.c_struct(), o.c_struct()
    _check(lib.nf4_merge_lora(ctypes.byref(si), A.data_ptr(), B.data_ptr(), r, float(alpha), int(sign),
                              ctypes.byref(so), wp, wn, _stream_ptr(stream)))
    return o


def device_status(stream=None) -> None:
    """Synchronise and raise QnError(QN_ETIMEOUT) if a bounded device wait expired."""
    _check(lib.qn_device_status(_stream_ptr(stream)))
