"""Python binding of the flamia C ABI (include/flamia.h).

Argument marshalling only: torch tensors supply device pointers and the
current CUDA stream; every step of the attention path runs in the library's
own CUDA kernels.  There is no fallback: if the library is missing or a call
returns an error status, a RuntimeError is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libflamia.so")

FLAMIA_OK = 0
FORMAT_MXFP8 = 0
FORMAT_MXFP8_NVFP4 = 1
FORMAT_HADAMARD = 0x10
FORMAT_TOKEN_SCALES = 0x20
FLAG_NVFP4_QK = 0x1
FLAG_HADAMARD = 0x2
FLAG_NONCAUSAL = 0x4
FLAG_DETERMINISTIC_DQ = 0x8
FLAG_DQ_FP16 = 0x10
FLAG_DQ_CAUSAL_SCALE = 0x20
FLAG_SCHEDULE_STATIC = 0x40
FLAG_SCHEDULE_RULE = 0x80
FLAG_DS_ROW_EXPONENTS = 0x100
FLAG_TOKEN_SCALES = 0x200
FLAG_DS_ZERO_COUNT = 0x400
FLAG_BWD_CTA_PAIR = 0x800
FLAG_BWD_ONE_CTA = 0x1000
DEV_BAD_SEQLENS = 0x1
DEV_CAPACITY = 0x2
DEV_TIMEOUT = 0x4
DEV_RANGE = 0x8

_LIB = None


class QTensorStruct(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("nvfp4_codes", ctypes.c_void_p), ("nvfp4_scales", ctypes.c_void_p)]


_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_QP = ctypes.POINTER(QTensorStruct)
SIGNATURES = {
    "flamia_quantize_tokenblock": (_i, [_vp, _i, _i, _i, _vp, _i, _i, _vp, _vp, _QP, _vp, _vp]),
    "flamia_quantize_qkv": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _i, _i, _QP, _QP, _QP, _vp,
                                 _vp]),
    "flamia_worklist_bytes": (_sz, [_i, _i]),
    "flamia_build_worklist": (_i, [_vp, _i, _i, _vp, _sz, _vp, _vp]),
    "flamia_attn_fwd": (_i, [_QP, _QP, _QP, _vp, _i, _i, _i, _i, _f, _i, _vp, _vp, _vp, _vp, _vp]),
    "flamia_attn_fwd_gqa": (_i, [_QP, _QP, _QP, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _vp, _vp,
                                 _vp, _vp]),
    "flamia_fwd_workspace_bytes": (_sz, [_i, _i, _i]),
    "flamia_bwd_ds_counts_offset": (_sz, [_i, _i, _i]),
    "flamia_bwd_workspace_bytes": (_sz, [_i, _i, _i]),
    "flamia_attn_bwd": (_i, [_QP, _QP, _QP, _QP, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp,
                             _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "flamia_attn_bwd_gqa": (_i, [_QP, _QP, _QP, _QP, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i,
                                 _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "flamia_build_worklist_static": (_i, [_vp, _i, _i, _vp, _sz, _vp, _vp]),
    "flamia_status_str": (ctypes.c_char_p, [_i]),
    "flamia_debug_mma_tile": (_i, [_i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "flamia_debug_bounded_waits": (_i, [_vp, _vp, _vp]),
    "flamia_debug_launch_count": (ctypes.c_ulonglong, []),
    "flamia_debug_tmem_ldred": (_i, [_vp, _vp, _vp, _vp]),
    "flamia_debug_pair_mma": (_i, [_i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
}


def load(path: str = LIB_PATH):
    """Loads the built library (raises if it was not built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(path):
            raise RuntimeError(f"flamia CUDA library not built ({path}); "
                               "run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _check(status: int, what: str):
    if status != FLAMIA_OK:
        msg = load().flamia_status_str(status).decode()
        raise RuntimeError(f"{what} failed: {msg} ({status})")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise RuntimeError("flamia needs CUDA tensors")
    if not t.is_contiguous():
        raise RuntimeError("flamia needs contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


class QTensor:
    """Caller-owned buffers of one quantised operand (allocated by torch)."""

    def __init__(self, T: int, H: int, d: int, nvfp4: bool = False, device="cuda"):
        self.codes = torch.empty((T, H, d), dtype=torch.uint8, device=device)
        self.scales = torch.empty((H, T), dtype=torch.uint8, device=device)
        self.nvfp4_codes = torch.empty((T, H, d // 2), dtype=torch.uint8, device=device) if nvfp4 else None
        self.nvfp4_scales = torch.empty((T, H, d // 16), dtype=torch.uint8, device=device) if nvfp4 else None

    def struct(self) -> QTensorStruct:
        s = QTensorStruct()
        s.codes = self.codes.data_ptr()
        s.scales = self.scales.data_ptr()
        s.nvfp4_codes = self.nvfp4_codes.data_ptr() if self.nvfp4_codes is not None else None
        s.nvfp4_scales = self.nvfp4_scales.data_ptr() if self.nvfp4_scales is not None else None
        return s


def flamia_quantize_tokenblock(x, cu_seqlens, out: QTensor, fmt: int = FORMAT_MXFP8, o=None,
                               D=None, dev_status=None):
    T, H, d = x.shape
    st = out.struct()
    _check(load().flamia_quantize_tokenblock(
        _ptr(x), T, H, d, _ptr(cu_seqlens), cu_seqlens.numel() - 1, fmt, _ptr(o), _ptr(D),
        ctypes.byref(st), _ptr(dev_status), _stream()), "flamia_quantize_tokenblock")


def flamia_quantize_qkv(xq, xk, xv, cu_seqlens, q: QTensor, k: QTensor, v: QTensor,
                        fmt_qk: int = FORMAT_MXFP8, dev_status=None):
    T, H, d = xq.shape
    sq, sk, sv = q.struct(), k.struct(), v.struct()
    _check(load().flamia_quantize_qkv(
        _ptr(xq), _ptr(xk), _ptr(xv), T, H, xk.shape[1], d, _ptr(cu_seqlens),
        cu_seqlens.numel() - 1, fmt_qk, ctypes.byref(sq), ctypes.byref(sk), ctypes.byref(sv),
        _ptr(dev_status), _stream()), "flamia_quantize_qkv")


def flamia_worklist_bytes(T: int, ndocs: int) -> int:
    return int(load().flamia_worklist_bytes(T, ndocs))


def flamia_build_worklist(cu_seqlens, T: int, wl, dev_status=None):
    _check(load().flamia_build_worklist(_ptr(cu_seqlens), cu_seqlens.numel() - 1, T, _ptr(wl),
                                        wl.numel() * wl.element_size(), _ptr(dev_status),
                                        _stream()), "flamia_build_worklist")


def flamia_build_worklist_static(cu_seqlens, T: int, wl, dev_status=None):
    """Work list with the builder's scratch in the library's static device
    array (no allocation); same output as flamia_build_worklist."""
    _check(load().flamia_build_worklist_static(_ptr(cu_seqlens), cu_seqlens.numel() - 1, T,
                                               _ptr(wl), wl.numel() * wl.element_size(),
                                               _ptr(dev_status), _stream()),
           "flamia_build_worklist_static")


def flamia_attn_fwd(q: QTensor, k: QTensor, v: QTensor, cu_seqlens, T, H, d, softmax_scale,
                    wl, o, lse, flags: int = 0, dev_status=None):
    sq, sk, sv = q.struct(), k.struct(), v.struct()
    _check(load().flamia_attn_fwd(ctypes.byref(sq), ctypes.byref(sk), ctypes.byref(sv),
                                  _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, H, d,
                                  float(softmax_scale), flags, _ptr(wl), _ptr(o), _ptr(lse),
                                  _ptr(dev_status), _stream()), "flamia_attn_fwd")


def flamia_attn_fwd_gqa(q: QTensor, k: QTensor, v: QTensor, cu_seqlens, T, H, H_kv, d,
                        softmax_scale, wl, o, lse, flags: int = 0, dev_status=None):
    sq, sk, sv = q.struct(), k.struct(), v.struct()
    _check(load().flamia_attn_fwd_gqa(ctypes.byref(sq), ctypes.byref(sk), ctypes.byref(sv),
                                      _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, H, H_kv, d,
                                      float(softmax_scale), flags, _ptr(wl), _ptr(o), _ptr(lse),
                                      _ptr(dev_status), _stream()), "flamia_attn_fwd_gqa")


def flamia_bwd_ds_counts_offset(T: int, H: int, d: int) -> int:
    return int(load().flamia_bwd_ds_counts_offset(T, H, d))


def flamia_fwd_workspace_bytes(T: int, H: int, d: int) -> int:
    return int(load().flamia_fwd_workspace_bytes(T, H, d))


def flamia_bwd_workspace_bytes(T: int, H: int, d: int) -> int:
    return int(load().flamia_bwd_workspace_bytes(T, H, d))


def flamia_attn_bwd(q: QTensor, k: QTensor, v: QTensor, dout: QTensor, D, lse, cu_seqlens, T, H,
                    d, softmax_scale, wl, dq, dk, dv, ws, flags: int = 0, dev_status=None):
    sq, sk, sv, sd = q.struct(), k.struct(), v.struct(), dout.struct()
    _check(load().flamia_attn_bwd(ctypes.byref(sq), ctypes.byref(sk), ctypes.byref(sv),
                                  ctypes.byref(sd), _ptr(D), _ptr(lse), _ptr(cu_seqlens),
                                  cu_seqlens.numel() - 1, T, H, d, float(softmax_scale), flags,
                                  _ptr(wl), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                                  ws.numel() * ws.element_size(), _ptr(dev_status), _stream()),
           "flamia_attn_bwd")


def flamia_attn_bwd_gqa(q: QTensor, k: QTensor, v: QTensor, dout: QTensor, D, lse, cu_seqlens,
                        T, H, H_kv, d, softmax_scale, wl, dq, dk, dv, ws, flags: int = 0,
                        dev_status=None):
    sq, sk, sv, sd = q.struct(), k.struct(), v.struct(), dout.struct()
    _check(load().flamia_attn_bwd_gqa(ctypes.byref(sq), ctypes.byref(sk), ctypes.byref(sv),
                                      ctypes.byref(sd), _ptr(D), _ptr(lse), _ptr(cu_seqlens),
                                      cu_seqlens.numel() - 1, T, H, H_kv, d, float(softmax_scale),
                                      flags, _ptr(wl), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                                      ws.numel() * ws.element_size(), _ptr(dev_status),
                                      _stream()), "flamia_attn_bwd_gqa")


def flamia_debug_tmem_ldred(x, vals, mx):
    _check(load().flamia_debug_tmem_ldred(_ptr(x), _ptr(vals), _ptr(mx), _stream()),
           "flamia_debug_tmem_ldred")


def flamia_debug_pair_mma(shape, variant, a, b, sfa, sfb, d_out, tmem_cols, dev_status):
    _check(load().flamia_debug_pair_mma(shape, variant, _ptr(a), _ptr(b), _ptr(sfa), _ptr(sfb),
                                        _ptr(d_out), _ptr(tmem_cols), _ptr(dev_status),
                                        _stream()),
           "flamia_debug_pair_mma")


def flamia_debug_launch_count() -> int:
    """Kernel launches the library has enqueued since it was loaded."""
    return int(load().flamia_debug_launch_count())


def flamia_debug_bounded_waits(turn, dev_status):
    _check(load().flamia_debug_bounded_waits(_ptr(turn), _ptr(dev_status), _stream()),
           "flamia_debug_bounded_waits")


def flamia_debug_mma_tile(mode, N, a_mn, b_mn, variant, a, b, sfa, sfb, d_out, dev_status=None):
    _check(load().flamia_debug_mma_tile(mode, N, a_mn, b_mn, variant, _ptr(a), _ptr(b), _ptr(sfa),
                                        _ptr(sfb), _ptr(d_out), _ptr(dev_status), _stream()),
           "flamia_debug_mma_tile")


class TrainingCall:
    """Buffers and the sequence of C-ABI calls of one attention training call
    (quantise Q, K, V -> work list -> forward -> quantise dO with D -> backward)
    for fixed shapes.  All buffers are torch allocations owned by this object."""

    def __init__(self, T, H, d, cu_seqlens, softmax_scale, nvfp4_qk: bool = False,
                 hadamard: bool = False, causal: bool = True, H_kv=None,
                 deterministic_dq: bool = False, dq_accum: str = "fp32", schedule: str = "dynamic",
                 ds_rows: bool = False, token_scales: bool = False,
                 ds_zero_count: bool = False, bwd_ctas: str = "rule", device="cuda"):
        self.T, self.H, self.d = T, H, d
        self.H_kv = H if H_kv is None else H_kv
        self.scale = softmax_scale
        self.cu = cu_seqlens
        self.flags = ((FLAG_NVFP4_QK if nvfp4_qk else 0) | (FLAG_HADAMARD if hadamard else 0) |
                      (0 if causal else FLAG_NONCAUSAL) |
                      (FLAG_DETERMINISTIC_DQ if deterministic_dq else 0) |
                      {"fp32": 0, "fp16_sequence": FLAG_DQ_FP16,
                       "fp16_causal": FLAG_DQ_FP16 | FLAG_DQ_CAUSAL_SCALE}[dq_accum] |
                      {"dynamic": 0, "rule": FLAG_SCHEDULE_RULE,
                       "static": FLAG_SCHEDULE_STATIC}[schedule] |
                      (FLAG_DS_ROW_EXPONENTS if ds_rows else 0) |
                      (FLAG_TOKEN_SCALES if token_scales else 0) |
                      (FLAG_DS_ZERO_COUNT if ds_zero_count else 0))
        # backward only: one- or two-CTA items (head dim 128), or the library's rule
        self.bwd_flags = self.flags | {"rule": 0, "one": FLAG_BWD_ONE_CTA,
                                       "pair": FLAG_BWD_CTA_PAIR}[bwd_ctas]
        self.fmt_qk = ((FORMAT_MXFP8_NVFP4 if nvfp4_qk else FORMAT_MXFP8) |
                       (FORMAT_HADAMARD if hadamard else 0) |
                       (FORMAT_TOKEN_SCALES if token_scales else 0))
        # dO takes the same scale blocks as Q, K and V
        self.fmt_do = FORMAT_MXFP8 | (FORMAT_TOKEN_SCALES if token_scales else 0)
        self.q = QTensor(T, H, d, nvfp4_qk, device)
        self.k = QTensor(T, self.H_kv, d, nvfp4_qk, device)
        self.v = QTensor(T, self.H_kv, d, False, device)
        self.dout = QTensor(T, H, d, False, device)
        ndocs = cu_seqlens.numel() - 1
        self.wl = torch.empty(flamia_worklist_bytes(T, ndocs), dtype=torch.uint8, device=device)
        self.ws = torch.empty(flamia_bwd_workspace_bytes(T, H, d), dtype=torch.uint8, device=device)
        self.o = torch.empty((T, H, d), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((H, T), dtype=torch.float32, device=device)
        self.D = torch.empty((H, T), dtype=torch.float32, device=device)
        self.dq = torch.empty((T, H, d), dtype=torch.bfloat16, device=device)
        self.dk = torch.empty((T, self.H_kv, d), dtype=torch.bfloat16, device=device)
        self.dv = torch.empty_like(self.dk)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        # the work list is built on a side stream while Q, K, V are quantised;
        # high priority, so its small launches take SMs ahead of the waiting
        # CTAs of the quantiser's one large launch
        self.side = torch.cuda.Stream(device, priority=-1)
        self.wl_ready = torch.cuda.Event()

    def forward(self, xq, xk, xv):
        main = torch.cuda.current_stream()
        # cu_seqlens is ready and the previous call has finished with the list
        self.side.wait_stream(main)
        with torch.cuda.stream(self.side):
            flamia_build_worklist(self.cu, self.T, self.wl, dev_status=self.status)
            self.wl_ready.record(self.side)
        flamia_quantize_qkv(xq, xk, xv, self.cu, self.q, self.k, self.v, self.fmt_qk,
                            dev_status=self.status)
        main.wait_event(self.wl_ready)
        flamia_attn_fwd_gqa(self.q, self.k, self.v, self.cu, self.T, self.H, self.H_kv, self.d,
                            self.scale, self.wl, self.o, self.lse, self.flags,
                            dev_status=self.status)
        return self.o, self.lse

    def backward(self, xdo):
        flamia_quantize_tokenblock(xdo, self.cu, self.dout, self.fmt_do, o=self.o, D=self.D,
                                   dev_status=self.status)
        flamia_attn_bwd_gqa(self.q, self.k, self.v, self.dout, self.D, self.lse, self.cu, self.T,
                            self.H, self.H_kv, self.d, self.scale, self.wl, self.dq, self.dk,
                            self.dv, self.ws, self.bwd_flags, dev_status=self.status)
        return self.dq, self.dk, self.dv

    def __call__(self, xq, xk, xv, xdo):
        self.forward(xq, xk, xv)
        return self.backward(xdo)

    def ds_zero_counts(self):
        """(nonzero dS entries, those rounded to zero) of the last backward
        with ds_zero_count (reads device memory: call after it completed)."""
        off = flamia_bwd_ds_counts_offset(self.T, self.H, self.d)
        c = self.ws[off:off + 16].view(torch.int64).cpu()
        return int(c[0]), int(c[1])

    def check_status(self):
        st = int(self.status.item())
        if st != 0:
            raise RuntimeError(f"flamia device status 0x{st:x}")
