"""GB300 (sm_103a) FlashAttention-2 forward (plus the backward and an FP8 forward).

Thin Python binding over the C ABI declared in ``include/fa.h``: the functions
named ``fa_*`` here take plain integers (device addresses) and sizes exactly
like their C counterparts; ``forward`` / ``forward_qk`` add argument
marshalling for torch tensors (shapes, allocation of the outputs, the current
stream).  Every step of the computation runs in the CUDA kernels of
``libfa_gb300.so``; there is no CPU path.  If the library has not been built
(``python -m attention_forward_fa2_gb300.build``) any call raises.

What is computed ("GPU 内核与 FlashAttention" §10, §11.3, §14.1):
``O = softmax(scale * Q K^T) V`` per (batch, head), plus the fp32 natural-log
log-sum-exp of every score row; ``backward`` gives dQ, dK, dV from dO, O and the
log-sum-exp (§13); ``quantize_fp8`` / ``forward_fp8`` (and their ``_varlen``
forms) run the forward on block-quantised e4m3 inputs (§15.5).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa_gb300.so")
# The same library with the kernel's phase clocks compiled in (profiling only;
# `python -m attention_forward_fa2_gb300.build --phase`).
PHASE_LIB_PATH = os.path.join(PKG, "libfa_gb300_phase.so")

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_ALIGN = -3
FA_ERR_CUDA = -4
FA_ERR_TIMEOUT = -5
FA_ERR_NO_DEVICE = -6
FA_ERR_BAD_SEQLENS = -7
FA_ERR_SCRATCH_LIMIT = -8

FA_FLAG_CAUSAL = 1

# Every symbol include/fa.h declares.
EXPORTS = (
    "fa_fwd", "fa_fwd_qk", "fa_fwd_ex", "fa_check_status", "fa_strerror", "fa_last_cuda_error",
    "fa_set_timeout_ns", "fa_set_config", "fa_get_config", "fa_autotune",
    "fa_selftest_wait_timeout", "fa_version", "fa_splitkv_num_splits",
    "fa_splitkv_workspace_bytes", "fa_fwd_splitkv", "fa_fwd_splitkv_noalloc",
    "fa_bwd_workspace_bytes", "fa_bwd", "fa_bwd_varlen", "fa_fp8_sizes", "fa_quantize_fp8", "fa_fwd_fp8",
    "fa_fp8_varlen_sizes", "fa_quantize_fp8_varlen", "fa_fwd_fp8_varlen", "fa_set_phase_buffer",
)


class FaError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = "%s (FA code %d)" % (strerror(code) if _lib is not None else "error", code)
        if code == FA_ERR_CUDA and _lib is not None:
            msg += ", cudaError %d" % _lib.fa_last_cuda_error()
        super().__init__((what + ": " if what else "") + msg)


_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """Load libfa_gb300.so (raises if it is missing: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        _lib = load_library(LIB_PATH)
        return _lib


def load_library(path: str) -> ctypes.CDLL:
    """Load a build of the library (the default one or the phase-clock one) and
    declare the argument types of every C entry."""
    if not os.path.exists(path):
        raise RuntimeError("%s is not built; run `python -m attention_forward_fa2_gb300.build`"
                           % os.path.basename(path))
    L = ctypes.CDLL(path)
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, vp, vp]
    L.fa_fwd_qk.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, vp, vp, vp]
    L.fa_fwd_ex.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, vp, vp, ci, vp]
    L.fa_check_status.argtypes = [vp, ctypes.POINTER(ci)]
    L.fa_strerror.argtypes = [ci]
    L.fa_strerror.restype = ctypes.c_char_p
    L.fa_last_cuda_error.argtypes = []
    L.fa_set_timeout_ns.argtypes = [ctypes.c_ulonglong]
    L.fa_set_config.argtypes = [ctypes.c_char_p]
    L.fa_get_config.argtypes = [ci, ci, ci, ctypes.c_char_p, ci]
    L.fa_autotune.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, vp, vp]
    L.fa_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, vp]
    L.fa_version.argtypes = []
    L.fa_splitkv_num_splits.argtypes = [ci, ci, ci, ci, ci, ci]
    L.fa_splitkv_workspace_bytes.argtypes = [ci, ci, ci, ci, ci]
    L.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, ci, vp,
                                 ctypes.c_ulonglong, vp]
    L.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
    L.fa_bwd_workspace_bytes.argtypes = [ci, ci, ci, ci]
    L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp,
                         ctypes.c_longlong, vp]
    L.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci,
                                vp, ctypes.c_longlong, vp]
    L.fa_fp8_sizes.argtypes = [ci, ci, ci, ci, ci, ci, ctypes.POINTER(ctypes.c_longlong)]
    L.fa_quantize_fp8.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, ci, vp, vp, vp, vp, vp, vp, vp]
    L.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp]
    L.fa_fp8_varlen_sizes.argtypes = [ci, ci, ci, ci, ci, ci, ci, ci, ctypes.POINTER(ctypes.c_longlong)]
    L.fa_quantize_fp8_varlen.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, vp, vp, vp, vp, vp,
                                         vp, vp]
    L.fa_fwd_fp8_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, cf,
                                    ci, vp]
    L.fa_set_phase_buffer.argtypes = [vp, ctypes.c_longlong]
    for name in EXPORTS:
        if name != "fa_strerror":
            getattr(L, name).restype = ci
    L.fa_splitkv_workspace_bytes.restype = ctypes.c_longlong
    L.fa_bwd_workspace_bytes.restype = ctypes.c_longlong
    return L


# ------------------------------------------------------------ raw C-ABI calls
def fa_fwd(q, k, v, o, lse, B, N, H, d, scale, cu_seqlens, stream) -> int:
    return lib().fa_fwd(q, k, v, o, lse, B, N, H, d, scale, cu_seqlens, stream)


def fa_fwd_qk(q, k, v, o, lse, B, Nq, Nk, H, d, scale, cu_q, cu_k, stream) -> int:
    return lib().fa_fwd_qk(q, k, v, o, lse, B, Nq, Nk, H, d, scale, cu_q, cu_k, stream)


def fa_fwd_ex(q, k, v, o, lse, B, Nq, Nk, H, Hk, d, scale, cu_q, cu_k, flags, stream) -> int:
    return lib().fa_fwd_ex(q, k, v, o, lse, B, Nq, Nk, H, Hk, d, scale, cu_q, cu_k, flags, stream)


def fa_fwd_splitkv(q, k, v, o, lse, B, Nq, Nk, H, Hk, d, scale, flags, num_splits, workspace,
                   workspace_bytes, stream) -> int:
    return lib().fa_fwd_splitkv(q, k, v, o, lse, B, Nq, Nk, H, Hk, d, scale, flags, num_splits,
                                workspace, workspace_bytes, stream)


def fa_fwd_splitkv_noalloc(q, k, v, o, lse, B, Nq, Nk, H, Hk, d, scale, flags, num_splits,
                           stream) -> int:
    """Key-split forward using the library's fixed scratch (no allocation)."""
    return lib().fa_fwd_splitkv_noalloc(q, k, v, o, lse, B, Nq, Nk, H, Hk, d, scale, flags,
                                        num_splits, stream)


def splitkv_num_splits(B, Nq, Nk, H, d, requested=0) -> int:
    n = lib().fa_splitkv_num_splits(B, Nq, Nk, H, d, int(requested))
    if n < 0:
        raise FaError(n, "fa_splitkv_num_splits")
    return n


def splitkv_workspace_bytes(B, Nq, H, d, num_splits) -> int:
    n = lib().fa_splitkv_workspace_bytes(B, Nq, H, d, int(num_splits))
    if n < 0:
        raise FaError(int(n), "fa_splitkv_workspace_bytes")
    return int(n)


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, Nq, Nk, H, Hk, d, scale, flags, workspace,
           workspace_bytes, stream) -> int:
    return lib().fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, Nq, Nk, H, Hk, d, scale, flags,
                        workspace, workspace_bytes, stream)


def fa_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, cu_q, cu_k, B, max_q, max_k, H, Hk, d, scale, flags,
                  workspace, workspace_bytes, stream) -> int:
    return lib().fa_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, cu_q, cu_k, B, max_q, max_k, H, Hk, d, scale,
                               flags, workspace, workspace_bytes, stream)


def bwd_workspace_bytes(B, Nq, H, d) -> int:
    n = lib().fa_bwd_workspace_bytes(B, Nq, H, d)
    if n < 0:
        raise FaError(int(n), "fa_bwd_workspace_bytes")
    return int(n)


def fp8_sizes(B, Nq, Nk, H, Hk, d):
    """(q8 bytes, k8 bytes, vt8 bytes, q_scale, k_scale, v_scale element counts)."""
    out = (ctypes.c_longlong * 6)()
    rc = lib().fa_fp8_sizes(B, Nq, Nk, H, Hk, d, out)
    if rc != FA_OK:
        raise FaError(rc, "fa_fp8_sizes")
    return tuple(int(x) for x in out)


def fa_quantize_fp8(q, k, v, B, Nq, Nk, H, Hk, d, q8, k8, vt8, q_scale, k_scale, v_scale, stream) -> int:
    return lib().fa_quantize_fp8(q, k, v, B, Nq, Nk, H, Hk, d, q8, k8, vt8, q_scale, k_scale, v_scale, stream)


def fa_fwd_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, o, lse, B, Nq, Nk, H, Hk, d, scale, flags,
               stream) -> int:
    return lib().fa_fwd_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, o, lse, B, Nq, Nk, H, Hk, d, scale,
                            flags, stream)


def fp8_varlen_sizes(B, total_q, total_k, max_seqlen_q, max_seqlen_k, H, Hk, d):
    """fp8_sizes for packed sequences (the layouts of fa_quantize_fp8_varlen)."""
    out = (ctypes.c_longlong * 6)()
    rc = lib().fa_fp8_varlen_sizes(B, total_q, total_k, max_seqlen_q, max_seqlen_k, H, Hk, d, out)
    if rc != FA_OK:
        raise FaError(rc, "fa_fp8_varlen_sizes")
    return tuple(int(x) for x in out)


def fa_quantize_fp8_varlen(q, k, v, cu_q, cu_k, B, total_q, total_k, max_q, max_k, H, Hk, d, q8, k8, vt8,
                           q_scale, k_scale, v_scale, stream) -> int:
    return lib().fa_quantize_fp8_varlen(q, k, v, cu_q, cu_k, B, total_q, total_k, max_q, max_k, H, Hk, d, q8, k8,
                                        vt8, q_scale, k_scale, v_scale, stream)


def fa_fwd_fp8_varlen(q8, k8, vt8, q_scale, k_scale, v_scale, o, lse, cu_q, cu_k, B, total_q, total_k, max_q,
                      max_k, H, Hk, d, scale, flags, stream) -> int:
    return lib().fa_fwd_fp8_varlen(q8, k8, vt8, q_scale, k_scale, v_scale, o, lse, cu_q, cu_k, B, total_q,
                                   total_k, max_q, max_k, H, Hk, d, scale, flags, stream)


def fa_check_status(stream=None):
    info = (ctypes.c_int * 3)()
    rc = lib().fa_check_status(stream, info)
    return rc, tuple(info)


def fa_autotune(q, k, v, o, lse, B, N, H, d, scale, cu_seqlens, stream) -> int:
    return lib().fa_autotune(q, k, v, o, lse, B, N, H, d, scale, cu_seqlens, stream)


def fa_selftest_wait_timeout(timeout_ns: int, stream=None) -> int:
    return lib().fa_selftest_wait_timeout(int(timeout_ns), stream)


def strerror(code: int) -> str:
    return lib().fa_strerror(int(code)).decode()


def version() -> int:
    return lib().fa_version()


def set_timeout_ns(ns: int) -> None:
    lib().fa_set_timeout_ns(int(ns))


def set_config(spec) -> None:
    rc = lib().fa_set_config(spec.encode() if spec else None)
    if rc != FA_OK:
        raise FaError(rc, "set_config(%r)" % (spec,))


def get_config(d: int, N: int, varlen: bool = False) -> str:
    buf = ctypes.create_string_buffer(128)
    rc = lib().fa_get_config(int(d), int(N), int(bool(varlen)), buf, 128)
    if rc != FA_OK:
        raise FaError(rc, "get_config")
    return buf.value.decode()


# ------------------------------------------------------ torch-tensor wrappers
class _NoDeviceSwitch:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


_NO_SWITCH = _NoDeviceSwitch()


def _on_device(device):
    """Make `device` current for the call (no-op when it already is)."""
    import torch
    if device.index is None or device.index == torch.cuda.current_device():
        return _NO_SWITCH
    return torch.cuda.device(device)


def _stream_handle(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check_tensor(name, t, dtype, ndim):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (the library has no CPU path)" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims, got %s" % (name, ndim, tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def forward_qk(q, k, v, scale=None, cu_seqlens_q=None, cu_seqlens_k=None,
               max_seqlen_q=None, max_seqlen_k=None, out=None, lse=None, stream=None,
               causal=False):
    """Attention forward with separate query / key lengths.

    Dense: q [B, Nq, H, d], k/v [B, Nk, Hk, d] (bf16, CUDA, contiguous), H a
    multiple of Hk (grouped key/value heads).
    Variable length: q [total_q, H, d], k/v [total_k, Hk, d], cu_seqlens_* int32
    [B + 1] on the device, max_seqlen_* the longest query / key sequence.
    causal: mask keys j > i + (Nk - Nq) (bottom-right aligned).
    Returns (o, lse): o like q (bf16), lse [B, H, Nq] fp32 (natural log).
    """
    import torch
    varlen = cu_seqlens_q is not None or cu_seqlens_k is not None
    if varlen:
        if cu_seqlens_q is None or cu_seqlens_k is None or max_seqlen_q is None or max_seqlen_k is None:
            raise ValueError("variable-length form needs cu_seqlens_q/k and max_seqlen_q/k")
        for name, t in (("q", q), ("k", k), ("v", v)):
            _check_tensor(name, t, torch.bfloat16, 3)
        _check_tensor("cu_seqlens_q", cu_seqlens_q, torch.int32, 1)
        _check_tensor("cu_seqlens_k", cu_seqlens_k, torch.int32, 1)
        B = cu_seqlens_q.numel() - 1
        if cu_seqlens_k.numel() != B + 1:
            raise ValueError("cu_seqlens_q and cu_seqlens_k differ in length")
        _, H, d = q.shape
        Hk = k.shape[1]
        if k.shape[2] != d or v.shape != k.shape:
            raise ValueError("k/v shape mismatch")
        Nq, Nk = int(max_seqlen_q), int(max_seqlen_k)
    else:
        for name, t in (("q", q), ("k", k), ("v", v)):
            _check_tensor(name, t, torch.bfloat16, 4)
        B, Nq, H, d = q.shape
        Nk, Hk = k.shape[1], k.shape[2]
        if k.shape != (B, Nk, Hk, d) or v.shape != k.shape:
            raise ValueError("k/v shape mismatch")
    if Hk == 0 or H % Hk:
        raise ValueError("query heads (%d) must be a multiple of key/value heads (%d)" % (H, Hk))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_tensor("out", out, torch.bfloat16, q.dim())
        if out.shape != q.shape:
            raise ValueError("out shape mismatch")
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    else:
        _check_tensor("lse", lse, torch.float32, 3)
        if tuple(lse.shape) != (B, H, Nq):
            raise ValueError("lse must be [B, H, Nq]")
    with _on_device(q.device):
        rc = fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                       B, Nq, Nk, H, Hk, d, float(scale),
                       cu_seqlens_q.data_ptr() if varlen else None,
                       cu_seqlens_k.data_ptr() if varlen else None,
                       FA_FLAG_CAUSAL if causal else 0, _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_ex")
    return out, lse


def forward(q, k, v, scale=None, cu_seqlens=None, max_seqlen=None, out=None, lse=None,
            stream=None, causal=False):
    """Self-attention shapes (the C entry fa_fwd): dense q/k/v [B, N, H, d], or
    packed [total, H, d] with one cu_seqlens for queries and keys."""
    if cu_seqlens is not None:
        if max_seqlen is None:
            raise ValueError("max_seqlen is required with cu_seqlens")
        return forward_qk(q, k, v, scale, cu_seqlens, cu_seqlens, max_seqlen, max_seqlen,
                          out=out, lse=lse, stream=stream, causal=causal)
    return forward_qk(q, k, v, scale, out=out, lse=lse, stream=stream, causal=causal)


def check_status(stream=None):
    """Synchronise and return (code, (block, warp, site)) of the first device error."""
    import torch
    with torch.cuda.device(torch.cuda.current_device()):
        return fa_check_status(_stream_handle(stream))


def autotune(q, k, v, scale=None, cu_seqlens=None, max_seqlen=None, stream=None):
    """Time the candidate kernel configs on these tensors and keep the fastest
    for their (d, N bucket, varlen) key.  Returns the chosen config spec."""
    import torch
    varlen = cu_seqlens is not None
    if varlen:
        B = cu_seqlens.numel() - 1
        _, H, d = q.shape
        N = int(max_seqlen)
    else:
        B, N, H, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    rc = fa_autotune(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                     B, N, H, d, float(scale), cu_seqlens.data_ptr() if varlen else None,
                     _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_autotune")
    return get_config(d, N, varlen)


def forward_splitkv(q, k, v, scale=None, causal=False, num_splits=None, workspace=None, out=None,
                    lse=None, stream=None):
    """Key-split form for short query sets (dense q [B, Nq, H, d], k/v
    [B, Nk, Hk, d]).  num_splits None / 0 lets the library choose; workspace is
    a CUDA tensor of at least splitkv_workspace_bytes(...) bytes (allocated here
    through torch when None).  Returns (o, lse) like forward_qk."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(name, t, torch.bfloat16, 4)
    B, Nq, H, d = q.shape
    Nk, Hk = k.shape[1], k.shape[2]
    if k.shape != (B, Nk, Hk, d) or v.shape != k.shape:
        raise ValueError("k/v shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(q.device):
        splits = splitkv_num_splits(B, Nq, Nk, H, d, num_splits or 0)
        need = splitkv_workspace_bytes(B, Nq, H, d, splits)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        elif not workspace.is_cuda:
            raise ValueError("workspace must be a CUDA tensor")
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
        rc = fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                            B, Nq, Nk, H, Hk, d, float(scale), FA_FLAG_CAUSAL if causal else 0,
                            splits, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                            _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv")
    return out, lse


def backward(q, k, v, o, lse, dout, scale=None, causal=False, workspace=None, dq=None, dk=None,
             dv=None, stream=None):
    """Gradients (dq, dk, dv) of O = softmax(scale q k^T) v given dout = dL/dO.

    q, o, dout: [B, Nq, H, d] bf16; k, v: [B, Nk, Hk, d] bf16 (H a multiple of
    Hk); lse: [B, H, Nq] fp32 from the forward with the same causal flag;
    contiguous CUDA tensors on one device, d = 64 or 128.  workspace: optional uint8
    tensor of at least bwd_workspace_bytes(B, Nq, H, d) bytes."""
    import torch
    B, Nq, H, d = q.shape
    Nk, Hk = k.shape[1], k.shape[2]
    for t in (q, k, v, o, dout):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v, o, dout must be contiguous bf16 CUDA tensors")
    if o.shape != q.shape or dout.shape != q.shape or v.shape != k.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("shape mismatch")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B, H, Nq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = bwd_workspace_bytes(B, Nq, H, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    with _on_device(q.device):
        rc = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                    lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Nq, Nk, H, Hk, d,
                    float(scale), FA_FLAG_CAUSAL if causal else 0, workspace.data_ptr(),
                    workspace.numel(), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd")
    return dq, dk, dv


def backward_varlen(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                    scale=None, causal=False, workspace=None, dq=None, dk=None, dv=None, stream=None):
    """Gradients (dq, dk, dv) for packed sequences (the variable-length forward's
    layout): q, o, dout [total_q, H, d]; k, v [total_k, Hk, d]; cu_seqlens_q/k
    int32 [B + 1] on the device; lse [B, H, max_seqlen_q] as the forward wrote it."""
    import torch
    total_q, H, d = q.shape
    Hk = k.shape[1]
    B = cu_seqlens_q.numel() - 1
    for t in (q, k, v, o, dout):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v, o, dout must be contiguous bf16 CUDA tensors")
    if o.shape != q.shape or dout.shape != q.shape or v.shape != k.shape or k.shape[2] != d:
        raise ValueError("shape mismatch")
    for c in (cu_seqlens_q, cu_seqlens_k):
        if c.dtype != torch.int32 or not c.is_cuda or c.numel() != B + 1:
            raise ValueError("cu_seqlens must be int32 CUDA tensors of B + 1 entries")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, max_seqlen_q) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B, H, max_seqlen_q]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = bwd_workspace_bytes(B, max_seqlen_q, H, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    with _on_device(q.device):
        rc = fa_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                           lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cu_seqlens_q.data_ptr(),
                           cu_seqlens_k.data_ptr(), B, int(max_seqlen_q), int(max_seqlen_k), H, Hk, d,
                           float(scale), FA_FLAG_CAUSAL if causal else 0, workspace.data_ptr(),
                           workspace.numel(), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_varlen")
    return dq, dk, dv


class Fp8Tensors:
    """e4m3 codes and scales of one (q, k, v) triple (see quantize_fp8)."""

    def __init__(self, q8, k8, vt8, q_scale, k_scale, v_scale, shape):
        self.q8, self.k8, self.vt8 = q8, k8, vt8
        self.q_scale, self.k_scale, self.v_scale = q_scale, k_scale, v_scale
        self.B, self.Nq, self.Nk, self.H, self.Hk, self.d = shape


def quantize_fp8(q, k, v, stream=None):
    """Block-quantise bf16 q [B, Nq, H, d], k/v [B, Nk, Hk, d] to e4m3 (d = 128)."""
    import torch
    B, Nq, H, d = q.shape
    Nk, Hk = k.shape[1], k.shape[2]
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    n_q8, n_k8, n_vt8, n_qs, n_ks, n_vs = fp8_sizes(B, Nq, Nk, H, Hk, d)
    dev = q.device
    q8 = torch.empty(max(n_q8, 16), dtype=torch.uint8, device=dev)
    k8 = torch.empty(max(n_k8, 16), dtype=torch.uint8, device=dev)
    vt8 = torch.empty(max(n_vt8, 16), dtype=torch.uint8, device=dev)
    qs = torch.empty(max(n_qs, 1), dtype=torch.float32, device=dev)
    ks = torch.empty(max(n_ks, 1), dtype=torch.float32, device=dev)
    vs = torch.empty(max(n_vs, 1), dtype=torch.float32, device=dev)
    with _on_device(dev):
        rc = fa_quantize_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, Nq, Nk, H, Hk, d, q8.data_ptr(),
                             k8.data_ptr(), vt8.data_ptr(), qs.data_ptr(), ks.data_ptr(), vs.data_ptr(),
                             _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_quantize_fp8")
    return Fp8Tensors(q8, k8, vt8, qs, ks, vs, (B, Nq, Nk, H, Hk, d))


class Fp8VarlenTensors:
    """e4m3 codes and scales of packed sequences (see quantize_fp8_varlen)."""

    def __init__(self, q8, k8, vt8, q_scale, k_scale, v_scale, cu_seqlens_q, cu_seqlens_k, shape):
        self.q8, self.k8, self.vt8 = q8, k8, vt8
        self.q_scale, self.k_scale, self.v_scale = q_scale, k_scale, v_scale
        self.cu_seqlens_q, self.cu_seqlens_k = cu_seqlens_q, cu_seqlens_k
        (self.B, self.total_q, self.total_k, self.max_seqlen_q, self.max_seqlen_k,
         self.H, self.Hk, self.d) = shape


def quantize_fp8_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, stream=None):
    """Block-quantise packed bf16 q [total_q, H, d], k/v [total_k, Hk, d] per sequence (d = 128)."""
    import torch
    total_q, H, d = q.shape
    total_k, Hk = k.shape[0], k.shape[1]
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    _check_tensor("cu_seqlens_q", cu_seqlens_q, torch.int32, 1)
    _check_tensor("cu_seqlens_k", cu_seqlens_k, torch.int32, 1)
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k differ in length")
    shape = (B, total_q, total_k, int(max_seqlen_q), int(max_seqlen_k), H, Hk, d)
    n_q8, n_k8, n_vt8, n_qs, n_ks, n_vs = fp8_varlen_sizes(*shape)
    dev = q.device
    q8 = torch.empty(max(n_q8, 16), dtype=torch.uint8, device=dev)
    k8 = torch.empty(max(n_k8, 16), dtype=torch.uint8, device=dev)
    vt8 = torch.empty(max(n_vt8, 16), dtype=torch.uint8, device=dev)
    qs = torch.empty(max(n_qs, 1), dtype=torch.float32, device=dev)
    ks = torch.empty(max(n_ks, 1), dtype=torch.float32, device=dev)
    vs = torch.empty(max(n_vs, 1), dtype=torch.float32, device=dev)
    with _on_device(dev):
        rc = fa_quantize_fp8_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), cu_seqlens_q.data_ptr(),
                                    cu_seqlens_k.data_ptr(), *shape, q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(),
                                    qs.data_ptr(), ks.data_ptr(), vs.data_ptr(), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_quantize_fp8_varlen")
    return Fp8VarlenTensors(q8, k8, vt8, qs, ks, vs, cu_seqlens_q, cu_seqlens_k, shape)


def forward_fp8_varlen(t, scale=None, causal=False, out=None, lse=None, stream=None):
    """FP8 forward on Fp8VarlenTensors t; returns (o bf16 [total_q, H, d], lse fp32 [B, H, max_seqlen_q])."""
    import torch
    dev = t.q8.device
    if scale is None:
        scale = 1.0 / math.sqrt(t.d)
    out = torch.empty((t.total_q, t.H, t.d), dtype=torch.bfloat16, device=dev) if out is None else out
    lse = torch.empty((t.B, t.H, t.max_seqlen_q), dtype=torch.float32, device=dev) if lse is None else lse
    # Empty outputs (no query rows) still pass non-null pointers.
    o_arg = out if out.numel() else torch.empty(16, dtype=torch.bfloat16, device=dev)
    lse_arg = lse if lse.numel() else torch.empty(1, dtype=torch.float32, device=dev)
    with _on_device(dev):
        rc = fa_fwd_fp8_varlen(t.q8.data_ptr(), t.k8.data_ptr(), t.vt8.data_ptr(), t.q_scale.data_ptr(),
                               t.k_scale.data_ptr(), t.v_scale.data_ptr(), o_arg.data_ptr(), lse_arg.data_ptr(),
                               t.cu_seqlens_q.data_ptr(), t.cu_seqlens_k.data_ptr(), t.B, t.total_q, t.total_k,
                               t.max_seqlen_q, t.max_seqlen_k, t.H, t.Hk, t.d, float(scale),
                               FA_FLAG_CAUSAL if causal else 0, _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_fp8_varlen")
    return out, lse


def forward_fp8(t, scale=None, causal=False, out=None, lse=None, stream=None):
    """FP8 forward on Fp8Tensors t; returns (o bf16 [B, Nq, H, d], lse fp32 [B, H, Nq])."""
    import torch
    dev = t.q8.device
    if scale is None:
        scale = 1.0 / math.sqrt(t.d)
    out = torch.empty((t.B, t.Nq, t.H, t.d), dtype=torch.bfloat16, device=dev) if out is None else out
    lse = torch.empty((t.B, t.H, t.Nq), dtype=torch.float32, device=dev) if lse is None else lse
    with _on_device(dev):
        rc = fa_fwd_fp8(t.q8.data_ptr(), t.k8.data_ptr(), t.vt8.data_ptr(), t.q_scale.data_ptr(),
                        t.k_scale.data_ptr(), t.v_scale.data_ptr(), out.data_ptr(), lse.data_ptr(), t.B,
                        t.Nq, t.Nk, t.H, t.Hk, t.d, float(scale), FA_FLAG_CAUSAL if causal else 0,
                        _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_fp8")
    return out, lse
