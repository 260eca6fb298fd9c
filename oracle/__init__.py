"""fp64 CPU oracle for the attention forward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import this package.  The product package never does,
and the oracle imports nothing from the product.

The arithmetic lives in ``attn_ref.c`` (plain C, double precision, OpenMP over
(batch, head)); this module only compiles it with gcc and marshals numpy arrays.
What each function computes, and the passage of the pages it follows, is stated
in ``attn_ref.c``:

* ``attn_dense``      full definition, S and P materialised per (batch, head)
                      ("GPU 内核与 FlashAttention" §10, §11.1, §13.2); optional causal
                      mask (§14.4, bottom-right aligned) and grouped K/V heads (§14.2)
* ``attn_dense_rows`` the same definition for selected (b, h, i) rows
* ``attn_varlen``     packed variable-length form, lse [B, H, max_seqlen_q]
                      ("Flash Attention实现深度解析" §3.1)
* ``attn_online``     the blockwise online recurrence ("GPU 内核与 FlashAttention"
                      §11.3 and §14.1), used only to check that it is exact
* ``attn_bwd_dense``  the backward pass (§13.1): dQ, dK, dV and D_i from the full
                      materialised P, with the causal mask and grouped heads
* ``e4m3_decode`` / ``e4m3_encode`` / ``quantize_fp8``  the e4m3 format from its
                      definition and block quantisation (§15.5): the reference for
                      the quantiser
* ``attn_fp8_dense``  the definition evaluated on dequantised e4m3 inputs (optionally
                      also each row's largest score and sum_j P_ij |v_j|, the plain
                      quantities the FP8 error bound is written in)

Inputs are bf16 bit patterns (``numpy.uint16``); outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_ref.c into oracle/_build/liboracle.so (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        ci, cd = ctypes.c_int, ctypes.c_double
        lib.oracle_attn_dense.argtypes = [u16p, u16p, u16p, ci, ci, ci, ci, ci, ci, cd, ci,
                                          f64p, f64p]
        lib.oracle_attn_dense_rows.argtypes = [u16p, u16p, u16p, ci, ci, ci, ci, ci, ci, cd, ci,
                                               ci, i64p, f64p, f64p]
        lib.oracle_attn_varlen.argtypes = [u16p, u16p, u16p, i32p, i32p, ci, ci, ci, ci, cd, ci,
                                           ci, f64p, f64p]
        lib.oracle_attn_online.argtypes = [u16p, u16p, u16p, ci, ci, ci, ci, ci, cd, ci,
                                           f64p, f64p]
        lib.oracle_attn_bwd_dense.argtypes = [u16p, u16p, u16p, u16p, ci, ci, ci, ci, ci, ci, cd,
                                              ci, f64p, f64p, f64p, f64p]
        u8p = ctypes.POINTER(ctypes.c_uint8)
        f32p = ctypes.POINTER(ctypes.c_float)
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_quantize_e4m3.argtypes = [f32p, ctypes.c_longlong, ctypes.c_float, u8p]
        lib.oracle_quantize_e4m3.restype = None
        lib.oracle_attn_fp8_dense.argtypes = [u8p, u8p, u8p, f32p, f32p, f32p, ci, ci, ci, ci, ci, ci, ci,
                                              cd, ci, f64p, f64p, f64p, f64p]
        for name in ("oracle_attn_dense", "oracle_attn_dense_rows", "oracle_attn_varlen",
                     "oracle_attn_online", "oracle_attn_bwd_dense", "oracle_attn_fp8_dense",
                     "oracle_num_threads"):
            getattr(lib, name).restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ci]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
        return lib


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (numpy.uint16), got %s" % a.dtype)
    return a


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def num_threads() -> int:
    """OpenMP threads the oracle will use."""
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def _default_scale(d: int, scale):
    return (1.0 / np.sqrt(d)) if scale is None else float(scale)


def attn_dense(q, k, v, scale=None, causal=False):
    """q: [B, Nq, H, d], k/v: [B, Nk, Hk, d] (uint16 bf16 bits), H a multiple of Hk.

    Returns (o [B, Nq, H, d] float64, lse [B, H, Nq] float64)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Nq, H, d = q.shape
    Nk, Hk = k.shape[1], k.shape[2]
    if k.shape != (B, Nk, Hk, d) or v.shape != k.shape or H % Hk:
        raise ValueError("shape mismatch")
    o = np.zeros((B, Nq, H, d), np.float64)
    lse = np.zeros((B, H, Nq), np.float64)
    rc = _load().oracle_attn_dense(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                   _ptr(v, ctypes.c_uint16), B, Nq, Nk, H, Hk, d,
                                   _default_scale(d, scale), int(bool(causal)),
                                   _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise MemoryError("oracle_attn_dense failed (%d)" % rc)
    return o, lse


def attn_dense_rows(q, k, v, rows, scale=None, causal=False):
    """Selected rows of the dense definition; rows: int array [n, 3] of (b, h, i).

    Returns (o_rows [n, d], lse_rows [n])."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Nq, H, d = q.shape
    Nk, Hk = k.shape[1], k.shape[2]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = rows.shape[0]
    o = np.zeros((n, d), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = _load().oracle_attn_dense_rows(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                        _ptr(v, ctypes.c_uint16), B, Nq, Nk, H, Hk, d,
                                        _default_scale(d, scale), int(bool(causal)), n,
                                        _ptr(rows, ctypes.c_int64),
                                        _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle_attn_dense_rows failed (%d)" % rc)
    return o, lse


def attn_varlen(q, k, v, cu_q, cu_k, max_seqlen_q, scale=None, causal=False):
    """Packed form: q [total_q, H, d], k/v [total_k, Hk, d], cu_* int32 [B+1].

    Returns (o [total_q, H, d], lse [B, H, max_seqlen_q]); lse entries beyond a
    sequence's length are NaN (never written)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    cu_q = np.ascontiguousarray(cu_q, dtype=np.int32)
    cu_k = np.ascontiguousarray(cu_k, dtype=np.int32)
    _, H, d = q.shape
    Hk = k.shape[1]
    B = cu_q.shape[0] - 1
    o = np.zeros(q.shape, np.float64)
    lse = np.full((B, H, max_seqlen_q), np.nan, np.float64)
    rc = _load().oracle_attn_varlen(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                    _ptr(v, ctypes.c_uint16), _ptr(cu_q, ctypes.c_int32),
                                    _ptr(cu_k, ctypes.c_int32), B, H, Hk, d,
                                    _default_scale(d, scale), int(bool(causal)),
                                    int(max_seqlen_q),
                                    _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle_attn_varlen failed (%d)" % rc)
    return o, lse


def attn_online(q, k, v, block, scale=None):
    """Blockwise online recurrence with `block` keys per step (dense form)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    o = np.zeros((B, Nq, H, d), np.float64)
    lse = np.zeros((B, H, Nq), np.float64)
    rc = _load().oracle_attn_online(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                    _ptr(v, ctypes.c_uint16), B, Nq, Nk, H, d,
                                    _default_scale(d, scale), int(block),
                                    _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle_attn_online failed (%d)" % rc)
    return o, lse


def attn_bwd_dense(q, k, v, dout, scale=None, causal=False):
    """Backward pass.  q, dout: [B, Nq, H, d]; k, v: [B, Nk, Hk, d] (uint16 bf16 bits).

    Returns (dq [B, Nq, H, d], dk [B, Nk, Hk, d], dv [B, Nk, Hk, d], delta [B, H, Nq]),
    all float64; delta[b, h, i] = D_i = sum_j P_ij dP_ij."""
    q, k, v, dout = _u16(q), _u16(k), _u16(v), _u16(dout)
    B, Nq, H, d = q.shape
    Nk, Hk = k.shape[1], k.shape[2]
    if k.shape != (B, Nk, Hk, d) or v.shape != k.shape or dout.shape != q.shape or H % Hk:
        raise ValueError("shape mismatch")
    dq = np.zeros((B, Nq, H, d), np.float64)
    dk = np.zeros((B, Nk, Hk, d), np.float64)
    dv = np.zeros((B, Nk, Hk, d), np.float64)
    delta = np.zeros((B, H, Nq), np.float64)
    rc = _load().oracle_attn_bwd_dense(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                       _ptr(v, ctypes.c_uint16), _ptr(dout, ctypes.c_uint16),
                                       B, Nq, Nk, H, Hk, d, _default_scale(d, scale),
                                       int(bool(causal)), _ptr(dq, ctypes.c_double),
                                       _ptr(dk, ctypes.c_double), _ptr(dv, ctypes.c_double),
                                       _ptr(delta, ctypes.c_double))
    if rc != 0:
        raise MemoryError("oracle_attn_bwd_dense failed (%d)" % rc)
    return dq, dk, dv, delta


def e4m3_decode(codes):
    """Values of e4m3 codes (uint8 array -> float64 array)."""
    lib = _load()
    table = np.array([lib.oracle_e4m3_decode(c) for c in range(256)], np.float64)
    return table[np.asarray(codes, np.uint8)]


def e4m3_encode(x):
    """Nearest e4m3 codes of float64 values (ties to even, saturating)."""
    lib = _load()
    x = np.asarray(x, np.float64)
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in x.ravel()], np.uint8).reshape(x.shape)


def _quantize_block(x, scale):
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _load().oracle_quantize_e4m3(_ptr(x, ctypes.c_float), x.size, ctypes.c_float(scale),
                                 _ptr(out, ctypes.c_uint8))
    return out


def _block_scale(x):
    amax = np.float32(np.abs(np.asarray(x, np.float32)).max()) if np.asarray(x).size else np.float32(0)
    return np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)


def quantize_fp8(q, k, v):
    """Block quantisation of bf16 bit arrays q [B, Nq, H, d], k/v [B, Nk, Hk, d]:
    returns (q8, k8, vt8 [B, Hk, d, nk_pad], q_scale [B, H, qb], k_scale [B, Hk, kb],
    v_scale [B, Hk]) with scale = amax / 448 in float32 and codes of x / scale."""
    import torch
    f = lambda bits: torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(
        torch.bfloat16).to(torch.float32).numpy()
    qf, kf, vf = f(q), f(k), f(v)
    B, Nq, H, d = qf.shape
    Nk, Hk = kf.shape[1], kf.shape[2]
    qb, kb, nkp = (Nq + 127) // 128, (Nk + 127) // 128, (Nk + 15) // 16 * 16
    q8 = np.zeros(qf.shape, np.uint8)
    k8 = np.zeros(kf.shape, np.uint8)
    vt8 = np.zeros((B, Hk, d, nkp), np.uint8)
    qs = np.zeros((B, H, qb), np.float32)
    ks = np.zeros((B, Hk, kb), np.float32)
    vs = np.zeros((B, Hk), np.float32)
    for b in range(B):
        for h in range(H):
            for i in range(qb):
                blk = qf[b, i * 128:(i + 1) * 128, h]
                qs[b, h, i] = _block_scale(blk)
                q8[b, i * 128:(i + 1) * 128, h] = _quantize_block(blk, qs[b, h, i])
        for h in range(Hk):
            for j in range(kb):
                blk = kf[b, j * 128:(j + 1) * 128, h]
                ks[b, h, j] = _block_scale(blk)
                k8[b, j * 128:(j + 1) * 128, h] = _quantize_block(blk, ks[b, h, j])
            vs[b, h] = _block_scale(vf[b, :, h])
            vt8[b, h, :, :Nk] = _quantize_block(vf[b, :, h].T, vs[b, h])
    return q8, k8, vt8, qs, ks, vs


def attn_fp8_dense(q8, k8, vt8, q_scale, k_scale, v_scale, Nq, Nk, scale=None, causal=False,
                   with_bound_terms=False):
    """The attention definition on dequantised e4m3 inputs (layouts of quantize_fp8).

    Returns (o [B, Nq, H, d], lse [B, H, Nq]) in float64.  With
    ``with_bound_terms`` also (rowmax [B, H, Nq], abs_o [B, Nq, H, d]): the
    largest score each row sees and sum_j P_ij |v_j| (the weights of the
    definition applied to the magnitudes of V)."""
    q8, k8, vt8 = (np.ascontiguousarray(x, np.uint8) for x in (q8, k8, vt8))
    qs, ks, vs = (np.ascontiguousarray(x, np.float32) for x in (q_scale, k_scale, v_scale))
    B, _, H, d = q8.shape
    Hk, nkp = vt8.shape[1], vt8.shape[3]
    o = np.zeros((B, Nq, H, d), np.float64)
    lse = np.zeros((B, H, Nq), np.float64)
    rowmax = np.zeros((B, H, Nq), np.float64) if with_bound_terms else None
    abs_o = np.zeros((B, Nq, H, d), np.float64) if with_bound_terms else None
    null = ctypes.POINTER(ctypes.c_double)()
    rc = _load().oracle_attn_fp8_dense(_ptr(q8, ctypes.c_uint8), _ptr(k8, ctypes.c_uint8),
                                       _ptr(vt8, ctypes.c_uint8), _ptr(qs, ctypes.c_float),
                                       _ptr(ks, ctypes.c_float), _ptr(vs, ctypes.c_float), B, Nq, Nk, H,
                                       Hk, d, nkp, _default_scale(d, scale), int(bool(causal)),
                                       _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                                       _ptr(rowmax, ctypes.c_double) if with_bound_terms else null,
                                       _ptr(abs_o, ctypes.c_double) if with_bound_terms else null)
    if rc != 0:
        raise MemoryError("oracle_attn_fp8_dense failed (%d)" % rc)
    if with_bound_terms:
        return o, lse, rowmax, abs_o
    return o, lse
