"""ctypes front end of the C oracle (oracle.c).

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  The library under
``weight_streaming_warp_gb300`` never does, and the oracle never imports it: the
two share no code.  Inputs and outputs are numpy arrays on the host; every
function here marshals arguments and calls the C code, nothing more.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        L.orc_f32_to_f16.argtypes = [ctypes.c_float]
        L.orc_f32_to_f16.restype = ctypes.c_uint16
        L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_f16_to_f32.restype = ctypes.c_float
        L.orc_quantize_q8.argtypes = [p, i64, i64, i64, i32, p, p]
        L.orc_quantize_q8.restype = i32
        L.orc_gemv_bf16.argtypes = [p, i64, i64, i64, p, ctypes.c_double, p]
        L.orc_gemv_bf16.restype = None
        L.orc_gemv_q8_0.argtypes = [p, p, i64, i64, i64, p, p, p]
        L.orc_gemv_q8_0.restype = None
        L.orc_moe_gemv_q8_0.argtypes = [p, p, i64, i64, i64, p, p, p, i64, p]
        L.orc_moe_gemv_q8_0.restype = i64
        L.orc_gemm_bf16.argtypes = [p, i64, i64, i64, p, i64, i64, p]
        L.orc_gemm_bf16.restype = None
        L.orc_dequant_q8_0_kv.argtypes = [p, p, i64, i64, i64, p]
        L.orc_dequant_q8_0_kv.restype = None
        L.orc_attn_decode.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64, i64, i64, ctypes.c_double, p]
        L.orc_attn_decode.restype = None
        L.orc_attn_prefill.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64, i64, i64, i64,
                                       ctypes.c_double, p]
        L.orc_attn_prefill.restype = i32
        _lib = L
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError("expected %s, got %s" % (np.dtype(dtype), a.dtype))
    return np.ascontiguousarray(a)


def f32_to_f16_bits(v: float) -> int:
    return int(lib().orc_f32_to_f16(ctypes.c_float(v)))


def f16_bits_to_f32(h: int) -> float:
    return float(lib().orc_f16_to_f32(ctypes.c_uint16(h)))


def quantize_q8(x, block, n=None):
    """x: float32 [rows][ldx] (or 1-D) -> (q int8 [rows][n], scales).

    The first n columns of each row are quantized (n defaults to the row length,
    which is also the row stride ldx).  Scales are uint16 binary16 bit patterns for
    block 32 and float32 for block 256.
    """
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None, :]
    rows, ld = x.shape
    n = ld if n is None else n
    if n % block:
        raise ValueError("n must be a multiple of the block")
    q = np.zeros((rows, n), np.int8)
    sc = np.zeros((rows, n // block), np.uint16 if block == 32 else np.float32)
    rc = lib().orc_quantize_q8(_ptr(x), rows, n, ld, block, _ptr(q), _ptr(sc))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return q, sc


def gemv_bf16(W_bits, x, alpha=1.0, K=None):
    """W_bits: uint16 [M][ld] bf16 bit patterns; x: float [K] -> float64 [M]."""
    W = _c(W_bits, np.uint16)
    M, ld = W.shape
    K = ld if K is None else K
    xd = np.ascontiguousarray(np.asarray(x, dtype=np.float64)[:K])
    y = np.zeros(M, np.float64)
    lib().orc_gemv_bf16(_ptr(W), M, K, ld, _ptr(xd), float(alpha), _ptr(y))
    return y


def gemv_q8_0(Wq, Wd_bits, xq, xd_bits, K=None):
    """Wq int8 [M][ldq], Wd uint16 [M][K/32], xq int8 [K], xd uint16 [K/32] -> fp64 [M]."""
    Wq = _c(Wq, np.int8)
    Wd = _c(Wd_bits, np.uint16)
    xq = _c(xq, np.int8).reshape(-1)
    xd = _c(xd_bits, np.uint16).reshape(-1)
    M, ldq = Wq.shape
    K = ldq if K is None else K
    if Wd.shape != (M, K // 32) or xq.size < K or xd.size < K // 32:
        raise ValueError("shape mismatch")
    y = np.zeros(M, np.float64)
    lib().orc_gemv_q8_0(_ptr(Wq), _ptr(Wd), M, K, ldq, _ptr(xq), _ptr(xd), _ptr(y))
    return y


def moe_gemv_q8_0(Wq, Wd_bits, xq, xd_bits, ids, y_init=None):
    """Wq int8 [E][Mo][K], Wd uint16 [E][Mo][K/32], xq int8 [R][K], xd uint16 [R][K/32],
    ids int32 [R] -> (y fp64 [R][Mo], number of rows with an id outside [0, E))."""
    Wq = _c(Wq, np.int8)
    Wd = _c(Wd_bits, np.uint16)
    xq = _c(xq, np.int8)
    xd = _c(xd_bits, np.uint16)
    ids = _c(ids, np.int32)
    E, Mo, K = Wq.shape
    R = ids.shape[0]
    y = (np.zeros((R, Mo), np.float64) if y_init is None
         else np.array(y_init, dtype=np.float64, copy=True))
    bad = lib().orc_moe_gemv_q8_0(_ptr(Wq), _ptr(Wd), E, Mo, K, _ptr(xq), _ptr(xd),
                                  _ptr(ids), R, _ptr(y))
    return y, int(bad)


def gemm_bf16(W_bits, X_bits, K=None):
    """W uint16 [M][ld], X uint16 [N][ldx] -> Y fp64 [N][M] (first K columns used)."""
    W = _c(W_bits, np.uint16)
    X = _c(X_bits, np.uint16)
    M, ld = W.shape
    N, ldx = X.shape
    K = min(ld, ldx) if K is None else K
    Y = np.zeros((N, M), np.float64)
    lib().orc_gemm_bf16(_ptr(W), M, K, ld, _ptr(X), N, ldx, _ptr(Y))
    return Y


def dequant_q8_0_kv(q, d_bits):
    """q int8 [depth][heads][head_dim], d uint16 [depth][heads][head_dim/32]
    -> out uint16 (binary16 bits) [heads][depth][head_dim]."""
    q = _c(q, np.int8)
    d = _c(d_bits, np.uint16)
    depth, heads, hd = q.shape
    out = np.zeros((heads, depth, hd), np.uint16)
    lib().orc_dequant_q8_0_kv(_ptr(q), _ptr(d), depth, heads, hd, _ptr(out))
    return out


def attn_decode(q, k_bits, v_bits, scale, layout="per_head"):
    """q fp32 [heads][group][head_dim]; k, v uint16 (binary16 bits) laid out
    [heads][depth][head_dim] (layout "per_head") or [depth][heads][head_dim]
    ("position_major") -> out fp64 [heads][group][head_dim]."""
    q = _c(q, np.float32)
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    heads, group, hd = q.shape
    if layout == "per_head":
        depth = k.shape[1]
        ps, hs = hd, depth * hd
    elif layout == "position_major":
        depth = k.shape[0]
        ps, hs = heads * hd, hd
    else:
        raise ValueError(layout)
    out = np.zeros((heads, group, hd), np.float64)
    lib().orc_attn_decode(_ptr(q), _ptr(k), _ptr(v), depth, heads, group, hd, ps, hs, ps, hs,
                          float(scale), _ptr(out))
    return out


def attn_prefill(q_bits, k_bits, v_bits, scale, layout="per_head"):
    """q uint16 (binary16 bits) [heads][group][nq][head_dim]; k, v uint16 laid out
    [heads][depth][head_dim] ("per_head") or [depth][heads][head_dim] ("position_major")
    -> out fp64 [heads][group][nq][head_dim].  Query i sits at position depth - nq + i
    and sees positions 0 .. depth - nq + i."""
    q = _c(q_bits, np.uint16)
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    heads, group, nq, hd = q.shape
    if layout == "per_head":
        depth = k.shape[1]
        ps, hs = hd, depth * hd
    elif layout == "position_major":
        depth = k.shape[0]
        ps, hs = heads * hd, hd
    else:
        raise ValueError(layout)
    out = np.zeros((heads, group, nq, hd), np.float64)
    rc = lib().orc_attn_prefill(_ptr(q), _ptr(k), _ptr(v), depth, heads, group, nq, hd, ps, hs, ps, hs,
                                float(scale), _ptr(out))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out

