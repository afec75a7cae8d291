"""weight_streaming_warp_gb300 -- Python binding of libwsw.so, the GB300 (sm_103a)
decode-time weight-streaming hot path.

Every function marshals torch tensors into the C ABI declared in include/wsw.h and
launches the library's CUDA kernels on the current torch stream.  Nothing here
computes: outputs are allocated with torch (device memory) and filled by the
kernels.  The shared library is built in-tree by ``weight_streaming_warp_gb300.build``
(or ``__graft_entry__.build()``); if it is missing, every call raises.  There is no
CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

__all__ = [
    "LaunchOpts", "WswError", "library_path", "load", "quantize_q8", "gemv_bf16",
    "gemv_bf16_chain", "gemv_q8_0", "quantize_gemv_q8_0", "moe_gemv_q8_0", "dequant_q8_0_kv", "gemm_bf16",
    "upload_padded", "status_string", "abi_version", "moe_workspace_bytes", "gemv_bf16_plan",
    "bounded_wait_check", "attn_decode_f16", "attn_decode_workspace_bytes", "attn_prefill_f16",
    "attn_prefill_q8_0", "attn_prefill_q8_0_workspace_bytes",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libwsw.so")
_lib = None

_i64, _i32, _p, _f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_float


class WswError(RuntimeError):
    pass


class _COpts(ctypes.Structure):
    _fields_ = [("rows_per_warp", ctypes.c_int32), ("load_bytes", ctypes.c_int32),
                ("pdl", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
                ("l2_prefetch_steps", ctypes.c_int32)]


class _CLink(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("M", ctypes.c_int64), ("K", ctypes.c_int64),
                ("ld", ctypes.c_int64), ("x", ctypes.c_void_p), ("alpha", ctypes.c_float),
                ("y", ctypes.c_void_p)]


class _CPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("load_bytes", "rows_per_warp", "pdl", "ctas", "threads",
                                               "log2_segments", "x_in_smem", "l2_prefetch_steps")]


@dataclass
class LaunchOpts:
    """Launch knobs (0 = library default).  None of them changes a result bit."""
    rows_per_warp: int = 0
    load_bytes: int = 0
    pdl: int = 0
    ctas_per_sm: int = 0
    l2_prefetch_steps: int = 0  # chain only: -1 = off

    def _c(self):
        return _COpts(self.rows_per_warp, self.load_bytes, self.pdl, self.ctas_per_sm, self.l2_prefetch_steps)


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libwsw.so (once).  Raises WswError if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise WswError("libwsw.so is not built (%s); run python -m weight_streaming_warp_gb300.build"
                       % _LIB_PATH)
    L = ctypes.CDLL(_LIB_PATH)
    L.wsw_status_string.argtypes = [ctypes.c_int]
    L.wsw_status_string.restype = ctypes.c_char_p
    L.wsw_abi_version.argtypes = []
    L.wsw_abi_version.restype = ctypes.c_int
    L.wsw_quantize_q8.argtypes = [_p, _i64, _i64, _i64, _i32, _p, _p, _p, _p]
    L.wsw_gemv_bf16.argtypes = [_p, _i64, _i64, _i64, _p, _f32, _p, _p, _p]
    L.wsw_gemv_bf16_chain.argtypes = [_i64, _p, _p, _p]
    L.wsw_gemv_q8_0.argtypes = [_p, _p, _i64, _i64, _i64, _p, _p, _p, _p, _p]
    L.wsw_quantize_gemv_q8_0.argtypes = [_p, _p, _i64, _i64, _i64, _p, _p, _p, _p, _p, _p]
    L.wsw_moe_gemv_q8_0.argtypes = [_p, _p, _i64, _i64, _i64, _p, _p, _p, _i64, _p, _p, _p, ctypes.c_size_t, _p, _p]
    L.wsw_moe_workspace_bytes.argtypes = [_i64, _i64, _i64]
    L.wsw_moe_workspace_bytes.restype = ctypes.c_size_t
    L.wsw_dequant_q8_0_kv.argtypes = [_p, _p, _i64, _i64, _i64, _p, _p, _p]
    L.wsw_gemm_bf16.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _i64, _p, _p, _p]
    L.wsw_gemv_bf16_plan.argtypes = [_p, _i64, _i64, _i64, _i32, _i32, _p, _p]
    L.wsw_bounded_wait_check.argtypes = [_i32, _p, _p]
    L.wsw_attn_decode_workspace_bytes.argtypes = [_i64, _i64, _i64]
    L.wsw_attn_decode_workspace_bytes.restype = ctypes.c_size_t
    L.wsw_attn_decode_f16.argtypes = [_p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _f32, _p, _p,
                                      ctypes.c_size_t, _p, _p]
    L.wsw_attn_prefill_f16.argtypes = [_p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _f32,
                                       _p, _p, _p]
    L.wsw_attn_prefill_q8_0_workspace_bytes.argtypes = [_i64, _i64, _i64, _i64, _i64]
    L.wsw_attn_prefill_q8_0_workspace_bytes.restype = ctypes.c_size_t
    L.wsw_attn_prefill_q8_0.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _f32, _i64, _p,
                                        ctypes.c_size_t, _p, _p, _p]
    L.wsw_attn_prefill_q8_0.restype = ctypes.c_int
    for f in ("wsw_quantize_q8", "wsw_gemv_bf16", "wsw_gemv_bf16_chain", "wsw_gemv_q8_0", "wsw_quantize_gemv_q8_0",
              "wsw_moe_gemv_q8_0", "wsw_dequant_q8_0_kv", "wsw_gemm_bf16", "wsw_gemv_bf16_plan",
              "wsw_bounded_wait_check", "wsw_attn_decode_f16", "wsw_attn_prefill_f16"):
        getattr(L, f).restype = ctypes.c_int
    _lib = L
    return L


def status_string(code: int) -> str:
    return load().wsw_status_string(code).decode()


def abi_version() -> int:
    return load().wsw_abi_version()


def _check(code: int, what: str):
    if code != 0:
        raise WswError("%s failed: %s" % (what, status_string(code)))


def _opts(opts):
    if opts is None:
        return None
    if isinstance(opts, dict):
        opts = LaunchOpts(**opts)
    return ctypes.byref(opts._c())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dev(t: torch.Tensor, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise WswError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise WswError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t


def _rowmajor(t: torch.Tensor, name):
    """(rows, cols, row stride) of a 2-D tensor whose last dim is contiguous."""
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise WswError("%s must be 2-D with unit stride in the last dimension" % name)
    return t.shape[0], t.shape[1], (t.stride(0) if t.shape[0] > 1 else max(t.shape[1], t.stride(0)))


# ---------------------------------------------------------------- calls ----

def quantize_q8(x: torch.Tensor, block: int = 32, out=None, opts=None):
    """x fp32 [rows][n] (or [n]) -> (q int8 [rows][n], scales).  Scales are fp16
    [rows][n/32] for block 32 and fp32 [rows][n/256] for block 256."""
    _dev(x, torch.float32, "x")
    squeeze = x.dim() == 1
    x2 = x.view(1, -1) if squeeze else x
    rows, n, ldx = _rowmajor(x2, "x")
    if out is None:
        q = torch.empty((rows, n), dtype=torch.int8, device=x.device)
        sc = torch.empty((rows, n // block), dtype=torch.float16 if block == 32 else torch.float32,
                         device=x.device)
    else:
        q, sc = out
    _check(load().wsw_quantize_q8(x2.data_ptr(), rows, n, ldx, block, q.data_ptr(), sc.data_ptr(),
                                  _stream(), _opts(opts)), "quantize_q8")
    return (q.view(-1), sc.view(-1)) if squeeze else (q, sc)


def gemv_bf16(W: torch.Tensor, x: torch.Tensor, alpha: float = 1.0, K=None, out=None, opts=None):
    """y fp32 [M] = alpha * W[:, :K] . x with W bf16 [M][ld] (row stride ld >= K)."""
    _dev(W, torch.bfloat16, "W")
    _dev(x, torch.float32, "x")
    M, cols, ld = _rowmajor(W, "W")
    K = cols if K is None else int(K)
    y = torch.empty(M, dtype=torch.float32, device=W.device) if out is None else out
    _check(load().wsw_gemv_bf16(W.data_ptr(), M, K, ld, x.data_ptr(), float(alpha), y.data_ptr(),
                                _stream(), _opts(opts)), "gemv_bf16")
    return y


def gemv_bf16_chain(links, opts=None):
    """links: iterable of (W, K, x, alpha, y) with W bf16 [M][ld] and x/y fp32 device
    tensors (x may be a view of an earlier link's y).  Launches every link back to
    back on the current stream, PDL-linked unless opts.pdl == 0 is given."""
    arr = (_CLink * len(links))()
    keep = []
    for i, (W, K, x, alpha, y) in enumerate(links):
        _dev(W, torch.bfloat16, "W")
        M, cols, ld = _rowmajor(W, "W")
        arr[i] = _CLink(W.data_ptr(), M, cols if K is None else int(K), ld, x.data_ptr(), float(alpha),
                        y.data_ptr())
        keep.append((W, x, y))
    _check(load().wsw_gemv_bf16_chain(len(links), ctypes.cast(arr, ctypes.c_void_p), _stream(),
                                      _opts(opts)), "gemv_bf16_chain")


def gemv_q8_0(Wq, Wd, xq, xd, K=None, out=None, opts=None):
    """y fp32 [M] from q8_0 weights (Wq int8 [M][ldq], Wd fp16 [M][K/32]) and a q8_0
    activation (xq int8 [K], xd fp16 [K/32])."""
    _dev(Wq, torch.int8, "Wq")
    _dev(Wd, torch.float16, "Wd")
    _dev(xq, torch.int8, "xq")
    _dev(xd, torch.float16, "xd")
    M, cols, ldq = _rowmajor(Wq, "Wq")
    K = cols if K is None else int(K)
    y = torch.empty(M, dtype=torch.float32, device=Wq.device) if out is None else out
    _check(load().wsw_gemv_q8_0(Wq.data_ptr(), Wd.data_ptr(), M, K, ldq, xq.data_ptr(), xd.data_ptr(),
                                y.data_ptr(), _stream(), _opts(opts)), "gemv_q8_0")
    return y


def quantize_gemv_q8_0(Wq, Wd, x, K=None, out=None, x_out=None, opts=None):
    """y fp32 [M] from q8_0 weights and the fp32 activation x [K], quantized to q8_0
    (block 32) inside the same launch; equals gemv_q8_0(Wq, Wd, *quantize_q8(x, 32))
    bit for bit.  x_out = (xq int8 [K], xd fp16 [K/32]) receives the quantized x."""
    _dev(Wq, torch.int8, "Wq")
    _dev(Wd, torch.float16, "Wd")
    _dev(x, torch.float32, "x")
    M, cols, ldq = _rowmajor(Wq, "Wq")
    K = cols if K is None else int(K)
    y = torch.empty(M, dtype=torch.float32, device=Wq.device) if out is None else out
    xq_p = xd_p = None
    if x_out is not None:
        _dev(x_out[0], torch.int8, "xq_out")
        _dev(x_out[1], torch.float16, "xd_out")
        xq_p, xd_p = x_out[0].data_ptr(), x_out[1].data_ptr()
    _check(load().wsw_quantize_gemv_q8_0(Wq.data_ptr(), Wd.data_ptr(), M, K, ldq, x.data_ptr(), xq_p, xd_p,
                                         y.data_ptr(), _stream(), _opts(opts)), "quantize_gemv_q8_0")
    return y


def moe_workspace_bytes(E, K, R) -> int:
    """Device workspace bytes that moe_gemv_q8_0 can use for these sizes (0: none)."""
    return int(load().wsw_moe_workspace_bytes(E, K, R))


def moe_gemv_q8_0(Wq, Wd, xq, xd, ids, out=None, err_flag=None, opts=None, ws=None):
    """Grouped q8_0 mat-vec.  Wq int8 [E][Mo][K], Wd fp16 [E][Mo][K/32], xq int8 [R][K],
    xd fp16 [R][K/32], ids int32 [R] -> y fp32 [R][Mo].  Rows with an id outside
    [0, E) are skipped and set err_flag (an int32 device tensor) nonzero.  ws: a uint8
    device tensor of at least moe_workspace_bytes(E, K, R) bytes; by default one is
    allocated when the call can use it, ws=False runs without one."""
    _dev(Wq, torch.int8, "Wq")
    _dev(Wd, torch.float16, "Wd")
    _dev(xq, torch.int8, "xq")
    _dev(xd, torch.float16, "xd")
    _dev(ids, torch.int32, "ids")
    E, Mo, K = Wq.shape
    R = ids.shape[0]
    for t, nm in ((Wq, "Wq"), (Wd, "Wd"), (xq, "xq"), (xd, "xd"), (ids, "ids")):
        if not t.is_contiguous():
            raise WswError("%s must be contiguous" % nm)
    y = torch.empty((R, Mo), dtype=torch.float32, device=Wq.device) if out is None else out
    errp = err_flag.data_ptr() if err_flag is not None else None
    if ws is None:
        nbytes = moe_workspace_bytes(E, K, R)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=Wq.device) if nbytes else False
    wsp, wsn = (ws.data_ptr(), ws.numel()) if ws is not False else (None, 0)
    _check(load().wsw_moe_gemv_q8_0(Wq.data_ptr(), Wd.data_ptr(), E, Mo, K, xq.data_ptr(),
                                    xd.data_ptr(), ids.data_ptr(), R, y.data_ptr(), errp, wsp, wsn,
                                    _stream(), _opts(opts)), "moe_gemv_q8_0")
    return y


def dequant_q8_0_kv(q, d, out=None, opts=None):
    """q int8 [depth][heads][head_dim], d fp16 [depth][heads][head_dim/32] ->
    fp16 [heads][depth][head_dim]."""
    _dev(q, torch.int8, "q")
    _dev(d, torch.float16, "d")
    if not (q.is_contiguous() and d.is_contiguous()):
        raise WswError("q and d must be contiguous")
    depth, heads, hd = q.shape
    o = torch.empty((heads, depth, hd), dtype=torch.float16, device=q.device) if out is None else out
    _check(load().wsw_dequant_q8_0_kv(q.data_ptr(), d.data_ptr(), depth, heads, hd, o.data_ptr(),
                                      _stream(), _opts(opts)), "dequant_q8_0_kv")
    return o


def gemm_bf16(W, X, K=None, out=None, opts=None):
    """Y fp32 [N][M] = X[:, :K] . W[:, :K]^T with W bf16 [M][ld], X bf16 [N][ldx]."""
    _dev(W, torch.bfloat16, "W")
    _dev(X, torch.bfloat16, "X")
    M, wc, ld = _rowmajor(W, "W")
    N, xc, ldx = _rowmajor(X, "X")
    K = min(wc, xc) if K is None else int(K)
    Y = torch.empty((N, M), dtype=torch.float32, device=W.device) if out is None else out
    _check(load().wsw_gemm_bf16(W.data_ptr(), M, K, ld, X.data_ptr(), N, ldx, Y.data_ptr(),
                                _stream(), _opts(opts)), "gemm_bf16")
    return Y


def gemv_bf16_plan(W_addr: int, M: int, K: int, ld: int, sm_count: int = 152, chain: bool = False,
                   opts=None) -> dict:
    """The launch that gemv_bf16 (chain=False) or a link of gemv_bf16_chain (chain=True)
    makes for a weight matrix at device address W_addr (only its alignment matters),
    as a dict of the wsw_gemv_plan fields.  Host only: no CUDA call."""
    p = _CPlan()
    _check(load().wsw_gemv_bf16_plan(ctypes.c_void_p(W_addr), M, K, ld, sm_count, int(bool(chain)),
                                      _opts(opts), ctypes.byref(p)), "wsw_gemv_bf16_plan")
    return {n: getattr(p, n) for n, _ in _CPlan._fields_}


def bounded_wait_check(arrive: bool) -> torch.Tensor:
    """Run the tensor-core kernels' bounded wait on its own; returns the int32 device
    status it writes (0 = WSW_OK after an arrival, 6 = WSW_ERR_TIMEOUT after about a
    second without one)."""
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _check(load().wsw_bounded_wait_check(int(bool(arrive)), status.data_ptr(), _stream()),
           "wsw_bounded_wait_check")
    return status


def attn_decode_workspace_bytes(depth, heads, group) -> int:
    return int(load().wsw_attn_decode_workspace_bytes(depth, heads, group))


def attn_decode_f16(q, k, v, scale=None, out=None, ws=None, opts=None):
    """One decoding step of attention.  q fp32 [heads][group][head_dim]; k and v fp16
    views indexed [head][position][dim] with unit stride in dim and any head and
    position strides (the per-head-contiguous scratch as is, the position-major cache
    as cache.permute(1, 0, 2)).  scale defaults to 1/sqrt(head_dim).  Returns out fp32
    [heads][group][head_dim].  ws: a uint8 device tensor of at least
    attn_decode_workspace_bytes(depth, heads, group) bytes, zero-filled before its first
    use (every call leaves it ready for the next), allocated if None."""
    _dev(q, torch.float32, "q")
    _dev(k, torch.float16, "k")
    _dev(v, torch.float16, "v")
    if q.dim() != 3 or not q.is_contiguous():
        raise WswError("q must be a contiguous [heads][group][head_dim] tensor")
    heads, group, hd = q.shape
    for t, n in ((k, "k"), (v, "v")):
        if t.dim() != 3 or t.shape[0] != heads or t.shape[2] != hd or t.shape[1] != k.shape[1] or t.stride(2) != 1:
            raise WswError("%s must be a [heads][depth][head_dim] view with unit stride in head_dim" % n)
    depth = k.shape[1]
    if scale is None:
        scale = 1.0 / float(hd) ** 0.5
    y = out if out is not None else torch.empty((heads, group, hd), dtype=torch.float32, device=q.device)
    need = attn_decode_workspace_bytes(depth, heads, group)
    if ws is None:
        ws = torch.zeros(max(need, 1), dtype=torch.uint8, device=q.device)
    _check(load().wsw_attn_decode_f16(q.data_ptr(), k.data_ptr(), v.data_ptr(), depth, heads, group, hd,
                                      k.stride(1), k.stride(0), v.stride(1), v.stride(0), float(scale),
                                      y.data_ptr(), ws.data_ptr(), ws.numel(), _stream(), _opts(opts)),
           "attn_decode_f16")
    return y


def attn_prefill_f16(q, k, v, scale=None, out=None, opts=None):
    """Causal prefill attention on the tensor cores.  q fp16 [heads][group][nq][head_dim]
    (contiguous); k and v fp16 views indexed [head][position][dim] with unit stride in
    dim and any head and position strides (multiples of 8).  Query i sits at position
    depth - nq + i and sees positions 0 .. depth - nq + i.  scale defaults to
    1/sqrt(head_dim).  Returns out fp32 [heads][group][nq][head_dim]."""
    _dev(q, torch.float16, "q")
    _dev(k, torch.float16, "k")
    _dev(v, torch.float16, "v")
    if q.dim() != 4 or not q.is_contiguous():
        raise WswError("q must be a contiguous [heads][group][nq][head_dim] tensor")
    heads, group, nq, hd = q.shape
    for t, n in ((k, "k"), (v, "v")):
        if t.dim() != 3 or t.shape[0] != heads or t.shape[2] != hd or t.shape[1] != k.shape[1] or t.stride(2) != 1:
            raise WswError("%s must be a [heads][depth][head_dim] view with unit stride in head_dim" % n)
    depth = k.shape[1]
    if scale is None:
        scale = 1.0 / float(hd) ** 0.5
    y = out if out is not None else torch.empty((heads, group, nq, hd), dtype=torch.float32, device=q.device)
    _check(load().wsw_attn_prefill_f16(q.data_ptr(), k.data_ptr(), v.data_ptr(), depth, heads, group, nq, hd,
                                       k.stride(1), k.stride(0), v.stride(1), v.stride(0), float(scale),
                                       y.data_ptr(), _stream(), _opts(opts)), "attn_prefill_f16")
    return y


def attn_prefill_q8_0_workspace_bytes(depth, heads, group, nq, window) -> int:
    return int(load().wsw_attn_prefill_q8_0_workspace_bytes(depth, heads, group, nq, window))


def attn_prefill_q8_0(q, kq, kd, vq, vd, window, scale=None, out=None, ws=None, opts=None):
    """Causal prefill attention over a q8_0 KV cache, dequantized and attended one window
    of `window` positions at a time (a multiple of 128), so the binary16 scratch holds one
    window of K and V.  q fp16 [heads][group][nq][head_dim]; kq, vq int8
    [depth][heads][head_dim]; kd, vd fp16 [depth][heads][head_dim/32].  ws: a uint8 device
    tensor of at least attn_prefill_q8_0_workspace_bytes(...) bytes, allocated if None.
    Returns out fp32 [heads][group][nq][head_dim]."""
    _dev(q, torch.float16, "q")
    for t, n, dt in ((kq, "kq", torch.int8), (vq, "vq", torch.int8), (kd, "kd", torch.float16),
                     (vd, "vd", torch.float16)):
        _dev(t, dt, n)
        if not t.is_contiguous():
            raise WswError("%s must be contiguous" % n)
    if q.dim() != 4 or not q.is_contiguous():
        raise WswError("q must be a contiguous [heads][group][nq][head_dim] tensor")
    heads, group, nq, hd = q.shape
    depth = kq.shape[0]
    if scale is None:
        scale = 1.0 / float(hd) ** 0.5
    y = out if out is not None else torch.empty((heads, group, nq, hd), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = torch.empty(max(attn_prefill_q8_0_workspace_bytes(depth, heads, group, nq, window), 1),
                         dtype=torch.uint8, device=q.device)
    _check(load().wsw_attn_prefill_q8_0(q.data_ptr(), kq.data_ptr(), kd.data_ptr(), vq.data_ptr(), vd.data_ptr(),
                                        depth, heads, group, nq, hd, float(scale), int(window), ws.data_ptr(),
                                        ws.numel(), y.data_ptr(), _stream(), _opts(opts)), "attn_prefill_q8_0")
    return y


def upload_padded(W: torch.Tensor, ld: int, device=None) -> torch.Tensor:
    """Copy a [M][K] weight into a new [M][ld] device buffer whose pad columns are
    zero (so they can never hold NaNs) and return the [M][K] view with row stride ld.
    Padding the row stride by one cache line breaks cache-set aliasing of rows whose
    byte length is a multiple of the set stride."""
    M, K = W.shape
    if ld < K:
        raise WswError("ld must be >= K")
    dev = device if device is not None else (W.device if W.is_cuda else torch.device("cuda"))
    buf = torch.zeros((M, ld), dtype=W.dtype, device=dev)
    buf[:, :K].copy_(W, non_blocking=True)
    return buf[:, :K]
