"""The C-ABI library loads on a machine without a GPU, exports every function that
include/wsw.h declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

import weight_streaming_warp_gb300 as wsw

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(wsw_[a-z0-9_]+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    from weight_streaming_warp_gb300 import build
    build.build()
    return wsw.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"wsw_quantize_q8", "wsw_gemv_bf16", "wsw_gemv_q8_0", "wsw_moe_gemv_q8_0",
            "wsw_dequant_q8_0_kv", "wsw_gemm_bf16", "wsw_gemv_bf16_chain"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n


def test_abi_version_and_status_strings(lib):
    assert wsw.abi_version() == 7
    assert wsw.status_string(0) == "WSW_OK"
    assert wsw.status_string(1) == "WSW_ERR_INVALID_ARG"
    assert wsw.status_string(2) == "WSW_ERR_MISALIGNED"
    assert wsw.status_string(4) == "WSW_ERR_WORKSPACE"
    assert wsw.status_string(99) == "WSW_ERR_UNKNOWN"


INVALID, MISALIGNED, UNSUPPORTED = 1, 2, 3
P = ctypes.c_void_p


class _Opts(ctypes.Structure):
    _fields_ = [("rows_per_warp", ctypes.c_int32), ("load_bytes", ctypes.c_int32),
                ("pdl", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
                ("l2_prefetch_steps", ctypes.c_int32)]


def test_quantize_rejects_on_host(lib):
    f = lib.wsw_quantize_q8
    x = P(4096)
    assert f(x, 1, 64, 64, 16, P(4096), P(4096), None, None) == INVALID  # block size
    assert f(x, 1, 48, 64, 32, P(4096), P(4096), None, None) == INVALID  # n % block
    assert f(x, 1, 64, 32, 32, P(4096), P(4096), None, None) == INVALID  # ldx < n
    assert f(None, 1, 64, 64, 32, P(4096), P(4096), None, None) == INVALID
    assert f(x, -1, 64, 64, 32, P(4096), P(4096), None, None) == INVALID
    assert f(P(4098), 1, 64, 64, 32, P(4096), P(4096), None, None) == MISALIGNED
    assert f(x, 0, 64, 64, 32, None, None, None, None) == 0  # empty: nothing to do
    assert f(x, 3, 0, 0, 256, None, None, None, None) == 0
    bad = _Opts(3, 0, 0, 0)
    assert f(x, 1, 64, 64, 32, P(4096), P(4096), None, ctypes.byref(bad)) == INVALID
    bad = _Opts(0, 12, 0, 0)
    assert f(x, 1, 64, 64, 32, P(4096), P(4096), None, ctypes.byref(bad)) == INVALID


def test_gemv_rejects_on_host(lib):
    f = lib.wsw_gemv_bf16
    assert f(P(4096), 4, 64, 32, P(4096), ctypes.c_float(1.0), P(4096), None, None) == INVALID
    assert f(None, 4, 64, 64, P(4096), ctypes.c_float(1.0), P(4096), None, None) == INVALID
    assert f(P(4097), 4, 64, 64, P(4096), ctypes.c_float(1.0), P(4096), None, None) == MISALIGNED
    assert f(P(4096), 0, 64, 64, None, ctypes.c_float(1.0), None, None, None) == 0
    g = lib.wsw_gemv_q8_0
    assert g(P(4096), P(4096), 4, 48, 64, P(4096), P(4096), P(4096), None, None) == INVALID  # K % 32
    assert g(P(4096), P(4096), 4, 64, 80, P(4096), P(4096), P(4096), None, None) == INVALID  # ldq % 32
    assert g(P(4096), P(4096), 4, 64, 32, P(4096), P(4096), P(4096), None, None) == INVALID  # ldq < K
    assert g(P(4096), P(4097), 4, 64, 64, P(4096), P(4096), P(4096), None, None) == MISALIGNED
    q = lib.wsw_quantize_gemv_q8_0
    assert q(P(4096), P(4096), 4, 48, 64, P(4096), None, None, P(4096), None, None) == INVALID  # K % 32
    assert q(P(4096), P(4096), 4, 64, 64, P(4096), P(4096), None, P(4096), None, None) == INVALID  # xq without xd
    assert q(P(4096), P(4096), 4, 64, 64, None, None, None, P(4096), None, None) == INVALID  # no x
    assert q(P(4096), P(4096), 4, 64, 64, P(4098), None, None, P(4096), None, None) == MISALIGNED  # x
    assert q(P(4096), P(4096), 0, 64, 64, P(4096), None, None, None, None, None) == 0


def test_other_calls_reject_on_host(lib):
    m = lib.wsw_moe_gemv_q8_0
    assert m(P(4096), P(4096), 8, 16, 48, P(4096), P(4096), P(4096), 4, P(4096), None, None, 0, None, None) == INVALID
    assert m(P(4096), P(4096), 4096, 16, 64, P(4096), P(4096), P(4096), 4, P(4096), None, None, 0, None,
             None) == UNSUPPORTED
    assert m(P(4096), P(4096), 8, 16, 64, P(4096), P(4096), P(4096), 70000, P(4096), None, None, 0, None,
             None) == UNSUPPORTED
    assert m(P(4096), P(4096), 8, 16, 64, P(4096), P(4096), P(4096), 0, P(4096), None, None, 0, None, None) == 0
    w = lib.wsw_moe_workspace_bytes
    assert w(128, 2048, 16) == 0 and w(128, 2048, 256) == 0 and w(128, 96, 4096) == 0
    assert w(128, 2048, 4097) == 0 and w(513, 2048, 1024) == 0 and w(8, 4096, 1024) == 0  # CUDA-core sizes
    # sorted positions (R + 3 per used expert, rounded to 4): fp16 rows, fp32 scales, list, header
    n = w(128, 2048, 4096)
    rp = 4096 + 3 * 128
    assert n >= rp * 2048 * 2 + rp * 64 * 4 + rp * 2 and n % 256 == 0
    d = lib.wsw_dequant_q8_0_kv
    assert d(P(4096), P(4096), 16, 4, 100, P(4096), None, None) == INVALID
    assert d(P(4096), P(4097), 16, 4, 128, P(4096), None, None) == MISALIGNED
    assert d(P(4096), P(4096), 0, 4, 128, P(4096), None, None) == 0
    g = lib.wsw_gemm_bf16
    assert g(P(4096), 16, 64, 64, P(4104), 8, 64, P(4096), None, None) == MISALIGNED
    assert g(P(4096), 16, 60, 64, P(4096), 8, 64, P(4096), None, None) == MISALIGNED
    assert g(P(4096), 16, 64, 32, P(4096), 8, 64, P(4096), None, None) == INVALID
    c = lib.wsw_gemv_bf16_chain
    assert c(-1, None, None, None) == INVALID
    assert c(0, None, None, None) == 0
    ab = lib.wsw_attn_decode_workspace_bytes
    # one arrival counter per head (padded to 16 bytes), then one record (max, sum, two
    # pad, 128 values) per (chunk, head, query); chunks of whole 16-position steps,
    # about 152 of them over all heads
    assert ab(32768, 4, 8) == 16 + 38 * 4 * 8 * 132 * 4
    assert ab(65536, 1, 1) == 16 + 152 * 132 * 4
    assert ab(1, 5, 1) == 32 + 5 * 132 * 4
    assert ab(0, 4, 1) == 0 and ab(64, 4, 16) == 0
    a = lib.wsw_attn_decode_f16
    A = P(4096)
    def att(depth=64, heads=4, group=8, hd=128, kps=128, khs=8192, vps=128, vhs=8192, k=A, ws=A, wsn=1 << 20):
        return a(A, k, A, depth, heads, group, hd, kps, khs, vps, vhs, ctypes.c_float(0.1), A, ws, wsn, None, None)
    assert att(depth=0) == INVALID
    assert att(ws=None) == INVALID
    assert att(group=3) == UNSUPPORTED
    assert att(hd=64) == UNSUPPORTED
    assert att(kps=132) == MISALIGNED
    assert att(k=P(4104)) == MISALIGNED
    assert att(wsn=100) == 4  # WSW_ERR_WORKSPACE
    pf = lib.wsw_attn_prefill_f16

    def pre(depth=1024, heads=4, group=8, nq=512, hd=128, kps=128, khs=131072, vps=128, vhs=131072, q=A, k=A,
            out=A):
        return pf(q, k, A, depth, heads, group, nq, hd, kps, khs, vps, vhs, ctypes.c_float(0.1), out, None, None)
    assert pre(nq=0) == INVALID
    assert pre(depth=100, nq=512) == INVALID  # the batch is longer than the cache
    assert pre(q=None) == INVALID
    assert pre(hd=64) == UNSUPPORTED
    assert pre(depth=1 << 31) == UNSUPPORTED
    assert pre(kps=132) == MISALIGNED
    assert pre(out=P(4100)) == MISALIGNED
    assert pf(A, A, A, 1024, 4, 8, 512, 128, 128, 131072, 128, 131072, ctypes.c_float(0.0), A, None, None) == INVALID
    assert pre(heads=0, q=None, k=None, out=None) == 0
    wb = lib.wsw_attn_prefill_q8_0_workspace_bytes
    wb.restype = ctypes.c_size_t
    one = 4 * 4096 * 128 * 2  # one window of K (or V) as binary16
    assert wb(32768, 4, 8, 512, 4096) == 2 * one + 4 * 8 * 512 * 132 * 4
    assert wb(4096, 4, 8, 512, 4096) == 2 * one  # a single window carries no state
    assert wb(4096, 4, 8, 512, 100) == 0 and wb(0, 4, 8, 512, 128) == 0
    p8 = lib.wsw_attn_prefill_q8_0

    def pq(window=256, ws=A, wsn=1 << 30, kq=A):
        return p8(A, kq, A, A, A, 1024, 4, 8, 512, 128, ctypes.c_float(0.1), window, ws, ctypes.c_size_t(wsn), A,
                  None, None)
    assert pq(window=200) == INVALID
    assert pq(kq=None) == INVALID
    assert pq(wsn=1000) == 4  # WSW_ERR_WORKSPACE
    assert pq(ws=P(4112)) == 4  # not 256-byte aligned
    b = lib.wsw_bounded_wait_check
    assert b(2, P(4096), None) == INVALID
    assert b(0, None, None) == INVALID
    assert b(1, P(4098), None) == MISALIGNED


def test_attn_decode_workspace_covers_every_chunk(lib):
    """Host planning of the decode attention: the workspace is the 16-byte padded
    counter area plus one 132-float record per (chunk, head, query); the chunks are whole
    16-position steps that cover the depth exactly (the last one non-empty), and there
    are about one per SM over all heads (at most 152 per head, at most 152 in total once
    the heads leave more than one chunk each)."""
    ab = lib.wsw_attn_decode_workspace_bytes
    for heads in (1, 2, 3, 4, 7, 8, 32, 64, 151, 152, 153, 1000):
        for group in (1, 2, 4, 8):
            for depth in (1, 15, 16, 17, 100, 999, 4096, 32768, 65537, 1 << 20):
                n = ab(depth, heads, group)
                counters = (heads * 4 + 15) // 16 * 16
                rec = heads * group * 132 * 4
                assert n > counters and (n - counters) % rec == 0, (depth, heads, group)
                splits = (n - counters) // rec
                want = max(152 // heads, 1)
                assert 1 <= splits <= min(want, depth), (depth, heads, group, splits)
                if heads <= 152:
                    assert splits * heads <= 152
                # some whole-step chunk size makes exactly `splits` chunks of the depth
                chunk = -(-depth // want)
                chunk = -(-chunk // 16) * 16
                assert chunk % 16 == 0 and (splits - 1) * chunk < depth <= splits * chunk


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(wsw, "_lib", None)
    monkeypatch.setattr(wsw, "_LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(wsw.WswError):
        wsw.load()
