"""gemv_q8_0 on the GPU against the fp64 oracle (tolerance 1e-4), the GPU quantizer
feeding it, and bit-identity across launch knobs and row strides."""
import numpy as np
import pytest
import torch

from helpers import TOL_Q8, check_tol, f16_bits, mag_q8, need_gpu, u16_to_torch
from weight_streaming_warp_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _make(orc, seed, M, K):
    W = syn.normal(seed, "Wq%dx%d" % (M, K), (M, K), 0.02, torch.bfloat16).float().numpy()
    Wq, Wd = orc.quantize_q8(W, 32)
    x = syn.normal(seed, "xq%d" % K, (1, K)).numpy()
    xq, xd = orc.quantize_q8(x, 32)
    return Wq, Wd, xq[0], xd[0]


def _dev(Wq, Wd, xq, xd):
    return (torch.from_numpy(Wq).cuda(), u16_to_torch(Wd, torch.float16).cuda(),
            torch.from_numpy(xq).cuda(), u16_to_torch(xd, torch.float16).cuda())


@pytest.fixture(scope="module")
def cfg2(orc):
    return _make(orc, 0, 14336, 4096)


def test_config_14336x4096_all_rows(orc, cfg2):
    wsw = need_gpu()
    Wq, Wd, xq, xd = cfg2
    y = wsw.gemv_q8_0(*_dev(Wq, Wd, xq, xd))
    y64 = orc.gemv_q8_0(Wq, Wd, xq, xd)
    check_tol(y.cpu().numpy(), y64, mag_q8(Wq, Wd, xq, xd), TOL_Q8, "14336x4096")


def test_gpu_quantizer_then_gemv(orc, cfg2):
    """The activation quantized on the GPU (bit-exact) feeds the PDL-linked GEMV."""
    wsw = need_gpu()
    Wq, Wd, _, _ = cfg2
    x = syn.normal(0, "xq4096", (1, 4096))
    Wqd, Wdd = torch.from_numpy(Wq).cuda(), u16_to_torch(Wd, torch.float16).cuda()
    xq, xd = wsw.quantize_q8(x.cuda()[0], 32, opts={"pdl": 1})
    y = wsw.gemv_q8_0(Wqd, Wdd, xq, xd, opts={"pdl": 1})
    xqr, xdr = orc.quantize_q8(x.numpy(), 32)
    assert (xq.cpu().numpy() == xqr[0]).all() and (f16_bits(xd) == xdr[0]).all()
    y64 = orc.gemv_q8_0(Wq, Wd, xqr[0], xdr[0])
    check_tol(y.cpu().numpy(), y64, mag_q8(Wq, Wd, xqr[0], xdr[0]), TOL_Q8, "chain")


@pytest.mark.parametrize("M,K", [(1, 32), (17, 544), (3, 4128), (65, 768), (257, 2048), (8, 8192)])
def test_ragged_shapes(orc, M, K):
    wsw = need_gpu()
    Wq, Wd, xq, xd = _make(orc, 1, M, K)
    y = wsw.gemv_q8_0(*_dev(Wq, Wd, xq, xd))
    check_tol(y.cpu().numpy(), orc.gemv_q8_0(Wq, Wd, xq, xd), mag_q8(Wq, Wd, xq, xd), TOL_Q8, "%dx%d" % (M, K))


def test_power_of_two_scales_exact():
    """Scales 2^-3 .. and small integers: every fp32 step is exact, so the GPU result
    equals the closed form bit for bit."""
    wsw = need_gpu()
    M, K = 40, 256
    g = torch.Generator().manual_seed(1)
    Wq = torch.randint(-4, 5, (M, K), generator=g, dtype=torch.int8)
    xq = torch.randint(-4, 5, (K,), generator=g, dtype=torch.int8)
    Wd = (2.0 ** torch.randint(-6, 0, (M, K // 32), generator=g).float()).half()
    xd = (2.0 ** torch.randint(-4, 1, (K // 32,), generator=g).float()).half()
    y = wsw.gemv_q8_0(Wq.cuda(), Wd.cuda(), xq.cuda(), xd.cuda()).cpu()
    isum = (Wq.double().view(M, K // 32, 32) * xq.double().view(K // 32, 32)).sum(-1)
    ref = (isum * Wd.double() * xd.double()).sum(-1)
    assert torch.equal(y.double(), ref)


def test_launch_knobs_and_padded_stride_bit_identical(orc, cfg2):
    wsw = need_gpu()
    Wq, Wd, xq, xd = cfg2
    Wqd, Wdd, xqd, xdd = _dev(Wq[:2000], Wd[:2000], xq, xd)
    ref = wsw.gemv_q8_0(Wqd, Wdd, xqd, xdd).clone()
    for rpw in (1, 2, 4):
        for lb in (32, 16, 8, 4):
            for pdl in (0, 1):
                y = wsw.gemv_q8_0(Wqd, Wdd, xqd, xdd, opts=dict(rows_per_warp=rpw, load_bytes=lb, pdl=pdl))
                assert torch.equal(y.view(torch.int32), ref.view(torch.int32)), (rpw, lb, pdl)
    padded = torch.zeros((2000, 4096 + 64), dtype=torch.int8, device="cuda")
    padded[:, :4096] = Wqd
    y = wsw.gemv_q8_0(padded[:, :4096], Wdd, xqd, xdd)
    assert torch.equal(y.view(torch.int32), ref.view(torch.int32))
    # base address off by 4 bytes: 4-byte loads
    off = torch.zeros(2000 * 4096 + 4, dtype=torch.int8, device="cuda")
    view = off[4:].view(2000, 4096)
    view.copy_(Wqd)
    y = wsw.gemv_q8_0(view, Wdd, xqd, xdd)
    assert torch.equal(y.view(torch.int32), ref.view(torch.int32))


def test_degenerate_sizes():
    wsw = need_gpu()
    y = wsw.gemv_q8_0(torch.empty((0, 64), dtype=torch.int8, device="cuda"),
                      torch.empty((0, 2), dtype=torch.float16, device="cuda"),
                      torch.zeros(64, dtype=torch.int8, device="cuda"),
                      torch.zeros(2, dtype=torch.float16, device="cuda"))
    assert y.numel() == 0
    with pytest.raises(wsw.WswError):
        wsw.gemv_q8_0(torch.zeros((4, 48), dtype=torch.int8, device="cuda"),
                      torch.zeros((4, 1), dtype=torch.float16, device="cuda"),
                      torch.zeros(48, dtype=torch.int8, device="cuda"),
                      torch.zeros(1, dtype=torch.float16, device="cuda"))


# ------------------------------------------------ quantizer fused into the GEMV ----

def _fused_vs_two_calls(wsw, Wqd, Wdd, x, opts=None):
    """The fused call against quantize_q8 followed by gemv_q8_0: y, xq and xd all bit
    for bit; returns the quantized activation."""
    K = x.numel()
    xq_ref, xd_ref = wsw.quantize_q8(x, 32)
    y_ref = wsw.gemv_q8_0(Wqd, Wdd, xq_ref, xd_ref, K=K)
    xq = torch.full((K,), 99, dtype=torch.int8, device="cuda")
    xd = torch.full((K // 32,), 7.0, dtype=torch.float16, device="cuda")
    y = wsw.quantize_gemv_q8_0(Wqd, Wdd, x, K=K, x_out=(xq, xd), opts=opts)
    assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32))
    assert torch.equal(xq, xq_ref) and torch.equal(xd.view(torch.int16), xd_ref.view(torch.int16))
    return y, xq, xd


def test_fused_quantize_gemv_config(orc, cfg2):
    """14336 x 4096: the fused call equals the two calls bit for bit, its quantized x
    equals the oracle's bytes, and y is within 1e-4 of the fp64 oracle."""
    wsw = need_gpu()
    Wq, Wd, _, _ = cfg2
    x = syn.normal(0, "xq4096", (1, 4096))
    Wqd, Wdd = torch.from_numpy(Wq).cuda(), u16_to_torch(Wd, torch.float16).cuda()
    y, xq, xd = _fused_vs_two_calls(wsw, Wqd, Wdd, x.cuda()[0], opts={"pdl": 1})
    xqr, xdr = orc.quantize_q8(x.numpy(), 32)
    assert (xq.cpu().numpy() == xqr[0]).all() and (f16_bits(xd) == xdr[0]).all()
    check_tol(y.cpu().numpy(), orc.gemv_q8_0(Wq, Wd, xqr[0], xdr[0]), mag_q8(Wq, Wd, xqr[0], xdr[0]), TOL_Q8, "fused")


@pytest.mark.parametrize("M,K", [(1, 32), (17, 544), (3, 4128), (65, 768), (257, 2048), (8, 8192), (4000, 14336)])
def test_fused_ragged_shapes_and_knobs(orc, M, K):
    wsw = need_gpu()
    Wq, Wd, _, _ = _make(orc, 2, M, K)
    Wqd, Wdd = torch.from_numpy(Wq).cuda(), u16_to_torch(Wd, torch.float16).cuda()
    x = syn.normal(2, "fx%d" % K, (K,)).cuda()
    x[32:64] = 0.0  # an all-zero block (d = +0, q = 0) when K > 32
    for opts in (None, dict(rows_per_warp=1, load_bytes=8, pdl=0), dict(rows_per_warp=4, load_bytes=16)):
        _fused_vs_two_calls(wsw, Wqd, Wdd, x, opts)
    # x at an address that is 4- but not 16-byte aligned: scalar loads, same bytes
    buf = torch.zeros(K + 1, device="cuda")
    buf[1:] = x
    _fused_vs_two_calls(wsw, Wqd, Wdd, buf[1:])


def test_fused_without_outputs_and_degenerate():
    wsw = need_gpu()
    M, K = 300, 1024
    g = torch.Generator(device="cuda").manual_seed(3)
    Wqd = torch.randint(-127, 128, (M, K), dtype=torch.int8, device="cuda", generator=g)
    Wdd = (torch.rand((M, K // 32), device="cuda", generator=g) * 1e-2).half()
    x = torch.randn(K, device="cuda", generator=g)
    y = wsw.quantize_gemv_q8_0(Wqd, Wdd, x)
    y_ref = wsw.gemv_q8_0(Wqd, Wdd, *wsw.quantize_q8(x, 32))
    assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32))
    # no rows: only the quantized activation is produced
    xq = torch.empty(K, dtype=torch.int8, device="cuda")
    xd = torch.empty(K // 32, dtype=torch.float16, device="cuda")
    y0 = wsw.quantize_gemv_q8_0(Wqd[:0], Wdd[:0], x, x_out=(xq, xd))
    assert y0.numel() == 0
    xq_ref, xd_ref = wsw.quantize_q8(x, 32)
    assert torch.equal(xq, xq_ref) and torch.equal(xd.view(torch.int16), xd_ref.view(torch.int16))
