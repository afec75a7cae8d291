"""gemv_bf16 on the GPU against the fp64 oracle (tolerance 1e-3, normwise and
componentwise), bit-identity across launch knobs, padded rows and load widths."""
import numpy as np
import pytest
import torch

from helpers import TOL_BF16, bf16_bits, check_tol, mag_bf16, need_gpu
from weight_streaming_warp_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _inputs(seed, M, K, ld=None, sigma=0.02):
    W = syn.normal(seed, "W%dx%d" % (M, K), (M, K), sigma, torch.bfloat16)
    x = syn.normal(seed, "x%d" % K, (K,))
    return W, x


def _check(orc, W, x, y, alpha=1.0, what=""):
    Wb = bf16_bits(W)
    xr = x.double().numpy()
    y64 = orc.gemv_bf16(Wb, xr, alpha)
    check_tol(y.cpu().numpy(), y64, abs(alpha) * mag_bf16(Wb, xr), TOL_BF16, what)


def test_config_4096x4096_all_rows(orc):
    wsw = need_gpu()
    W, x = _inputs(0, 4096, 4096)
    y = wsw.gemv_bf16(W.cuda(), x.cuda())
    _check(orc, W, x, y, what="4096x4096")


@pytest.mark.parametrize("M,K", [(1, 8), (5, 1001), (33, 264), (257, 4104), (3, 7),
                                 (100, 25856), (19, 30000), (1000, 5120), (2, 256)])
def test_ragged_shapes(orc, M, K):
    wsw = need_gpu()
    W, x = _inputs(1, M, K)
    y = wsw.gemv_bf16(W.cuda(), x.cuda(), alpha=0.75)
    _check(orc, W, x, y, alpha=0.75, what="%dx%d" % (M, K))


@pytest.mark.parametrize("M,K", [(4096, 4096), (37, 1000), (129, 17408)])
def test_launch_knobs_are_bit_identical(M, K):
    """rows per warp, load width, PDL and CTAs per SM change how bytes are fetched,
    never the arithmetic: the output hash is the same for all of them."""
    wsw = need_gpu()
    W, x = _inputs(2, M, K)
    Wd, xd = W.cuda(), x.cuda()
    ref = wsw.gemv_bf16(Wd, xd).clone()
    for rpw in (1, 2, 4):
        for lb in (32, 16, 8, 4, 2):
            for cps in (1, 2):
                for pdl in (0, 1):
                    y = wsw.gemv_bf16(Wd, xd, opts=dict(rows_per_warp=rpw, load_bytes=lb, ctas_per_sm=cps, pdl=pdl))
                    assert torch.equal(y.view(torch.int32), ref.view(torch.int32)), (rpw, lb, cps, pdl)


def test_padded_row_stride_is_bit_identical():
    """One extra 128-byte line per row (ld = K + 64) changes no value."""
    wsw = need_gpu()
    M, K = 2560, 10240
    W, x = _inputs(3, M, K)
    Wd, xd = W.cuda(), x.cuda()
    Wp = wsw.upload_padded(Wd, K + 64)
    assert Wp.stride(0) == K + 64
    y0 = wsw.gemv_bf16(Wd, xd)
    y1 = wsw.gemv_bf16(Wp, xd)
    assert torch.equal(y0.view(torch.int32), y1.view(torch.int32))
    # the pad holds zeros
    full = Wp.as_strided((M, K + 64), (K + 64, 1))
    assert not full[:, K:].float().abs().sum().item()


def test_misaligned_base_degrades_load_width():
    wsw = need_gpu()
    M, K = 64, 520
    W, x = _inputs(4, M, K + 1)
    Wd = W.cuda()
    view = Wd[:, 1:]  # base + 2 bytes, pitch K + 1 elements
    xd = x[1:].contiguous().cuda()
    y = wsw.gemv_bf16(view, xd)
    y2 = wsw.gemv_bf16(view.contiguous(), xd)
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))


def test_one_hot_and_integer_inputs_exact():
    wsw = need_gpu()
    W, _ = _inputs(5, 300, 512)
    Wd = W.cuda()
    for k in (0, 257, 511):
        x = torch.zeros(512, device="cuda")
        x[k] = 1.0
        y = wsw.gemv_bf16(Wd, x)
        assert torch.equal(y, Wd[:, k].float())
    g = torch.Generator().manual_seed(0)
    Wi = torch.randint(-8, 9, (70, 1000), generator=g).float()
    xi = torch.randint(-5, 6, (1000,), generator=g).float()
    y = wsw.gemv_bf16(Wi.to(torch.bfloat16).cuda(), xi.cuda())
    assert torch.equal(y.cpu(), (Wi.double() @ xi.double()).float())


def test_degenerate_sizes():
    wsw = need_gpu()
    y = wsw.gemv_bf16(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"), torch.zeros(64, device="cuda"))
    assert y.numel() == 0
    W = torch.ones((5, 16), dtype=torch.bfloat16, device="cuda")
    y = torch.full((5,), 7.0, device="cuda")
    wsw.gemv_bf16(W, torch.ones(16, device="cuda"), K=0, out=y)
    assert (y == 0).all()


@pytest.mark.parametrize("name,M,K", [("qkv", 6144, 5120), ("gate_up", 34816, 5120),
                                      ("down", 5120, 17408), ("lm_head", 152064, 5120)])
def test_decode_chain_shapes_sampled_rows(orc, name, M, K):
    """Full-size weights generated on the device; sampled rows regenerated on the
    host and checked against the oracle."""
    wsw = need_gpu()
    W = syn.normal(0, "chain_" + name, (M, K), 0.02, torch.bfloat16, device="cuda")
    x = syn.normal(0, "chain_x_" + name, (K,))
    y = wsw.gemv_bf16(W, x.cuda()).cpu()
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, 48)]))
    Wr = syn.normal_rows(0, "chain_" + name, rows, K, 0.02, torch.bfloat16)
    Wb = bf16_bits(Wr)
    xr = x.double().numpy()
    y64 = orc.gemv_bf16(Wb, xr)
    check_tol(y.numpy()[rows], y64, mag_bf16(Wb, xr), TOL_BF16, name)
