"""gemm_bf16 (small-batch prefill) on the GPU against the fp64 oracle (tolerance
1e-3), packed against padded row stride (bit-identical), and each column against
the decode GEMV of the same row of X."""
import numpy as np
import pytest
import torch

from helpers import TOL_BF16, bf16_bits, bits_to_f64_bf16, check_tol, need_gpu
from weight_streaming_warp_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

M5, K5 = 2560, 10240


@pytest.fixture(scope="module")
def w5():
    return syn.normal(0, "W5", (M5, K5), 0.02, torch.bfloat16)


def _check(orc, W, X, Y, rows, what):
    Wb, Xb = bf16_bits(W[rows]), bf16_bits(X)
    Y64 = orc.gemm_bf16(Wb, Xb)  # [N][len(rows)]
    mag = np.abs(bits_to_f64_bf16(Xb)) @ np.abs(bits_to_f64_bf16(Wb)).T
    Yc = Y.cpu().numpy()[:, rows]
    for n in range(Yc.shape[0]):
        check_tol(Yc[n], Y64[n], mag[n], TOL_BF16, "%s n=%d" % (what, n))


@pytest.mark.parametrize("N", [8, 128, 512])
def test_config_prefill(orc, w5, N):
    wsw = need_gpu()
    X = syn.normal(0, "X5_%d" % N, (N, K5), 1.0, torch.bfloat16)
    Wd, Xd = w5.cuda(), X.cuda()
    Y = wsw.gemm_bf16(Wd, Xd)
    rows = np.arange(M5) if N == 8 else np.unique(np.concatenate([[0, M5 - 1], np.random.default_rng(N).integers(0, M5, 40)]))
    _check(orc, w5, X, Y, rows, "N=%d" % N)
    # one extra 128-byte line per weight row: same bits
    Wp = wsw.upload_padded(Wd, K5 + 64)
    Yp = wsw.gemm_bf16(Wp, Xd)
    assert torch.equal(Y.view(torch.int32), Yp.view(torch.int32))


def test_columns_match_decode_gemv(w5):
    wsw = need_gpu()
    X = syn.normal(1, "Xc", (8, K5), 1.0, torch.bfloat16)
    Wd = w5.cuda()
    Y = wsw.gemm_bf16(Wd, X.cuda())
    for n in range(8):
        y = wsw.gemv_bf16(Wd, X[n].float().cuda())
        rel = (Y[n] - y).norm() / y.norm()
        assert rel.item() < 1e-4  # two fp32 sums in different orders, each within 1e-3 of fp64


@pytest.mark.parametrize("M,K,N", [(1, 8, 1), (17, 24, 3), (130, 520, 9), (300, 1000, 40), (64, 4096, 129)])
def test_ragged(orc, M, K, N):
    wsw = need_gpu()
    W = syn.normal(2, "Wr%d_%d" % (M, K), (M, K), 0.02, torch.bfloat16)
    X = syn.normal(2, "Xr%d_%d" % (N, K), (N, K), 1.0, torch.bfloat16)
    Y = wsw.gemm_bf16(W.cuda(), X.cuda())
    _check(orc, W, X, Y, np.arange(M), "%dx%dx%d" % (M, K, N))


@pytest.mark.parametrize("M,K,N", [(2560, 8192, 300), (10240, 64, 512)])
def test_wide_batches(orc, M, K, N):
    """Batches of more than 256 rows (two batch tiles): split over a cluster (2560 x 8192,
    ragged N) and more weight tiles than SMs (10240 x 64).  Whole tiles and the ragged
    last batch rows against the fp64 oracle; every output against an fp32 product
    within the same bound."""
    wsw = need_gpu()
    W = syn.normal(3, "W2a%d_%d" % (M, K), (M, K), 0.02, torch.bfloat16)
    X = syn.normal(3, "X2a%d_%d" % (N, K), (N, K), 1.0, torch.bfloat16)
    Wd, Xd = W.cuda(), X.cuda()
    Y = wsw.gemm_bf16(Wd, Xd)
    tiles = [0, 1, M // 128 - 1]
    rows = np.unique(np.concatenate([np.arange(t * 128, t * 128 + 128, 2) for t in tiles] + [[M - 1]]))
    _check(orc, W, X, Y, rows, "%dx%dx%d" % (M, K, N))
    tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        ref = Xd.float() @ Wd.float().T
        mag = Xd.float().abs() @ Wd.float().abs().T
    finally:
        torch.backends.cuda.matmul.allow_tf32 = tf32
    assert ((Y - ref).abs() <= TOL_BF16 * mag + 1e-30).all()


def test_rejects_misaligned():
    wsw = need_gpu()
    W = torch.zeros((16, 72), dtype=torch.bfloat16, device="cuda")
    X = torch.zeros((4, 72), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(wsw.WswError):
        wsw.gemm_bf16(W[:, 1:65], X[:, :64])
