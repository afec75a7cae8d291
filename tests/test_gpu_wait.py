"""The bounded mbarrier wait of the tensor-core kernels, run on its own: with an arrival
it returns at once; without one nothing can complete the phase, the wait gives up
after about a second and reports WSW_ERR_TIMEOUT through device memory, and the CUDA
context stays usable (a mat-vec launched afterwards gives the same bits and still
agrees with the oracle).  No fault, trap or endless loop is involved."""
import time

import pytest
import torch

from helpers import TOL_BF16, bf16_bits, check_tol, mag_bf16, need_gpu
from weight_streaming_warp_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

WSW_OK, WSW_ERR_TIMEOUT = 0, 6


def test_wait_returns_after_an_arrival():
    wsw = need_gpu()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    status = wsw.bounded_wait_check(True)
    torch.cuda.synchronize()
    assert status.item() == WSW_OK
    assert time.perf_counter() - t0 < 0.5


def test_wait_gives_up_and_the_context_survives(orc):
    wsw = need_gpu()
    W = syn.normal(3, "Wwait", (640, 1536), 0.02, torch.bfloat16)
    x = syn.normal(3, "xwait", (1536,))
    Wg, xg = W.cuda(), x.cuda()
    y0 = wsw.gemv_bf16(Wg, xg)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    status = wsw.bounded_wait_check(False)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert status.item() == WSW_ERR_TIMEOUT
    assert 0.9 <= waited < 30.0, waited
    y1 = wsw.gemv_bf16(Wg, xg)
    assert torch.equal(y0.view(torch.int32), y1.view(torch.int32))
    Wb, xr = bf16_bits(W), x.double().numpy()
    check_tol(y1.cpu().numpy(), orc.gemv_bf16(Wb, xr, 1.0), mag_bf16(Wb, xr), TOL_BF16, "after the timeout")
