"""wsw_moe_gemv_q8_0_noalloc, the grouped MoE mat-vec for callers that cannot allocate
device memory (a plugin interface that receives only its input and output buffers, a
runtime whose memory pool is fixed at start-up).  It runs the tensor-core form on the
library's own scratch array instead of a caller workspace.  Its results are checked
against wsw_moe_gemv_q8_0 with a workspace on two calls in a row, which share that
scratch: bit for bit against the workspace form and within the q8_0 tolerance against
the oracle.  Sizes beyond the scratch are refused.

This file is collected last so that a run that stops at its first failure has run
every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

from helpers import TOL_Q8, check_tol, mag_q8, need_gpu, u16_to_torch
from weight_streaming_warp_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

UNSUPPORTED = 3


def _noalloc(wsw):
    L = wsw.load()
    f = L.wsw_moe_gemv_q8_0_noalloc
    p, i64 = ctypes.c_void_p, ctypes.c_int64
    f.argtypes = [p, p, i64, i64, i64, p, p, p, i64, p, p, p, p]
    f.restype = ctypes.c_int
    return f


def _problem(seed, En, Mo, K, T, topk):
    g = np.random.default_rng(seed)
    Wq = g.integers(-127, 128, size=(En, Mo, K)).astype(np.int8)
    Wd = g.integers(0x0c00, 0x1800, size=(En, Mo, K // 32)).astype(np.uint16)
    ids = syn.routing(seed, "noalloc", T, En, topk).numpy()
    R = T * topk
    xq = g.integers(-127, 128, size=(R, K)).astype(np.int8)
    xd = g.integers(0x2000, 0x2c00, size=(R, K // 32)).astype(np.uint16)
    return Wq, Wd, xq, xd, ids


def test_noalloc_matches_the_workspace_form_on_two_calls(orc):
    """Both forms run the same deterministic tensor-core kernel, so every valid row is
    equal bit for bit; each row is also checked against the oracle."""
    wsw = need_gpu()
    f = _noalloc(wsw)
    En, Mo, K, T, topk = 24, 384, 1024, 48, 8  # 384 routed rows: the tensor-core form
    Wq, Wd, _, _, _ = _problem(1, En, Mo, K, T, topk)
    Wqd, Wdd = torch.from_numpy(Wq).cuda(), u16_to_torch(Wd, torch.float16).cuda()
    assert wsw.moe_workspace_bytes(En, K, T * topk) > 0
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # the second call finds the first one's scratch contents
        _, _, xq, xd, ids = _problem(10 + call, En, Mo, K, T, topk)
        if call == 1:
            ids[3] = En  # an out-of-range id: flagged, its row left untouched
        xqd, xdd = torch.from_numpy(xq).cuda(), u16_to_torch(xd, torch.float16).cuda()
        idd = torch.from_numpy(ids).cuda()
        ref = torch.full((T * topk, Mo), 7.0, device="cuda")
        wsw.moe_gemv_q8_0(Wqd, Wdd, xqd, xdd, idd, out=ref)  # with a caller workspace
        y = torch.full((T * topk, Mo), 7.0, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = f(Wqd.data_ptr(), Wdd.data_ptr(), En, Mo, K, xqd.data_ptr(), xdd.data_ptr(), idd.data_ptr(),
               T * topk, y.data_ptr(), err.data_ptr(), stream, None)
        assert rc == 0, wsw.status_string(rc)
        torch.cuda.synchronize()
        assert (err.item() != 0) == (call == 1)
        assert torch.equal(y.view(torch.int32), ref.view(torch.int32)), "call %d: not bit-identical" % call
        y64, bad = orc.moe_gemv_q8_0(Wq, Wd, xq, xd, ids, y_init=np.full((T * topk, Mo), 7.0))
        assert bad == (1 if call == 1 else 0)
        yc = y.cpu().numpy()
        for m in range(T * topk):
            e = ids[m]
            if e >= En:
                assert (yc[m] == 7.0).all()
                continue
            check_tol(yc[m], y64[m], mag_q8(Wq[e], Wd[e], xq[m], xd[m]), TOL_Q8, "call %d row %d" % (call, m))


def test_noalloc_refuses_sizes_beyond_its_scratch():
    wsw = need_gpu()
    f = _noalloc(wsw)
    E, Mo, K, R = 128, 1536, 2048, 4096  # about 18 MB of workspace, more than the 8 MiB scratch
    assert wsw.moe_workspace_bytes(E, K, R) > (8 << 20)
    dummy = torch.zeros(64, dtype=torch.int32, device="cuda")  # never read: refused on the host
    p = dummy.data_ptr()
    assert f(p, p, E, Mo, K, p, p, p, R, p, None, torch.cuda.current_stream().cuda_stream, None) == UNSUPPORTED
