"""moe_gemv_q8_0 on the GPU: against the fp64 oracle (tolerance 1e-4), bit for bit
against the dense gemv_q8_0 on each row's expert, bad ids, unused experts."""
import numpy as np
import pytest
import torch

from helpers import TOL_Q8, check_tol, mag_q8, need_gpu, u16_to_torch
from weight_streaming_warp_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

E, TOPK = 128, 8
PROJ = {"gate_up": (1536, 2048), "down": (2048, 768)}


def _expert_weights(orc, name, Mo, K, experts):
    """q8_0 weights quantized from N(0, 0.02) bf16 for the listed experts; the
    others hold NaN scales (they must never be read)."""
    Wq = np.zeros((E, Mo, K), np.int8)
    Wd = np.full((E, Mo, K // 32), 0x7E00, np.uint16)  # binary16 NaN
    for e in experts:
        W = syn.normal(0, "%s_e%d" % (name, e), (Mo, K), 0.02, torch.bfloat16).float().numpy()
        Wq[e], Wd[e] = orc.quantize_q8(W, 32)
    return Wq, Wd


@pytest.fixture(scope="module")
def moe_weights(orc):
    return {p: _expert_weights(orc, p, Mo, K, range(E)) for p, (Mo, K) in PROJ.items()}


def _acts(orc, T, K, name):
    x = syn.normal(0, "%s_x%d" % (name, T), (T * TOPK, K)).numpy()
    return orc.quantize_q8(x, 32)


def _run(wsw, Wq, Wd, xq, xd, ids, opts=None, err_flag=None):
    return wsw.moe_gemv_q8_0(torch.from_numpy(Wq).cuda(), u16_to_torch(Wd, torch.float16).cuda(),
                             torch.from_numpy(xq).cuda(), u16_to_torch(xd, torch.float16).cuda(),
                             torch.from_numpy(ids).cuda(), opts=opts, err_flag=err_flag)


@pytest.mark.parametrize("proj", ["gate_up", "down"])
@pytest.mark.parametrize("T", [1, 16, 512])
def test_config_moe(orc, moe_weights, proj, T):
    wsw = need_gpu()
    Mo, K = PROJ[proj]
    Wq, Wd = moe_weights[proj]
    ids = syn.routing(0, "route%d" % T, T, E, TOPK).numpy()
    xq, xd = _acts(orc, T, K, proj)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = _run(wsw, Wq, Wd, xq, xd, ids, err_flag=err).cpu().numpy()
    assert err.item() == 0  # no bad id, and no bounded wait gave up
    R = T * TOPK
    rows = np.arange(R) if R <= 128 else np.unique(np.random.default_rng(T).integers(0, R, 64))
    for m in rows:
        e = ids[m]
        y64 = orc.gemv_q8_0(Wq[e], Wd[e], xq[m], xd[m])
        check_tol(y[m], y64, mag_q8(Wq[e], Wd[e], xq[m], xd[m]), TOL_Q8, "%s T=%d row %d" % (proj, T, m))


@pytest.mark.parametrize("T", [1, 16])
def test_rows_equal_dense_gemv_bitwise(orc, moe_weights, T):
    wsw = need_gpu()
    Mo, K = PROJ["gate_up"]
    Wq, Wd = moe_weights["gate_up"]
    ids = syn.routing(0, "route%d" % T, T, E, TOPK).numpy()
    xq, xd = _acts(orc, T, K, "gate_up")
    y = _run(wsw, Wq, Wd, xq, xd, ids)
    for m in range(T * TOPK):
        e = ids[m]
        yd = wsw.gemv_q8_0(torch.from_numpy(Wq[e]).cuda(), u16_to_torch(Wd[e], torch.float16).cuda(),
                           torch.from_numpy(xq[m]).cuda(), u16_to_torch(xd[m], torch.float16).cuda())
        assert torch.equal(yd.view(torch.int32), y[m].view(torch.int32)), m


def test_unused_experts_are_not_read(orc):
    wsw = need_gpu()
    Mo, K = 256, 512
    T = 4
    ids = syn.routing(5, "few", T, E, TOPK).numpy()
    Wq, Wd = _expert_weights(orc, "few", Mo, K, sorted(set(ids.tolist())))
    xq, xd = _acts(orc, T, K, "few")
    y = _run(wsw, Wq, Wd, xq, xd, ids).cpu().numpy()
    assert np.isfinite(y).all()
    for m in range(T * TOPK):
        e = ids[m]
        check_tol(y[m], orc.gemv_q8_0(Wq[e], Wd[e], xq[m], xd[m]), mag_q8(Wq[e], Wd[e], xq[m], xd[m]), TOL_Q8)


def test_bad_ids_set_the_flag_and_skip_rows(orc):
    wsw = need_gpu()
    Mo, K, En = 64, 128, 4
    g = np.random.default_rng(9)
    Wq = g.integers(-127, 128, size=(En, Mo, K)).astype(np.int8)
    Wd = g.integers(0x1000, 0x2000, size=(En, Mo, K // 32)).astype(np.uint16)
    xq = g.integers(-127, 128, size=(6, K)).astype(np.int8)
    xd = g.integers(0x1000, 0x2000, size=(6, K // 32)).astype(np.uint16)
    ids = np.array([0, 4, 3, -1, 1, 3], np.int32)
    y = torch.full((6, Mo), 5.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsw.moe_gemv_q8_0(torch.from_numpy(Wq).cuda(), u16_to_torch(Wd, torch.float16).cuda(),
                      torch.from_numpy(xq).cuda(), u16_to_torch(xd, torch.float16).cuda(),
                      torch.from_numpy(ids).cuda(), out=y, err_flag=err)
    assert err.item() == 1  # bit 0: a bad id; no wait gave up
    yc = y.cpu().numpy()
    assert (yc[1] == 5.0).all() and (yc[3] == 5.0).all()
    y64, bad = orc.moe_gemv_q8_0(Wq, Wd, xq, xd, ids)
    assert bad == 2
    for m in (0, 2, 4, 5):
        check_tol(yc[m], y64[m], mag_q8(Wq[ids[m]], Wd[ids[m]], xq[m], xd[m]), TOL_Q8)


def test_empty_and_single_row():
    wsw = need_gpu()
    Wq = torch.zeros((2, 8, 32), dtype=torch.int8, device="cuda")
    Wd = torch.zeros((2, 8, 1), dtype=torch.float16, device="cuda")
    y = wsw.moe_gemv_q8_0(Wq, Wd, torch.zeros((0, 32), dtype=torch.int8, device="cuda"),
                          torch.zeros((0, 1), dtype=torch.float16, device="cuda"),
                          torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert y.numel() == 0


def test_every_output_written_and_equal_to_dense(orc):
    """Experts with several token batches (CUDA-core form, <= 256 rows): every y entry
    is written, and sampled rows equal the dense mat-vec on their expert bit for bit."""
    wsw = need_gpu()
    En, Mo, K, T = 8, 256, 512, 32
    g = np.random.default_rng(11)
    Wq = g.integers(-127, 128, size=(En, Mo, K)).astype(np.int8)
    Wd = g.integers(0x0800, 0x1c00, size=(En, Mo, K // 32)).astype(np.uint16)
    ids = syn.routing(3, "dense_many", T, En, TOPK).numpy()
    R = T * TOPK
    xq = g.integers(-127, 128, size=(R, K)).astype(np.int8)
    xd = g.integers(0x0800, 0x1c00, size=(R, K // 32)).astype(np.uint16)
    y = torch.full((R, Mo), float("nan"), device="cuda")
    Wqd, Wdd = torch.from_numpy(Wq).cuda(), u16_to_torch(Wd, torch.float16).cuda()
    wsw.moe_gemv_q8_0(Wqd, Wdd, torch.from_numpy(xq).cuda(), u16_to_torch(xd, torch.float16).cuda(),
                      torch.from_numpy(ids).cuda(), out=y)
    assert not torch.isnan(y).any()
    for m in np.random.default_rng(0).integers(0, R, 24):
        e = ids[m]
        yd = wsw.gemv_q8_0(Wqd[e], Wdd[e], torch.from_numpy(xq[m]).cuda(), u16_to_torch(xd[m], torch.float16).cuda())
        assert torch.equal(yd.view(torch.int32), y[m].view(torch.int32)), m


@pytest.mark.parametrize("Mo,K,T,En,topk", [(200, 256, 200, 4, 2), (128, 768, 64, 16, 8), (384, 2048, 48, 8, 8)])
def test_tensor_core_form_against_oracle(orc, Mo, K, T, En, topk):
    """More than 256 rows: exact integer block sums on the tensor cores.  Experts with
    more than 64 rows (several token tiles), a partial 128-row tile, every output
    written and within 1e-4 of the fp64 oracle; a bad id is flagged and skipped."""
    wsw = need_gpu()
    g = np.random.default_rng(Mo + K + T)
    W = syn.normal(4, "tc%d_%d" % (Mo, K), (En * Mo, K), 0.02, torch.bfloat16).float().numpy()
    Wq, Wd = orc.quantize_q8(W, 32)
    Wq, Wd = Wq.reshape(En, Mo, K), Wd.reshape(En, Mo, K // 32)
    ids = syn.routing(4, "tc_route", T, En, topk).numpy()
    R = T * topk
    ids[5] = En  # out of range
    x = syn.normal(4, "tc_x%d" % K, (R, K)).numpy()
    xq, xd = orc.quantize_q8(x, 32)
    y64, bad = orc.moe_gemv_q8_0(Wq, Wd, xq, xd, ids)
    assert bad == 1
    assert wsw.moe_workspace_bytes(En, K, R) > 0
    for ws in (None, False):  # with the workspace (tensor cores) and without (CUDA cores)
        y = torch.full((R, Mo), float("nan"), device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        wsw.moe_gemv_q8_0(torch.from_numpy(Wq).cuda(), u16_to_torch(Wd, torch.float16).cuda(),
                          torch.from_numpy(xq).cuda(), u16_to_torch(xd, torch.float16).cuda(),
                          torch.from_numpy(ids).cuda(), out=y, err_flag=err, ws=ws)
        yc = y.cpu().numpy()
        assert err.item() == 1  # bit 0: a bad id; no wait gave up
        assert np.isnan(yc[5]).all()
        for m in range(R):
            if m == 5:
                continue
            e = ids[m]
            check_tol(yc[m], y64[m], mag_q8(Wq[e], Wd[e], xq[m], xd[m]), TOL_Q8, "row %d (ws %s)" % (m, ws is None))


@pytest.mark.parametrize("Mo,K,R", [(63, 96, 16), (256, 1024, 5), (1536, 2048, 1)])
def test_few_rows_gathered_form(orc, Mo, K, R):
    """At most 16 routed rows: each row streams its own expert (a repeated expert is
    read twice).  Rows equal the dense mat-vec on their expert bit for bit for every
    launch option; a bad id sets the flag and leaves its row untouched."""
    wsw = need_gpu()
    En = 6
    g = np.random.default_rng(Mo * 7 + R)
    Wq = g.integers(-127, 128, size=(En, Mo, K)).astype(np.int8)
    Wd = g.integers(0x0800, 0x1c00, size=(En, Mo, K // 32)).astype(np.uint16)
    xq = g.integers(-127, 128, size=(R, K)).astype(np.int8)
    xd = g.integers(0x0800, 0x1c00, size=(R, K // 32)).astype(np.uint16)
    ids = g.integers(0, En, size=R).astype(np.int32)
    if R > 2:
        ids[1] = ids[0]   # a repeated expert
        ids[R - 1] = En   # out of range
    Wqd, Wdd = torch.from_numpy(Wq).cuda(), u16_to_torch(Wd, torch.float16).cuda()
    xqd, xdd = torch.from_numpy(xq).cuda(), u16_to_torch(xd, torch.float16).cuda()
    ref = None
    for opts in (None, {"rows_per_warp": 1}, {"rows_per_warp": 4, "load_bytes": 8}, {"pdl": 1, "ctas_per_sm": 1}):
        y = torch.full((R, Mo), 7.0, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        wsw.moe_gemv_q8_0(Wqd, Wdd, xqd, xdd, torch.from_numpy(ids).cuda(), out=y, err_flag=err, opts=opts)
        if ref is None:
            ref = y.clone()
        assert torch.equal(y.view(torch.int32), ref.view(torch.int32)), opts
        assert err.item() == (1 if (ids >= En).any() else 0)
    for m in range(R):
        if ids[m] >= En:
            assert (ref[m] == 7.0).all()
            continue
        yd = wsw.gemv_q8_0(Wqd[ids[m]], Wdd[ids[m]], xqd[m], xdd[m])
        assert torch.equal(yd.view(torch.int32), ref[m].view(torch.int32)), m
        check_tol(ref[m].cpu().numpy(), orc.gemv_q8_0(Wq[ids[m]], Wd[ids[m]], xq[m], xd[m]),
                  mag_q8(Wq[ids[m]], Wd[ids[m]], xq[m], xd[m]), TOL_Q8, "row %d" % m)


def test_misaligned_weights_are_bit_identical(orc):
    """Weights 8 bytes off a 16-byte boundary (the load width degrades): the rows are bit
    for bit those of the aligned call and of the dense mat-vec on their expert."""
    wsw = need_gpu()
    En, Mo, K, T = 6, 512, 1024, 3
    g = np.random.default_rng(21)
    Wq = g.integers(-127, 128, size=(En, Mo, K)).astype(np.int8)
    Wd = g.integers(0x0800, 0x1c00, size=(En, Mo, K // 32)).astype(np.uint16)
    ids = syn.routing(6, "bulk_mis", T, En, 2).numpy()
    R = T * 2
    xq = g.integers(-127, 128, size=(R, K)).astype(np.int8)
    xd = g.integers(0x0800, 0x1c00, size=(R, K // 32)).astype(np.uint16)
    Wqd, Wdd = torch.from_numpy(Wq).cuda(), u16_to_torch(Wd, torch.float16).cuda()
    xqd, xdd, idd = torch.from_numpy(xq).cuda(), u16_to_torch(xd, torch.float16).cuda(), torch.from_numpy(ids).cuda()
    y = wsw.moe_gemv_q8_0(Wqd, Wdd, xqd, xdd, idd)
    buf = torch.empty(Wq.size + 8, dtype=torch.int8, device="cuda")
    Wmis = buf[8:].view(En, Mo, K)
    Wmis.copy_(Wqd)
    ym = wsw.moe_gemv_q8_0(Wmis, Wdd, xqd, xdd, idd)
    assert torch.equal(y.view(torch.int32), ym.view(torch.int32))
    for m in range(R):
        yd = wsw.gemv_q8_0(Wqd[ids[m]], Wdd[ids[m]], xqd[m], xdd[m])
        assert torch.equal(yd.view(torch.int32), y[m].view(torch.int32)), m


@pytest.mark.parametrize("Mo,K,R,En", [(64, 256, 17, 3), (99, 800, 100, 5), (256, 768, 256, 40), (1536, 2048, 128, 128)])
def test_bucketed_form_rows_equal_dense(orc, Mo, K, R, En):
    """17 to 256 routed rows (the bucketed CUDA-core form): many repeated experts, an odd
    Mo, a bad id; rows equal the dense mat-vec on their expert bit for bit for every
    launch option, and activations off a 16-byte boundary give the same bits."""
    wsw = need_gpu()
    g = np.random.default_rng(Mo + K + R)
    Wq = g.integers(-127, 128, size=(En, Mo, K)).astype(np.int8)
    Wd = g.integers(0x0800, 0x1c00, size=(En, Mo, K // 32)).astype(np.uint16)
    xq = g.integers(-127, 128, size=(R, K)).astype(np.int8)
    xd = g.integers(0x0800, 0x1c00, size=(R, K // 32)).astype(np.uint16)
    ids = g.integers(0, En, size=R).astype(np.int32)
    ids[R // 2] = -3  # out of range
    Wqd, Wdd = torch.from_numpy(Wq).cuda(), u16_to_torch(Wd, torch.float16).cuda()
    xqd, xdd = torch.from_numpy(xq).cuda(), u16_to_torch(xd, torch.float16).cuda()
    idd = torch.from_numpy(ids).cuda()
    ref = None
    for opts in (None, {"rows_per_warp": 1}, {"rows_per_warp": 4, "load_bytes": 8}, {"pdl": 1, "ctas_per_sm": 1}):
        y = torch.full((R, Mo), 7.0, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        wsw.moe_gemv_q8_0(Wqd, Wdd, xqd, xdd, idd, out=y, err_flag=err, opts=opts)
        if ref is None:
            ref = y.clone()
        assert torch.equal(y.view(torch.int32), ref.view(torch.int32)), opts
        assert err.item() == 1
    assert (ref[R // 2] == 7.0).all()
    raw = torch.zeros(xq.size + 8, dtype=torch.int8, device="cuda")
    xmis = raw[8:].view(R, K)
    xmis.copy_(xqd)
    ym = torch.full((R, Mo), 7.0, device="cuda")
    wsw.moe_gemv_q8_0(Wqd, Wdd, xmis, xdd, idd, out=ym)
    assert torch.equal(ym.view(torch.int32), ref.view(torch.int32))
    for m in range(R):
        if m == R // 2:
            continue
        if m % 7 == 0 or m < 4:
            yd = wsw.gemv_q8_0(Wqd[ids[m]], Wdd[ids[m]], xqd[m], xdd[m])
            assert torch.equal(yd.view(torch.int32), ref[m].view(torch.int32)), m
        if m % 31 == 0:
            check_tol(ref[m].cpu().numpy(), orc.gemv_q8_0(Wq[ids[m]], Wd[ids[m]], xq[m], xd[m]),
                      mag_q8(Wq[ids[m]], Wd[ids[m]], xq[m], xd[m]), TOL_Q8, "row %d" % m)
