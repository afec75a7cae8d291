"""The PDL-linked decode chain: y_i feeds x_{i+1}.  Checked end to end against the
fp64 oracle chain (normwise and componentwise per link), link by link against the
oracle on the x each link was fed (the full-size 257-link chain), and bit for bit
against the same links launched one at a time without programmatic dependent launch,
eagerly and inside a CUDA graph."""
import concurrent.futures as cf
import math
import os

import numpy as np
import pytest
import torch

from helpers import TOL_BF16, bf16_bits, check_tol, need_gpu
from weight_streaming_warp_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

# one decoder layer of the 27B-shaped dense model: (name, M, K)
LAYER = [("qkv", 6144, 5120), ("o", 5120, 5120), ("gate_up", 34816, 5120), ("down", 5120, 17408)]
LM_HEAD = ("lm_head", 152064, 5120)


def _links(n_layers, dims_scale=1, lm_head=True):
    shapes = []
    for layer in range(n_layers):
        for (nm, M, K) in LAYER:
            shapes.append(("%s%d" % (nm, layer), M // dims_scale, K // dims_scale))
    if lm_head:
        shapes.append((LM_HEAD[0], LM_HEAD[1] // dims_scale, LM_HEAD[2] // dims_scale))
    return shapes


def _build(shapes, seed=0):
    Ws = [syn.normal(seed, nm, (M, K), 0.02, torch.bfloat16, device="cuda") for (nm, M, K) in shapes]
    ys = [torch.empty(M, dtype=torch.float32, device="cuda") for (_, M, _) in shapes]
    x0 = syn.normal(seed, "x0", (shapes[0][2],)).cuda()
    links = []
    for i, (nm, M, K) in enumerate(shapes):
        x = x0 if i == 0 else ys[i - 1][:K]  # the previous output, truncated to this K
        links.append((Ws[i], K, x, 1.0 / (0.02 * math.sqrt(K)), ys[i]))
    return Ws, ys, x0, links


def _alpha(K):
    return 1.0 / (0.02 * math.sqrt(K))


def _mag(W, x, alpha):
    """Componentwise scale of a link: alpha * sum_k |W_rk x_k| per row, fp64 on the host,
    by chunks of rows."""
    xa = torch.from_numpy(np.abs(np.asarray(x, np.float64)))
    out = [(W[r0:r0 + 8192].cpu().double().abs() @ xa).numpy() for r0 in range(0, W.shape[0], 8192)]
    return abs(alpha) * np.concatenate(out)


def _orc_link(orc, W, x, alpha, pool=None, parts=1):
    """The oracle on one link; with a pool its rows are cut into `parts` ranges, one
    oracle call each (the arithmetic of a row does not change)."""
    Wb = bf16_bits(W)
    if pool is None:
        return orc.gemv_bf16(Wb, x, alpha)
    cuts = [Wb.shape[0] * j // parts for j in range(parts + 1)]
    return np.concatenate(list(pool.map(lambda j: orc.gemv_bf16(Wb[cuts[j]:cuts[j + 1]], x, alpha),
                                        range(parts))))


def _oracle_chain(orc, Ws, x0, shapes):
    """fp64 oracle chain from x0: (outputs, componentwise scales) per link."""
    x = x0.double().cpu().numpy()
    outs, mags = [], []
    for W, (nm, M, K) in zip(Ws, shapes):
        y = orc.gemv_bf16(bf16_bits(W), x[:K], _alpha(K))
        outs.append(y)
        mags.append(_mag(W, x[:K], _alpha(K)))
        x = y
    return outs, mags


def _assert_chain_close(ys, ref, what):
    outs, mags = ref
    for i, (y, r, mg) in enumerate(zip(ys, outs, mags)):
        check_tol(y.cpu().double().numpy(), r, mg, TOL_BF16, "%s link %d" % (what, i))


def test_two_layers_and_lm_head_full_shapes(orc):
    wsw = need_gpu()
    shapes = _links(2)
    Ws, ys, x0, links = _build(shapes)
    wsw.gemv_bf16_chain(links)
    torch.cuda.synchronize()
    ref = _oracle_chain(orc, Ws, x0, shapes)
    _assert_chain_close(ys, ref, "pdl chain")
    pdl = [y.clone() for y in ys]
    # plain stream order, one call per link
    for (W, K, x, a, y) in links:
        wsw.gemv_bf16(W, x, alpha=a, K=K, out=y)
    for a, b in zip(pdl, ys):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_many_links_in_a_cuda_graph(orc):
    """64 small layers + head (257 links), PDL edges captured in a CUDA graph."""
    wsw = need_gpu()
    shapes = _links(64, dims_scale=16)
    Ws, ys, x0, links = _build(shapes, seed=1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        wsw.gemv_bf16_chain(links)  # warm-up (and per-device set-up) before capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        wsw.gemv_bf16_chain(links)
    for y in ys:
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    ref = _oracle_chain(orc, Ws, x0, shapes)
    _assert_chain_close(ys, ref, "graph chain")
    graph_out = [y.clone() for y in ys]
    wsw.gemv_bf16_chain(links, opts={"pdl": 0})
    for a, b in zip(graph_out, ys):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("steps", [-1, 1, 4, 64])
def test_l2_prefetch_of_the_next_link_changes_no_bit(orc, steps):
    """The finishing warps of each link request the next link's first loads into L2
    (a padded, ragged last link included); the outputs stay bit for bit those of the
    links launched one at a time."""
    wsw = need_gpu()
    shapes = _links(1) + [("ragged", 1000, 4104)]
    Ws, ys, x0, links = _build(shapes, seed=2)
    Wp = wsw.upload_padded(Ws[-1], 4104 + 64)  # the last link reads a padded matrix
    links[-1] = (Wp, 4104) + links[-1][2:]
    wsw.gemv_bf16_chain(links, opts={"pdl": 1, "l2_prefetch_steps": steps})
    torch.cuda.synchronize()
    chained = [y.clone() for y in ys]
    for (W, K, x, a, y) in links:
        wsw.gemv_bf16(W, x, alpha=a, K=K, out=y)
    for a, b in zip(chained, ys):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    ref = _oracle_chain(orc, Ws, x0, shapes)
    _assert_chain_close(ys, ref, "prefetching chain")


def test_full_size_chain_links_and_logits(orc):
    """The benched chain at full size: 64 layers x [QKV, O, gate/up, down] + lm_head, 257
    PDL-linked links over 43 GB of bf16 weights.  Links 0-3, 252-255 and the lm_head are
    checked against the oracle on the x the GPU itself fed each of them (normwise and
    componentwise), and every link and the logits against the fp64 oracle chain run
    from x_0 (normwise)."""
    wsw = need_gpu()
    shapes = _links(64)
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    Ws = [torch.randn((M, K), generator=g, device="cuda").mul_(0.02).to(torch.bfloat16) for (_, M, K) in shapes]
    ys = [torch.empty(M, dtype=torch.float32, device="cuda") for (_, M, _) in shapes]
    x0 = syn.normal(11, "x0", (shapes[0][2],)).cuda()
    links = [(Ws[i], K, x0 if i == 0 else ys[i - 1][:K], _alpha(K), ys[i]) for i, (_, M, K) in enumerate(shapes)]
    wsw.gemv_bf16_chain(links)
    torch.cuda.synchronize()
    yh = [y.cpu().double().numpy() for y in ys]
    xh0 = x0.cpu().double().numpy()
    n = len(shapes)
    parts = max(1, os.cpu_count() or 1)
    with cf.ThreadPoolExecutor(max_workers=parts) as pool:
        for i in (0, 1, 2, 3, n - 5, n - 4, n - 3, n - 2, n - 1):
            K = shapes[i][2]
            x = xh0 if i == 0 else yh[i - 1][:K]
            y64 = _orc_link(orc, Ws[i], x, _alpha(K), pool, parts)
            check_tol(yh[i], y64, _mag(Ws[i], x, _alpha(K)), TOL_BF16, "link %d (%s)" % (i, shapes[i][0]))
        x = xh0
        for i, (nm, M, K) in enumerate(shapes):
            x = _orc_link(orc, Ws[i], x[:K], _alpha(K), pool, parts)
            rel = np.linalg.norm(yh[i] - x) / np.linalg.norm(x)
            assert np.isfinite(yh[i]).all() and rel <= TOL_BF16, "chain link %d (%s): %.3g" % (i, nm, rel)
    del Ws, ys, links
    torch.cuda.empty_cache()
