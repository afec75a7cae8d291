"""Causal prefill attention on the tensor cores (the flash-attention pass that reads the
dequantized binary16 KV) against the fp64 oracle.

Tolerance: the kernel rounds the softmax probabilities P to binary16 before the P V
product (relative error 2^-11 per probability) and accumulates in fp32, so an output
element differs from the exact one by at most about 2^-11 * (m_d + |out_d|), with
m_d = sum_p w_p |V_p,d| / sum_p w_p the weighted magnitude of the values.  The tests
require |out - out64| <= 1e-3 * (m_d + |out64_d|) per element (twice that bound) and the
same normwise per query row.

Cases: ragged query batches and depths (neither a multiple of the 128-row tiles), a
batch that fills the cache (its first query sees one position), a single query, both
of the page's layouts, large scores (the running maximum is raised mid-row), the
dequant-then-attend pipeline, and the configured depths 32768 and 65536 with 4 KV heads,
8 query heads each and 512 queries, checked on sampled queries (each one is the oracle
for a single query at the end of its visible prefix).

The windowed q8_0 pass (dequantize and attend one window of positions at a time, the
online-softmax state carried between windows) is checked the same way against the
oracle's attention over the oracle's dequantized cache: short last windows, windows past
the causal limit of early query tiles, one window, large scores, and the configured
depths with windows of 4096 and 8192 positions."""
import math

import numpy as np
import pytest
import torch

from helpers import f16_bits, need_gpu, u16_to_torch
from weight_streaming_warp_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

TOL = 1e-3


def _inputs(seed, heads, group, nq, depth, qsigma=1.0):
    q = syn.normal(seed, "pq%d_%d_%d" % (heads, group, nq), (heads, group, nq, 128), qsigma, torch.float16)
    k = syn.normal(seed, "pk%d_%d" % (heads, depth), (heads, depth, 128), dtype=torch.float16)
    v = syn.normal(seed, "pv%d_%d" % (heads, depth), (heads, depth, 128), dtype=torch.float16)
    return q, k, v


def _magnitude_row(qrow, kb, vb, scale):
    """sum_p w_p |V_p| / sum_p w_p over the visible positions of one query (fp64)."""
    kf = kb.view(np.float16).astype(np.float64)
    s = kf @ qrow.astype(np.float64) * scale
    w = np.exp(s - s.max())
    return (w @ np.abs(vb.view(np.float16).astype(np.float64))) / w.sum()


def _check_row(got, ref, mag, what):
    assert np.isfinite(got).all(), what
    bound = TOL * (mag + np.abs(ref))
    bad = np.nonzero(np.abs(got - ref) > bound)[0]
    assert bad.size == 0, "%s: %d dims over tolerance, first %d: %g vs %g (bound %g)" % (
        what, bad.size, bad[0], got[bad[0]], ref[bad[0]], bound[bad[0]])
    assert np.linalg.norm(got - ref) <= TOL * np.linalg.norm(mag + np.abs(ref)), what


def _run(wsw, q, k, v, layout, scale):
    qd = q.cuda()
    if layout == "per_head":
        kd, vd = k.cuda(), v.cuda()
    else:  # position-major cache [depth][heads][dim], read through strides
        kd = k.permute(1, 0, 2).contiguous().cuda().permute(1, 0, 2)
        vd = v.permute(1, 0, 2).contiguous().cuda().permute(1, 0, 2)
    out = wsw.attn_prefill_f16(qd, kd, vd, scale)
    torch.cuda.synchronize()
    return out.cpu().double().numpy()


def _check_all(orc, q, k, v, got, scale, what):
    qb, kb, vb = f16_bits(q), f16_bits(k), f16_bits(v)
    ref = orc.attn_prefill(qb, kb, vb, scale)
    heads, group, nq, _ = q.shape
    depth = k.shape[1]
    qf = qb.view(np.float16).astype(np.float64)
    for h in range(heads):
        for g in range(group):
            for i in range(nq):
                vis = depth - nq + i + 1
                mag = _magnitude_row(qf[h, g, i], kb[h, :vis], vb[h, :vis], scale)
                _check_row(got[h, g, i], ref[h, g, i], mag, "%s h%d g%d i%d" % (what, h, g, i))


@pytest.mark.parametrize("layout", ["per_head", "position_major"])
@pytest.mark.parametrize("heads,group,nq,depth", [(2, 3, 300, 1000), (1, 2, 128, 128), (2, 1, 1, 517),
                                                  (1, 1, 257, 640), (3, 2, 70, 9000)])
def test_small_cases_every_row(orc, layout, heads, group, nq, depth):
    wsw = need_gpu()
    q, k, v = _inputs(1, heads, group, nq, depth)
    scale = 1.0 / math.sqrt(128)
    got = _run(wsw, q, k, v, layout, scale)
    _check_all(orc, q, k, v, got, scale, "%s %dx%dx%d d%d" % (layout, heads, group, nq, depth))


def test_layouts_are_bit_identical():
    wsw = need_gpu()
    q, k, v = _inputs(2, 2, 2, 200, 1500)
    a = _run(wsw, q, k, v, "per_head", 0.09)
    b = _run(wsw, q, k, v, "position_major", 0.09)
    assert np.array_equal(a, b)


def test_large_scores_raise_the_running_maximum(orc):
    """Peaked scores (q scaled by 6): a row's maximum moves by far more than the lazy
    headroom over the tiles, so O and l are rescaled mid-row."""
    wsw = need_gpu()
    q, k, v = _inputs(3, 1, 2, 256, 2000, qsigma=6.0)
    scale = 1.0 / math.sqrt(128)
    got = _run(wsw, q, k, v, "per_head", scale)
    _check_all(orc, q, k, v, got, scale, "large scores")


def test_dequant_then_attend(orc):
    """The page's pipeline: a q8_0 cache dequantized once into the per-head binary16
    scratch, then the prefill pass over it."""
    wsw = need_gpu()
    heads, group, nq, depth = 2, 2, 150, 1100
    kv = syn.normal(4, "pkv", (2, depth * heads, 128), dtype=torch.float16).float().numpy()
    scratch = []
    for t in range(2):
        kq, kd = orc.quantize_q8(kv[t], 32)
        kq, kd = kq.reshape(depth, heads, 128), kd.reshape(depth, heads, 4)
        out = wsw.dequant_q8_0_kv(torch.from_numpy(kq).cuda(), u16_to_torch(kd, torch.float16).cuda())
        assert (f16_bits(out) == orc.dequant_q8_0_kv(kq, kd)).all()
        scratch.append(out)
    q = syn.normal(4, "pq_dq", (heads, group, nq, 128), dtype=torch.float16)
    scale = 1.0 / math.sqrt(128)
    got = wsw.attn_prefill_f16(q.cuda(), scratch[0], scratch[1], scale)
    torch.cuda.synchronize()
    _check_all(orc, q, scratch[0].cpu(), scratch[1].cpu(), got.cpu().double().numpy(), scale, "dequant then attend")


@pytest.mark.parametrize("depth", [32768, 65536])
@pytest.mark.parametrize("layout", ["per_head", "position_major"])
def test_config_depths_sampled_queries(orc, depth, layout):
    """4 KV heads x 8 query heads, 512 queries at the end of the cache; every query head
    is checked at queries on both sides of every tile boundary."""
    wsw = need_gpu()
    heads, group, nq = 4, 8, 512
    q, k, v = _inputs(5, heads, group, nq, depth)
    scale = 1.0 / math.sqrt(128)
    got = _run(wsw, q, k, v, layout, scale)
    qb, kb, vb = f16_bits(q), f16_bits(k), f16_bits(v)
    qf = qb.view(np.float16).astype(np.float64)
    for h in range(heads):
        for g in range(group):
            for i in (0, 1, 127, 128, 255, 256, 383, 384, 510, 511):
                vis = depth - nq + i + 1
                ref = orc.attn_prefill(np.ascontiguousarray(qb[h:h + 1, g:g + 1, i:i + 1]),
                                       np.ascontiguousarray(kb[h:h + 1, :vis]),
                                       np.ascontiguousarray(vb[h:h + 1, :vis]), scale)[0, 0, 0]
                mag = _magnitude_row(qf[h, g, i], kb[h, :vis], vb[h, :vis], scale)
                _check_row(got[h, g, i], ref, mag, "d%d %s h%d g%d i%d" % (depth, layout, h, g, i))


# ----------------------------------------------------------- windowed q8_0 pass --

def _q8_cache(orc, seed, heads, depth):
    """A q8_0 K or V cache [depth][heads][128] (+ scales) quantized by the oracle from
    N(0, 1) binary16 values, and its dequantized per-head binary16 form (the oracle's)."""
    x = syn.normal(seed, "q8kv%d_%d" % (heads, depth), (depth * heads, 128), dtype=torch.float16).float().numpy()
    q, d = orc.quantize_q8(x, 32)
    q, d = q.reshape(depth, heads, 128), d.reshape(depth, heads, 4)
    return q, d, orc.dequant_q8_0_kv(q, d)


def _run_windowed(wsw, orc, seed, heads, group, nq, depth, window, qsigma=1.0):
    kq, kd, kb = _q8_cache(orc, seed, heads, depth)
    vq, vd, vb = _q8_cache(orc, seed + 1, heads, depth)
    q = syn.normal(seed, "wq%d_%d_%d" % (heads, group, nq), (heads, group, nq, 128), qsigma, torch.float16)
    scale = 1.0 / math.sqrt(128)
    got = wsw.attn_prefill_q8_0(q.cuda(), torch.from_numpy(kq).cuda(), u16_to_torch(kd, torch.float16).cuda(),
                                torch.from_numpy(vq).cuda(), u16_to_torch(vd, torch.float16).cuda(), window, scale)
    torch.cuda.synchronize()
    return q, kb, vb, got.cpu().double().numpy(), scale


@pytest.mark.parametrize("heads,group,nq,depth,window", [
    (2, 2, 300, 1000, 256),   # four windows, the last one short
    (1, 2, 600, 700, 128),    # windows past the limit of early query tiles
    (2, 1, 100, 900, 1024),   # one window: no carried state
    (1, 1, 1, 777, 384)])     # a single query
def test_windowed_q8_0_every_row(orc, heads, group, nq, depth, window):
    """Dequantize-and-attend one window at a time against the oracle's attention over the
    oracle's dequantized cache."""
    wsw = need_gpu()
    q, kb, vb, got, scale = _run_windowed(wsw, orc, 7, heads, group, nq, depth, window)
    _check_all(orc, q, torch.from_numpy(kb.view(np.int16)).view(torch.float16),
               torch.from_numpy(vb.view(np.int16)).view(torch.float16), got, scale, "windowed w%d" % window)


def test_windowed_q8_0_large_scores(orc):
    """Peaked scores: the carried maximum is raised in later windows."""
    wsw = need_gpu()
    q, kb, vb, got, scale = _run_windowed(wsw, orc, 8, 1, 2, 200, 1500, 256, qsigma=6.0)
    _check_all(orc, q, torch.from_numpy(kb.view(np.int16)).view(torch.float16),
               torch.from_numpy(vb.view(np.int16)).view(torch.float16), got, scale, "windowed large scores")


@pytest.mark.parametrize("depth,window", [(32768, 4096), (65536, 8192)])
def test_windowed_q8_0_config_depths_sampled_queries(orc, depth, window):
    """The configured cache (4 KV heads, 8 query heads each, 512 queries) through a scratch
    of one window, checked on sampled queries of every query head."""
    wsw = need_gpu()
    heads, group, nq = 4, 8, 512
    q, kb, vb, got, scale = _run_windowed(wsw, orc, 9, heads, group, nq, depth, window)
    qb = f16_bits(q)
    qf = qb.view(np.float16).astype(np.float64)
    for h in range(heads):
        for g in range(group):
            for i in (0, 127, 128, 384, 511):
                vis = depth - nq + i + 1
                ref = orc.attn_prefill(np.ascontiguousarray(qb[h:h + 1, g:g + 1, i:i + 1]),
                                       np.ascontiguousarray(kb[h:h + 1, :vis]),
                                       np.ascontiguousarray(vb[h:h + 1, :vis]), scale)[0, 0, 0]
                mag = _magnitude_row(qf[h, g, i], kb[h, :vis], vb[h, :vis], scale)
                _check_row(got[h, g, i], ref, mag, "windowed d%d w%d h%d g%d i%d" % (depth, window, h, g, i))
