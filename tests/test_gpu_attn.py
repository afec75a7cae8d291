"""Decode attention on the GPU (the consumer of the dequantized binary16 KV) against the
fp64 oracle: tolerance 1e-4, normwise per output row and per element against the
weighted magnitude of the values; both layouts of the page's strides, every group size,
ragged depths, large scores, padded rows, and the dequant-then-attend pipeline."""
import math

import numpy as np
import pytest
import torch

from helpers import f16_bits, need_gpu, u16_to_torch
from weight_streaming_warp_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

TOL = 1e-4


def _inputs(seed, heads, group, depth, hd=128, qsigma=1.0):
    q = syn.normal(seed, "q%d_%d_%d" % (heads, group, depth), (heads, group, hd), qsigma)
    k = syn.normal(seed, "k%d_%d" % (heads, depth), (heads, depth, hd), dtype=torch.float16)
    v = syn.normal(seed, "v%d_%d" % (heads, depth), (heads, depth, hd), dtype=torch.float16)
    return q, k, v


def _magnitude(q, kb, vb, scale):
    """sum_p w_p |v_p| / sum_p w_p per (head, query, dim), in fp64 (the bound for the
    per-element check)."""
    kf = kb.view(np.float16).astype(np.float64)
    vf = np.abs(vb.view(np.float16).astype(np.float64))
    s = np.einsum("hgi,hpi->hgp", q.astype(np.float64), kf) * scale
    w = np.exp(s - s.max(axis=2, keepdims=True))
    return np.einsum("hgp,hpi->hgi", w, vf) / w.sum(axis=2, keepdims=True)


def _check(got, ref, mag, what):
    got = got.cpu().double().numpy()
    assert np.isfinite(got).all(), what
    for h in range(ref.shape[0]):
        for g in range(ref.shape[1]):
            rel = np.linalg.norm(got[h, g] - ref[h, g]) / np.linalg.norm(ref[h, g])
            assert rel <= TOL, "%s head %d query %d: %.3g" % (what, h, g, rel)
    assert (np.abs(got - ref) <= TOL * mag + 1e-30).all(), what


def _run_both_layouts(wsw, orc, q, k, v, scale, what, opts=None):
    kb, vb = f16_bits(k), f16_bits(v)
    ref = orc.attn_decode(q.numpy(), kb, vb, scale)
    mag = _magnitude(q.numpy(), kb, vb, scale)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    a = wsw.attn_decode_f16(qd, kd, vd, scale=scale, opts=opts)  # per-head scratch
    _check(a, ref, mag, what + " per-head")
    kc = kd.permute(1, 0, 2).contiguous()  # the position-major cache [depth][heads][dim]
    vc = vd.permute(1, 0, 2).contiguous()
    b = wsw.attn_decode_f16(qd, kc.permute(1, 0, 2), vc.permute(1, 0, 2), scale=scale, opts=opts)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32)), what + ": the layouts differ"
    return a


@pytest.mark.parametrize("depth", [32768, 65536])
@pytest.mark.parametrize("group", [1, 2, 4, 8])  # both forms: CUDA cores (1, 2), tensor cores (4, 8)
def test_config_depths(orc, depth, group):
    wsw = need_gpu()
    q, k, v = _inputs(0, 4, group, depth)
    _run_both_layouts(wsw, orc, q, k, v, 1 / math.sqrt(128), "depth %d group %d" % (depth, group))


@pytest.mark.parametrize("depth", [1, 2, 63, 64, 65, 1000, 4097])
@pytest.mark.parametrize("heads,group", [(1, 1), (4, 2), (3, 4), (2, 8)])
def test_ragged_depths_and_groups(orc, depth, heads, group):
    wsw = need_gpu()
    q, k, v = _inputs(1, heads, group, depth)
    _run_both_layouts(wsw, orc, q, k, v, 0.09, "depth %d heads %d group %d" % (depth, heads, group))


def test_large_scores_stay_finite_and_accurate(orc):
    wsw = need_gpu()
    q, k, v = _inputs(2, 4, 4, 3000, qsigma=30.0)  # scores of several hundred
    _run_both_layouts(wsw, orc, q, k, v, 1 / math.sqrt(128), "large scores")


def test_launch_options_change_no_bit(orc):
    wsw = need_gpu()
    q, k, v = _inputs(3, 4, 8, 5000)
    a = _run_both_layouts(wsw, orc, q, k, v, 0.1, "default")
    for opts in ({"pdl": 1}, {"ctas_per_sm": 1}):
        b = wsw.attn_decode_f16(q.cuda(), k.cuda(), v.cuda(), scale=0.1, opts=opts)
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), opts


def test_padded_rows_and_heads(orc):
    wsw = need_gpu()
    heads, group, depth = 4, 2, 777
    q, k, v = _inputs(4, heads, group, depth)
    ref = orc.attn_decode(q.numpy(), f16_bits(k), f16_bits(v), 0.1)
    mag = _magnitude(q.numpy(), f16_bits(k), f16_bits(v), 0.1)
    # rows 136 elements apart (one 16-byte pad) and a gap of 8 rows between heads
    buf_k = torch.full((heads, depth + 8, 136), float("nan"), dtype=torch.float16, device="cuda")
    buf_v = torch.full((heads, depth + 8, 136), float("nan"), dtype=torch.float16, device="cuda")
    buf_k[:, :depth, :128] = k.cuda()
    buf_v[:, :depth, :128] = v.cuda()
    got = wsw.attn_decode_f16(q.cuda(), buf_k[:, :depth, :128], buf_v[:, :depth, :128], scale=0.1)
    _check(got, ref, mag, "padded")


def test_dequant_then_attend(orc):
    """The page's pipeline: a q8_0 KV cache dequantized once to the per-head f16
    scratch, then read by the attention step."""
    wsw = need_gpu()
    depth, heads, hd, group = 4096, 4, 128, 8
    raw = syn.normal(5, "kvraw", (2, depth * heads, hd), dtype=torch.float16).float().numpy()
    qk, dk = orc.quantize_q8(raw[0], 32)
    qv, dv = orc.quantize_q8(raw[1], 32)
    qk, dk = qk.reshape(depth, heads, hd), dk.reshape(depth, heads, hd // 32)
    qv, dv = qv.reshape(depth, heads, hd), dv.reshape(depth, heads, hd // 32)
    ks = wsw.dequant_q8_0_kv(torch.from_numpy(qk).cuda(), u16_to_torch(dk, torch.float16).cuda())
    vs = wsw.dequant_q8_0_kv(torch.from_numpy(qv).cuda(), u16_to_torch(dv, torch.float16).cuda())
    q = syn.normal(5, "qpipe", (heads, group, hd))
    got = wsw.attn_decode_f16(q.cuda(), ks, vs, opts={"pdl": 1})
    kb, vb = orc.dequant_q8_0_kv(qk, dk), orc.dequant_q8_0_kv(qv, dv)
    ref = orc.attn_decode(q.numpy(), kb, vb, 1 / math.sqrt(hd))
    _check(got, ref, _magnitude(q.numpy(), kb, vb, 1 / math.sqrt(hd)), "dequant then attend")


def test_workspace_reused_across_shapes_and_left_zeroed(orc):
    """One zero-filled workspace serves calls of different shapes in turn: the last
    chunk of each head merges, then sets its arrival counter back to zero, and repeated
    calls give the same bits whichever CTA merged."""
    wsw = need_gpu()
    shapes = [(4, 1, 5000), (2, 8, 777), (1, 2, 64), (3, 4, 20000), (4, 1, 5000)]
    ws = torch.zeros(max(wsw.attn_decode_workspace_bytes(d, h, g) for h, g, d in shapes), dtype=torch.uint8,
                     device="cuda")
    for heads, group, depth in shapes:
        q, k, v = _inputs(6, heads, group, depth)
        kb, vb = f16_bits(k), f16_bits(v)
        ref = orc.attn_decode(q.numpy(), kb, vb, 0.1)
        mag = _magnitude(q.numpy(), kb, vb, 0.1)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        first = wsw.attn_decode_f16(qd, kd, vd, scale=0.1, ws=ws)
        _check(first, ref, mag, "shape %s" % ((heads, group, depth),))
        for _ in range(3):
            again = wsw.attn_decode_f16(qd, kd, vd, scale=0.1, ws=ws)
            assert torch.equal(first.view(torch.int32), again.view(torch.int32))
        torch.cuda.synchronize()
        assert int(ws[:4 * heads].view(torch.int32).abs().sum()) == 0, "counters left nonzero"
