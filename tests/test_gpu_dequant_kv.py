"""dequant_q8_0_kv on the GPU against the oracle, bit for bit."""
import numpy as np
import pytest
import torch

from helpers import f16_bits, need_gpu, u16_to_torch
from weight_streaming_warp_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _cache(orc, depth, heads, hd, seed=0):
    v = syn.normal(seed, "kv%d_%d_%d" % (depth, heads, hd), (depth * heads, hd), dtype=torch.float16)
    q, d = orc.quantize_q8(v.float().numpy(), 32)
    return q.reshape(depth, heads, hd), d.reshape(depth, heads, hd // 32)


def _check(wsw, orc, q, d, qdev=None, ddev=None, out=None):
    qdev = torch.from_numpy(q).cuda() if qdev is None else qdev
    ddev = u16_to_torch(d, torch.float16).cuda() if ddev is None else ddev
    o = wsw.dequant_q8_0_kv(qdev, ddev, out=out)
    ref = orc.dequant_q8_0_kv(q, d)
    got = f16_bits(o)
    assert got.shape == ref.shape and (got == ref).all()


@pytest.mark.parametrize("depth", [32768, 65536])
def test_config_depths(orc, depth):
    wsw = need_gpu()
    q, d = _cache(orc, depth, 4, 128)
    _check(wsw, orc, q, d)


@pytest.mark.parametrize("depth,heads,hd", [(1, 1, 32), (3, 4, 128), (7, 5, 96), (129, 2, 64), (1000, 8, 256)])
def test_ragged(orc, depth, heads, hd):
    wsw = need_gpu()
    q, d = _cache(orc, depth, heads, hd, seed=1)
    _check(wsw, orc, q, d)


def test_tags_land_per_head(orc):
    wsw = need_gpu()
    depth, heads, hd = 37, 4, 128
    p, h, i = np.meshgrid(np.arange(depth), np.arange(heads), np.arange(hd), indexing="ij")
    q = (((p * 7 + h * 31 + i * 3) % 255) - 127).astype(np.int8)
    d = np.full((depth, heads, hd // 32), 0x3C00, np.uint16)
    _check(wsw, orc, q, d)


def test_misaligned_buffers_take_the_element_path(orc):
    wsw = need_gpu()
    depth, heads, hd = 50, 4, 128
    q, d = _cache(orc, depth, heads, hd, seed=2)
    raw = torch.zeros(q.size + 1, dtype=torch.int8, device="cuda")
    qv = raw[1:].view(depth, heads, hd)
    qv.copy_(torch.from_numpy(q))
    outraw = torch.zeros(heads * depth * hd + 1, dtype=torch.float16, device="cuda")
    out = outraw[1:].view(heads, depth, hd)
    _check(wsw, orc, q, d, qdev=qv, out=out)


def test_rounding_and_extremes(orc):
    wsw = need_gpu()
    q = np.zeros((2, 1, 32), np.int8)
    d = np.zeros((2, 1, 1), np.uint16)
    q[0, 0, :6] = [3, 5, -3, 127, -127, 2]
    d[0, 0, 0] = 0x3C01  # 1 + 2^-10: products land on ties and near-ties
    q[1, 0, :3] = [127, 2, -1]
    d[1, 0, 0] = 0x7BFF  # 65504: overflow to inf
    _check(wsw, orc, q, d)
