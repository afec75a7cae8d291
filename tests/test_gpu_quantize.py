"""quantize_q8 on the GPU against the oracle: bit-exact q bytes and scale bits."""
import numpy as np
import pytest
import torch

from helpers import f16_bits, need_gpu
from weight_streaming_warp_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _compare(wsw, orc, x_host: torch.Tensor, block, xdev=None, opts=None):
    xdev = x_host.cuda() if xdev is None else xdev
    q, s = wsw.quantize_q8(xdev, block, opts=opts)
    torch.cuda.synchronize()
    xq = x_host.numpy() if x_host.dim() == 2 else x_host.numpy()[None, :]
    qr, sr = orc.quantize_q8(np.ascontiguousarray(xq), block)
    qg = q.cpu().numpy().reshape(qr.shape)
    assert (qg == qr).all(), "q differs at %s" % (np.argwhere(qg != qr)[:5],)
    if block == 32:
        sg = f16_bits(s).reshape(sr.shape)
    else:
        sg = s.cpu().numpy().reshape(sr.shape)
    assert (sg.view(np.uint32 if block == 256 else np.uint16) ==
            sr.view(np.uint32 if block == 256 else np.uint16)).all()
    return q, s


@pytest.mark.parametrize("block", [32, 256])
@pytest.mark.parametrize("rows,n", [(1, 4096), (1, 14336), (3, 512), (7, 768), (1, 256), (5, 2048)])
def test_quantize_matches_oracle(orc, block, rows, n):
    wsw = need_gpu()
    x = syn.normal(0, "q%d_%d" % (rows, n), (rows, n))
    _compare(wsw, orc, x, block)


@pytest.mark.parametrize("block", [32, 256])
def test_quantize_varied_block_scales(orc, block):
    """Blocks whose magnitudes span 1e-6 .. 1e4, zero blocks and single spikes."""
    wsw = need_gpu()
    nb = 64
    x = syn.normal(1, "v", (nb, block)).double()
    scale = 10.0 ** torch.linspace(-6, 4, nb, dtype=torch.float64)
    x = (x * scale[:, None]).float()
    x[3] = 0.0
    x[5] = 0.0
    x[5, 7] = -2.5
    x = x.reshape(1, nb * block)
    _compare(wsw, orc, x, block)


def test_quantize_ties_and_exact_grid(orc):
    wsw = need_gpu()
    x = torch.zeros(1, 64)
    x[0, 0] = 127.0
    x[0, 1:9] = torch.tensor([2.5, -2.5, 0.5, -0.5, 1.5, 126.5, -3.5, 0.49999997])
    k = torch.arange(-127, -95, dtype=torch.float32)
    x[0, 32:64] = k * 2.0 ** -7
    q, s = _compare(wsw, orc, x, 32)
    assert q[0, 1:9].tolist() == [3, -3, 1, -1, 2, 127, -4, 0]
    assert q[0, 32:64].tolist() == k.int().tolist()


def _near_tie_blocks(block, nblocks, seed):
    """Blocks whose first value is the amax and whose other values sit on, or a few
    ulps around, the half-integer multiples (n + 1/2) d of the block's scale
    d = fp32(amax / 127): the values where rounding v / d to an integer is decided in
    the last bits of the quotient."""
    rng = np.random.default_rng(seed)
    x = np.zeros((nblocks, block), np.float32)
    for b in range(nblocks):
        amax = np.float32(10.0 ** rng.uniform(-20, 20))
        d = np.float32(amax) / np.float32(127.0)
        n = rng.integers(-127, 127, block - 1)
        v = ((n + 0.5) * np.float64(d)).astype(np.float32)
        for k in range(block - 1):
            for _ in range(abs(int(rng.integers(-8, 9)))):
                v[k] = np.nextafter(v[k], np.float32(np.inf) if k % 2 else np.float32(-np.inf))
        v = np.clip(v, -amax, amax)
        x[b, 0] = amax if b % 2 else -amax
        x[b, 1:] = v
    return torch.from_numpy(x.reshape(1, -1))


@pytest.mark.parametrize("block", [32, 256])
def test_quantize_near_ties_against_oracle(orc, block):
    """Values on and around the rounding boundaries of x / d, over scales 1e-20 ..
    1e20: the codes equal the oracle's (exact fp32 division) bit for bit, in the
    quantizer and in the mat-vec that quantizes its own activation."""
    wsw = need_gpu()
    x = _near_tie_blocks(block, 4096 // block * 16, block)
    _compare(wsw, orc, x, block)
    if block == 32:
        n = x.shape[1]
        xr, dr = orc.quantize_q8(x.numpy(), 32)
        xq = torch.empty(n, dtype=torch.int8, device="cuda")
        xd = torch.empty(n // 32, dtype=torch.float16, device="cuda")
        Wq = torch.ones((8, n), dtype=torch.int8, device="cuda")
        Wd = torch.ones((8, n // 32), dtype=torch.float16, device="cuda")
        wsw.quantize_gemv_q8_0(Wq, Wd, x.cuda()[0], x_out=(xq, xd))
        assert (xq.cpu().numpy() == xr[0]).all() and (f16_bits(xd) == dr[0]).all()


@pytest.mark.parametrize("block", [32, 256])
def test_quantize_moe_batch_shape(orc, block):
    """T = 512 tokens x top_k 8 rows of the 2048-wide hidden state."""
    wsw = need_gpu()
    x = syn.normal(2, "moe", (4096, 2048))
    _compare(wsw, orc, x, block)


def test_quantize_strided_and_misaligned_rows(orc):
    wsw = need_gpu()
    for pad in (4, 1, 3):  # ldx = n + pad: vector path for 4, element path otherwise
        n = 256
        big = syn.normal(3, "s%d" % pad, (6, n + pad))
        xdev = big.cuda()[:, :n]
        _compare(wsw, orc, big[:, :n].contiguous(), 32, xdev=xdev)
    # base address not 16-byte aligned
    flat = syn.normal(3, "m", (1, 1 + 512))
    xdev = flat.cuda()[0, 1:]
    _compare(wsw, orc, flat[0, 1:].contiguous(), 256, xdev=xdev)


def test_quantize_launch_options_do_not_change_bits(orc):
    wsw = need_gpu()
    x = syn.normal(4, "o", (2, 4096)).cuda()
    ref = [t.clone() for t in wsw.quantize_q8(x, 32)]
    for opts in ({"pdl": 1}, {"ctas_per_sm": 1}, {"rows_per_warp": 4, "load_bytes": 2}):
        got = wsw.quantize_q8(x, 32, opts=opts)
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1].view(torch.int16), ref[1].view(torch.int16))


def test_quantize_empty_inputs():
    wsw = need_gpu()
    x = torch.empty((0, 64), device="cuda")
    q, s = wsw.quantize_q8(x, 32)
    assert q.numel() == 0 and s.numel() == 0
    x = torch.empty((3, 0), device="cuda")
    q, s = wsw.quantize_q8(x, 256)
    assert q.numel() == 0
    with pytest.raises(wsw.WswError):
        wsw.quantize_q8(torch.zeros(48, device="cuda"), 32)


@pytest.mark.parametrize("block", [32, 256])
def test_quantize_subnormal_blocks(orc, block):
    """Blocks of binary32 subnormals: an amax of 63 smallest steps makes amax / 127
    round to +0 (the block is stored as zero), 64 and 127 steps give d = 2^-149, and
    blocks of larger subnormals and of normal values sit beside them.  Bit-exact
    against the oracle, through the standalone quantizer and the fused mat-vec."""
    wsw = need_gpu()
    s = 2.0 ** -149
    rng = np.random.default_rng(5)
    rows = []
    for steps in (63, 64, 127, 1000, 2 ** 22, 2 ** 30):
        k = rng.integers(-min(steps, 2 ** 24), min(steps, 2 ** 24) + 1, size=block).astype(np.float64)
        k[rng.integers(block)] = steps
        rows.append((k * s).astype(np.float32))
    rows.append(np.zeros(block, np.float32))
    x = torch.from_numpy(np.concatenate(rows)[None, :])
    _compare(wsw, orc, x, block)
    if block == 32:
        K = x.shape[1]
        Wq = torch.ones((4, K), dtype=torch.int8, device="cuda")
        Wd = torch.ones((4, K // 32), dtype=torch.float16, device="cuda")
        xq = torch.empty(K, dtype=torch.int8, device="cuda")
        xd = torch.empty(K // 32, dtype=torch.float16, device="cuda")
        wsw.quantize_gemv_q8_0(Wq, Wd, x[0].cuda(), x_out=(xq, xd))
        torch.cuda.synchronize()
        qr, sr = orc.quantize_q8(x.numpy(), 32)
        assert (xq.cpu().numpy() == qr[0]).all() and (f16_bits(xd) == sr[0]).all()
