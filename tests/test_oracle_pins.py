"""Pins of the C oracle against facts that do not come from the oracle itself.

Each check is a closed form, an invariant, a special case that reduces to a
library routine (numpy's binary16 conversion, numpy's fp64 matmul), exact rational
arithmetic on tiny inputs, or a value printed on the source pages (tests/golden/).
They run without a GPU.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from weight_streaming_warp_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers --
def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split("=")
                vals[k.strip()] = [int(t) for t in v.split()]
    return vals


def fl32(r: Fraction) -> np.float32:
    """Correctly rounded (nearest, ties to even) binary32 of an exact rational."""
    if r == 0:
        return np.float32(0.0)
    f = np.float32(float(r))
    cands = {np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))}
    best = None
    for c in cands:
        dist = abs(Fraction(float(c)) - r)
        even = int(np.array(c, np.float32).view(np.uint32)) & 1 == 0
        key = (dist, not even)
        if best is None or key < best[0]:
            best = (key, c)
    return np.float32(best[1])


def round_half_away(r: Fraction) -> int:
    s = -1 if r < 0 else 1
    return s * math.floor(abs(r) + Fraction(1, 2))


def f16_bits(v) -> int:
    return int(np.array(v, np.float32).astype(np.float16).view(np.uint16))


def quantize_block_exact(xb):
    """The q8_0 rule evaluated with exact rationals and explicit binary32 rounding:
    amax = max|x|, d = fl32(amax / 127), q = round_half_away(fl32(x / d))."""
    amax = max(abs(Fraction(float(v))) for v in xb)
    if amax == 0:
        return [0] * len(xb), np.float32(0.0)
    d = fl32(amax / 127)
    q = []
    for v in xb:
        t = round_half_away(Fraction(float(fl32(Fraction(float(v)) / Fraction(float(d))))))
        q.append(max(-127, min(127, t)))
    return q, d


# ------------------------------------------------------- binary16 helpers --
def test_f16_from_f32_matches_numpy(orc):
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    # concentrate on half's range, its subnormals and the ties
    special = []
    for e in range(-26, 17):
        for m in (0, 1, 0x1000, 0x1001, 0x0fff, 0x2000, 0x7fffff, 0x3000):
            special.append(np.float32(np.ldexp(1.0 + m / 2**23, e)))
    special += [65504.0, 65519.99, 65520.0, 65536.0, 6.0e-8, 2.98e-8, 2.9802322e-8,
                5.9604645e-8, 8.940697e-8, 0.0, -0.0, np.inf, -np.inf]
    vals = np.concatenate([bits.view(np.float32), np.array(special, np.float32),
                           -np.array(special, np.float32)])
    vals = vals[np.isfinite(vals) | np.isinf(vals)]
    for v in vals:
        with np.errstate(over="ignore"):  # values past the binary16 range round to inf
            ref = int(np.array(v, np.float32).astype(np.float16).view(np.uint16))
        got = orc.f32_to_f16_bits(float(v))
        assert got == ref, (v, hex(got), hex(ref))


def test_f16_to_f32_exhaustive(orc):
    for h in range(0, 65536, 7):
        ref = np.array(h, np.uint16).view(np.float16).astype(np.float32)
        got = np.float32(orc.f16_bits_to_f32(h))
        if np.isnan(ref):
            assert np.isnan(got)
        else:
            assert got == ref and np.signbit(got) == np.signbit(ref), h


# ------------------------------------------------------------- quantizer --
def test_quantize_all_zero_block(orc):
    q, d = orc.quantize_q8(np.zeros((2, 64), np.float32), 32)
    assert not q.any() and not d.any()
    q, d = orc.quantize_q8(np.zeros((1, 256), np.float32), 256)
    assert not q.any() and d[0, 0] == 0.0


@pytest.mark.parametrize("block", [32, 256])
def test_quantize_subnormal_blocks(orc, block):
    """Blocks of binary32 subnormals, where d = fl(amax / 127) reaches the bottom of the
    range.  s = 2^-149 is the smallest subnormal.  amax = 63 s: amax / 127 < s / 2
    rounds to +0, and the block is stored as zero (x / 0 is undefined).  amax = 127 s:
    d = s exactly and q = x / s exactly.  amax = 64 s: amax / 127 is just above s / 2
    and rounds to d = s, so q = x / s (the amax value itself gives 64, not 127)."""
    s = np.float32(2.0 ** -149)
    rng = np.random.default_rng(11)
    for amax_steps, d_steps in ((63, 0), (127, 1), (64, 1)):
        k = rng.integers(-amax_steps, amax_steps + 1, size=block)
        k[rng.integers(block)] = -amax_steps if rng.integers(2) else amax_steps
        x = (k.astype(np.float32) * s).astype(np.float32)[None, :]
        assert (x[0] / s == k).all()  # the inputs are exact subnormal multiples
        q, d = orc.quantize_q8(x, block)
        if d_steps == 0:
            assert not q.any()
            assert (d == 0).all() and not np.signbit(d.astype(np.float32)).any()
        else:
            assert (q[0].astype(np.int64) == k).all()
            if block == 32:
                assert int(d[0, 0]) == 0  # binary16 has no subnormal this small: +0
            else:
                assert d[0, 0] == s


@pytest.mark.parametrize("block", [32, 256])
def test_quantize_single_nonzero(orc, block):
    for v in (1.0, -3.7, 1e-3, 250.0):
        for pos in (0, 5, block - 1):
            x = np.zeros((1, block), np.float32)
            x[0, pos] = v
            q, d = orc.quantize_q8(x, block)
            assert q[0, pos] == (127 if v > 0 else -127)
            assert np.count_nonzero(q) == 1
            d32 = fl32(Fraction(float(np.float32(abs(v)))) / 127)
            if block == 32:
                assert int(d[0, 0]) == f16_bits(d32)
            else:
                assert d[0, 0] == d32


@pytest.mark.parametrize("block", [32, 256])
def test_quantize_exact_grid(orc, block):
    """x = k * 2^e with amax = 127 * 2^e: d = 2^e exactly and q = k exactly."""
    rng = np.random.default_rng(2)
    for e in (-12, -3, 0, 4):
        k = rng.integers(-127, 128, size=block)
        k[rng.integers(0, block)] = -127
        x = (k * 2.0 ** e).astype(np.float32)[None, :]
        q, d = orc.quantize_q8(x, block)
        assert (q[0].astype(int) == k).all()
        if block == 32:
            assert int(d[0, 0]) == f16_bits(2.0 ** e)
        else:
            assert d[0, 0] == np.float32(2.0 ** e)


def test_quantize_ties_round_away_from_zero(orc):
    """amax = 127 gives d = 1 exactly, so x/d = x: halves round away from zero."""
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 127.0
    x[0, 1:9] = [2.5, -2.5, 0.5, -0.5, 1.5, 126.5, -3.5, 0.49999997]
    q, d = orc.quantize_q8(x, 32)
    assert list(q[0, :9]) == [127, 3, -3, 1, -1, 2, 127, -4, 0]
    assert int(d[0, 0]) == 0x3C00  # 1.0


def test_quantize_divides_by_fp32_scale_not_fp16(orc):
    """Find a block where q computed with the stored fp16 scale would differ; the
    oracle must follow the fp32 scale."""
    amax = np.float32(100.0)
    d32 = fl32(Fraction(float(amax)) / 127)
    d16 = np.float32(np.float16(d32))
    assert d16 != d32
    found = None
    for k in range(1, 127):
        # just below the k + 1/2 boundary measured with d32
        target = Fraction(float(d32)) * (Fraction(2 * k + 1, 2))
        x = fl32(target)
        for cand in (x, np.nextafter(x, np.float32(0)), np.nextafter(x, np.float32(np.inf))):
            q32 = round_half_away(Fraction(float(fl32(Fraction(float(cand)) / Fraction(float(d32))))))
            q16 = round_half_away(Fraction(float(fl32(Fraction(float(cand)) / Fraction(float(d16))))))
            if q32 != q16:
                found = (cand, q32)
                break
        if found:
            break
    assert found is not None
    xb = np.zeros((1, 32), np.float32)
    xb[0, 0] = amax
    xb[0, 1] = found[0]
    q, _ = orc.quantize_q8(xb, 32)
    assert q[0, 1] == found[1]


def test_quantize_divides_rather_than_multiplying_by_reciprocal(orc):
    """Search a block where round(x / d) and round(x * fl32(1/d)) differ; the
    oracle must take the quotient."""
    rng = np.random.default_rng(11)
    found = None
    for _ in range(4000):
        amax = np.float32(rng.uniform(0.5, 2.0))
        d = fl32(Fraction(float(amax)) / 127)
        rcp = fl32(1 / Fraction(float(d)))
        k = int(rng.integers(1, 127))
        x0 = fl32(Fraction(float(d)) * Fraction(2 * k + 1, 2))
        for cand in (x0, np.nextafter(x0, np.float32(0)), np.nextafter(x0, np.float32(np.inf))):
            if abs(cand) > amax:
                continue
            qa = round_half_away(Fraction(float(fl32(Fraction(float(cand)) / Fraction(float(d))))))
            qb = round_half_away(Fraction(float(fl32(Fraction(float(cand)) * Fraction(float(rcp))))))
            if qa != qb:
                found = (amax, cand, qa)
                break
        if found:
            break
    assert found is not None
    xb = np.zeros((1, 32), np.float32)
    xb[0, 0], xb[0, 1] = found[0], found[1]
    q, _ = orc.quantize_q8(xb, 32)
    assert q[0, 1] == found[2]


@pytest.mark.parametrize("block", [32, 256])
def test_quantize_brute_force_exact_rationals(orc, block):
    """Random blocks across scales against the rule evaluated with exact rationals."""
    rng = np.random.default_rng(3)
    nblk = 24 if block == 32 else 4
    x = (rng.standard_normal((1, nblk * block)) *
         np.repeat(10.0 ** rng.uniform(-4, 3, nblk), block)).astype(np.float32)
    # ties and near-ties: put exact multiples of half-steps into some blocks
    x[0, 3] = np.float32(0.0)
    q, d = orc.quantize_q8(x, block)
    for b in range(nblk):
        xb = x[0, b * block:(b + 1) * block]
        qe, de = quantize_block_exact(xb)
        assert list(q[0, b * block:(b + 1) * block].astype(int)) == qe
        if block == 32:
            assert int(d[0, b]) == f16_bits(de)
        else:
            assert d[0, b] == de


def test_superblock_scale_is_max_of_block_scales(orc):
    """fp16 rounding and x -> x/127 are monotone, so the superblock's scale equals
    the largest of its eight q8_0 block scales (after rounding both to fp16)."""
    x = syn.normal(0, "sb", (3, 256 * 4)).numpy()
    _, d32 = orc.quantize_q8(x, 32)
    _, d256 = orc.quantize_q8(x, 256)
    for r in range(3):
        for s in range(4):
            sub = d32[r, 8 * s:8 * s + 8].view(np.float16).astype(np.float32)
            assert f16_bits(d256[r, s]) == f16_bits(sub.max())


def test_superblock_count_from_page(orc):
    g = _read_golden("superblock_count_p3.txt")
    x = syn.normal(0, "x", (1, g["hidden"][0])).numpy()
    q, d = orc.quantize_q8(x, g["superblock"][0])
    assert d.shape == (1, g["superblocks"][0]) and q.shape == (1, g["hidden"][0])


@pytest.mark.parametrize("block", [32, 256])
def test_quantize_error_bound_and_range(orc, block):
    x = syn.normal(7, "e", (4, 2048), sigma=3.0).numpy()
    q, d = orc.quantize_q8(x, block)
    d = d.view(np.float16).astype(np.float64) if block == 32 else d.astype(np.float64)
    assert np.abs(q).max() <= 127
    qb = q.reshape(4, -1, block)
    assert (np.abs(qb).max(axis=2) == 127).all()
    # with the exact scale a/127 each element is within half a step (plus fp32 slack)
    amax = np.abs(x.reshape(4, -1, block)).max(axis=2, keepdims=True).astype(np.float64)
    err = np.abs(qb * (amax / 127) - x.reshape(4, -1, block))
    assert (err <= (amax / 127) * (0.5 + 1e-5)).all()


def test_quantize_row_stride_skips_padding(orc):
    x = np.full((3, 96), np.nan, np.float32)
    x[:, :64] = syn.normal(0, "p", (3, 64)).numpy()
    q1, d1 = orc.quantize_q8(x, 32, n=64)
    q2, d2 = orc.quantize_q8(np.ascontiguousarray(x[:, :64]), 32)
    assert (q1 == q2).all() and (d1 == d2).all()


# ------------------------------------------------------------- gemv bf16 --
def _bf16_bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bits_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_gemv_bf16_one_hot_picks_a_column(orc):
    W = _bf16_bits(syn.normal(0, "W", (37, 48), 0.02).numpy())
    for k in (0, 5, 47):
        x = np.zeros(48)
        x[k] = 1.0
        y = orc.gemv_bf16(W, x)
        assert (y == _bits_to_f64(W[:, k])).all()


def test_gemv_bf16_small_integers_exact(orc):
    rng = np.random.default_rng(4)
    Wi = rng.integers(-8, 9, size=(19, 70))
    xi = rng.integers(-5, 6, size=70)
    y = orc.gemv_bf16(_bf16_bits(Wi), xi.astype(np.float64))
    assert (y == (Wi @ xi).astype(np.float64)).all()
    y2 = orc.gemv_bf16(_bf16_bits(Wi), xi.astype(np.float64), alpha=0.25)
    assert (y2 == 0.25 * (Wi @ xi)).all()


def test_gemv_bf16_brute_force_rational(orc):
    for (M, K) in ((1, 1), (3, 7), (5, 33), (8, 64)):
        W = _bf16_bits(syn.normal(1, "W%d" % K, (M, K), 0.5).numpy())
        x = syn.normal(1, "x%d" % K, (K,)).numpy().astype(np.float64)
        y = orc.gemv_bf16(W, x, alpha=1.5)
        Wf = _bits_to_f64(W)
        for r in range(M):
            exact = Fraction(3, 2) * sum(Fraction(float(Wf[r, k])) * Fraction(float(x[k])) for k in range(K))
            mag = sum(abs(Wf[r, k] * x[k]) for k in range(K)) * 1.5
            assert abs(float(Fraction(float(y[r])) - exact)) <= (K + 2) * 2.0 ** -52 * mag + 1e-300


def test_gemv_bf16_padded_row_stride(orc):
    M, K, ld = 9, 40, 64
    Wp = np.full((M, ld), 0x7FC0, np.uint16)  # bf16 NaN in the pad
    Wp[:, :K] = _bf16_bits(syn.normal(0, "W", (M, K), 0.02).numpy())
    x = syn.normal(0, "x", (K,)).numpy()
    y_pad = orc.gemv_bf16(Wp, x, K=K)
    y_packed = orc.gemv_bf16(np.ascontiguousarray(Wp[:, :K]), x)
    assert np.isfinite(y_pad).all() and (y_pad == y_packed).all()


# ------------------------------------------------------------- gemv q8_0 --
def test_gemv_q8_0_power_of_two_scales_exact(orc):
    Wq = np.ones((2, 64), np.int8)
    Wq[1, :] = -2
    xq = np.arange(1, 65, dtype=np.int8)
    Wd = np.array([[f16_bits(2.0 ** -3), f16_bits(2.0 ** -1)],
                   [f16_bits(2.0 ** 2), f16_bits(1.0)]], np.uint16)
    xd = np.array([f16_bits(2.0 ** -2), f16_bits(2.0 ** -4)], np.uint16)
    y = orc.gemv_q8_0(Wq, Wd, xq, xd)
    s0, s1 = sum(range(1, 33)), sum(range(33, 65))  # 528, 1552
    assert y[0] == s0 * 2.0 ** -5 + s1 * 2.0 ** -5
    assert y[1] == -2 * s0 * 2.0 ** 0 + -2 * s1 * 2.0 ** -4


def test_gemv_q8_0_brute_force_rational(orc):
    rng = np.random.default_rng(5)
    for (M, K) in ((1, 32), (4, 96), (3, 256)):
        Wq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
        xq = rng.integers(-127, 128, size=K).astype(np.int8)
        Wd = np.array([f16_bits(v) for v in rng.uniform(1e-4, 1e-2, M * K // 32)], np.uint16).reshape(M, K // 32)
        xd = np.array([f16_bits(v) for v in rng.uniform(1e-3, 5e-2, K // 32)], np.uint16)
        y = orc.gemv_q8_0(Wq, Wd, xq, xd)
        wdf = Wd.view(np.float16).astype(np.float64)
        xdf = xd.view(np.float16).astype(np.float64)
        for r in range(M):
            exact = sum(Fraction(float(wdf[r, b])) * Fraction(float(xdf[b])) *
                        sum(int(Wq[r, 32 * b + i]) * int(xq[32 * b + i]) for i in range(32))
                        for b in range(K // 32))
            mag = sum(abs(float(wdf[r, b] * xdf[b])) * 32 * 127 * 127 for b in range(K // 32))
            assert abs(float(Fraction(float(y[r])) - exact)) <= (K // 32 + 1) * 2.0 ** -52 * mag


def test_gemv_q8_0_equals_dequantized_dot(orc):
    """Library check: numpy fp64 matmul on the dequantized operands."""
    W = syn.normal(0, "W", (64, 512), 0.02).numpy()
    x = syn.normal(0, "x", (1, 512)).numpy()
    Wq, Wd = orc.quantize_q8(W, 32)
    xq, xd = orc.quantize_q8(x, 32)
    y = orc.gemv_q8_0(Wq, Wd, xq[0], xd[0])
    Wdq = Wq.astype(np.float64) * np.repeat(Wd.view(np.float16).astype(np.float64), 32, axis=1)
    xdq = xq[0].astype(np.float64) * np.repeat(xd[0].view(np.float16).astype(np.float64), 32)
    ref = Wdq @ xdq
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)


def test_gemv_q8_0_row_stride(orc):
    rng = np.random.default_rng(6)
    Wq = rng.integers(-127, 128, size=(5, 96)).astype(np.int8)
    Wd = rng.integers(0x1000, 0x2000, size=(5, 2)).astype(np.uint16)
    xq = rng.integers(-127, 128, size=64).astype(np.int8)
    xd = rng.integers(0x1000, 0x2000, size=2).astype(np.uint16)
    y_pad = orc.gemv_q8_0(Wq, Wd, xq, xd, K=64)
    y_packed = orc.gemv_q8_0(np.ascontiguousarray(Wq[:, :64]), Wd, xq, xd)
    assert (y_pad == y_packed).all()


# ------------------------------------------------------------------- moe --
def test_moe_reduces_to_per_expert_gemv(orc):
    rng = np.random.default_rng(7)
    E, Mo, K, T, topk = 6, 16, 64, 5, 2
    Wq = rng.integers(-127, 128, size=(E, Mo, K)).astype(np.int8)
    Wd = rng.integers(0x0800, 0x2000, size=(E, Mo, K // 32)).astype(np.uint16)
    ids = syn.routing(0, "r", T, E, topk).numpy()
    R = T * topk
    xq = rng.integers(-127, 128, size=(R, K)).astype(np.int8)
    xd = rng.integers(0x0800, 0x2000, size=(R, K // 32)).astype(np.uint16)
    y, bad = orc.moe_gemv_q8_0(Wq, Wd, xq, xd, ids)
    assert bad == 0
    for m in range(R):
        ref = orc.gemv_q8_0(Wq[ids[m]], Wd[ids[m]], xq[m], xd[m])
        assert (y[m] == ref).all()
    # permuting the rows permutes the output exactly
    perm = rng.permutation(R)
    yp, _ = orc.moe_gemv_q8_0(Wq, Wd, xq[perm], xd[perm], ids[perm])
    assert (yp == y[perm]).all()


def test_moe_bad_ids_are_skipped(orc):
    rng = np.random.default_rng(8)
    E, Mo, K = 3, 4, 32
    Wq = rng.integers(-127, 128, size=(E, Mo, K)).astype(np.int8)
    Wd = rng.integers(0x0800, 0x2000, size=(E, Mo, 1)).astype(np.uint16)
    xq = rng.integers(-127, 128, size=(4, K)).astype(np.int8)
    xd = rng.integers(0x0800, 0x2000, size=(4, 1)).astype(np.uint16)
    ids = np.array([0, 3, -1, 2], np.int32)
    y, bad = orc.moe_gemv_q8_0(Wq, Wd, xq, xd, ids, y_init=np.full((4, Mo), 7.0))
    assert bad == 2
    assert (y[1] == 7.0).all() and (y[2] == 7.0).all()
    assert (y[3] == orc.gemv_q8_0(Wq[2], Wd[2], xq[3], xd[3])).all()


def test_routing_draws_distinct_experts():
    ids = syn.routing(0, "ids", 64, 128, 8).numpy().reshape(64, 8)
    for t in range(64):
        assert len(set(ids[t])) == 8 and ids[t].min() >= 0 and ids[t].max() < 128


# ------------------------------------------------------------------ gemm --
def test_gemm_bf16_matches_numpy(orc):
    W = _bf16_bits(syn.normal(0, "W", (24, 80), 0.02).numpy())
    X = _bf16_bits(syn.normal(0, "X", (9, 80)).numpy())
    Y = orc.gemm_bf16(W, X)
    ref = _bits_to_f64(X) @ _bits_to_f64(W).T
    assert np.allclose(Y, ref, rtol=1e-13, atol=1e-15)


def test_gemm_bf16_strides(orc):
    M, K, N = 6, 40, 3
    W = np.full((M, 72), 0x7FC0, np.uint16)
    X = np.full((N, 48), 0x7FC0, np.uint16)
    W[:, :K] = _bf16_bits(syn.normal(0, "W", (M, K), 0.02).numpy())
    X[:, :K] = _bf16_bits(syn.normal(0, "X", (N, K)).numpy())
    Y = orc.gemm_bf16(W, X, K=K)
    Yp = orc.gemm_bf16(np.ascontiguousarray(W[:, :K]), np.ascontiguousarray(X[:, :K]))
    assert np.isfinite(Y).all() and (Y == Yp).all()


def test_gemm_column_is_gemv(orc):
    W = _bf16_bits(syn.normal(0, "W", (10, 64), 0.02).numpy())
    X = _bf16_bits(syn.normal(0, "X", (3, 64)).numpy())
    Y = orc.gemm_bf16(W, X)
    for n in range(3):
        assert (Y[n] == orc.gemv_bf16(W, _bits_to_f64(X[n]))).all()


# ------------------------------------------------------------ kv dequant --
def test_kv_dequant_layout_tags(orc):
    """d = 1 and q = a tag of (p, h, i): the output must hold each tag at
    out[h][p][i] (integers up to 127 are exact in binary16)."""
    depth, heads, hd = 11, 4, 128
    p, h, i = np.meshgrid(np.arange(depth), np.arange(heads), np.arange(hd), indexing="ij")
    q = (((p * 7 + h * 31 + i * 3) % 255) - 127).astype(np.int8)
    d = np.full((depth, heads, hd // 32), 0x3C00, np.uint16)
    out = orc.dequant_q8_0_kv(q, d)
    assert out.shape == (heads, depth, hd)
    ref = np.transpose(q, (1, 0, 2)).astype(np.float16).view(np.uint16)
    assert (out == ref).all()


def test_kv_dequant_rounding_cases(orc):
    """Hand-derived binary16 results of one product each.
    1.0009765625 (1 + 2^-10) * 3 = 3.0029296875 = 3 + 1.5 ulp(2^-9): tie -> even -> 3.00390625.
    1.0009765625 * 5 = 5.0048828125 = 5 + 1.25 ulp(2^-8 at [4, 8)): -> 5 + 2^-8 = 5.00390625.
    2^-14 * 3 = 3 * 2^-14: a normal number, exact.
    2^-24 (smallest subnormal scale) * 127: exact subnormal 127 * 2^-24.
    65504 * 2 = 131008 overflows binary16 -> +inf."""
    cases = [(0x3C01, 3, 3.00390625), (0x3C01, 5, 5.00390625), (0x0400, 3, 3 * 2.0 ** -14),
             (0x0001, 127, 127 * 2.0 ** -24), (0x7BFF, 2, np.inf), (0x3C01, -3, -3.00390625)]
    for (dbits, qv, expect) in cases:
        q = np.zeros((1, 1, 32), np.int8)
        q[0, 0, 0] = qv
        d = np.array([[[dbits]]], np.uint16)
        out = orc.dequant_q8_0_kv(q, d)
        got = np.array(out[0, 0, 0], np.uint16).view(np.float16).astype(np.float64)
        assert got == expect, (hex(dbits), qv, got, expect)


def test_kv_layout_matches_page_strides():
    """The oracle's input walk [pos][head][dim] is the page's f16 K tensor
    ne = [HS, KV, n_head_kv], nb = [2, HS*n_head_kv*2, HS*2]; the output rows are
    HS*2 bytes apart.  Also the quoted scratch size at a 128k context."""
    g = _read_golden("kv_layout_p1.txt")
    hs, kv, nh = g["ne"]
    nb0, nb1, nb2 = g["nb"]
    elem = 2
    assert (nb0, nb1, nb2) == (elem, hs * nh * elem, hs * elem)
    # element (p, h, i) of the oracle's [depth][heads][head_dim] walk at byte offset:
    off = lambda p, h, i: elem * ((p * nh + h) * hs + i)
    assert off(1, 0, 0) - off(0, 0, 0) == nb1 and off(0, 1, 0) == nb2 and off(0, 0, 1) == nb0
    assert g["per_head_contiguous_row_bytes"][0] == hs * elem
    ctx = g["scratch_context"][0]
    assert 2 * nh * ctx * hs * elem == g["scratch_bytes_k_plus_v"][0]


def test_kv_round_trip(orc):
    """binary16 data quantized per 32 values and dequantized stays within half a step."""
    depth, heads, hd = 16, 4, 128
    v = syn.normal(0, "kv", (depth, heads, hd), dtype=torch.float16).float().numpy()
    q, d = orc.quantize_q8(v.reshape(-1, hd), 32)
    out = orc.dequant_q8_0_kv(q.reshape(depth, heads, hd), d.reshape(depth, heads, hd // 32))
    back = np.transpose(out.view(np.float16).astype(np.float64), (1, 0, 2))
    step = np.repeat(d.view(np.float16).astype(np.float64), 32, axis=1).reshape(depth, heads, hd)
    assert (np.abs(back - v) <= step * 0.5 + np.abs(v) * 2e-3 + 1e-7).all()
