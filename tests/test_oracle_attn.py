"""Pins of the oracle's decode attention (the consumer of the dequantized binary16 KV,
"vulkan : dequant q8_0 KV once in coopmat1", Overview and the stride discussion),
each against something other than the oracle's own formula: closed forms for one and
two positions, a uniform and a dominant key, invariances (position permutation, a
common score shift, linearity in V), the two layouts of the pages' strides, and the
query-head grouping."""
import math

import numpy as np
import pytest

import oracle


def f16(a):
    return np.asarray(a, dtype=np.float16).view(np.uint16)


def val(bits):
    return bits.view(np.float16).astype(np.float64)


def rnd(seed, shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


@pytest.fixture(scope="module", autouse=True)
def _lib():
    oracle.lib()


def test_one_position_returns_its_value_row():
    q = rnd(0, (2, 3, 128)).astype(np.float32)
    k, v = f16(rnd(1, (2, 1, 128))), f16(rnd(2, (2, 1, 128)))
    out = oracle.attn_decode(q, k, v, 0.3)
    for h in range(2):
        for g in range(3):
            assert np.array_equal(out[h, g], val(v[h, 0]))


def test_two_positions_closed_form():
    # out = v0 / (1 + e^(s1 - s0)) + v1 / (1 + e^(s0 - s1)); q has few bits so that
    # each score is an exact binary fraction
    q = (np.arange(16, dtype=np.float32) - 8.0).reshape(1, 1, 16) / 4
    kv = np.array([[1, -1] * 8, [0.5] * 16], np.float64)
    k = f16(kv.reshape(1, 2, 16))
    v = f16(rnd(3, (1, 2, 16)))
    scale = 0.25
    s = [scale * float(np.dot(q[0, 0].astype(np.float64), kv[p])) for p in range(2)]
    a0 = 1.0 / (1.0 + math.exp(s[1] - s[0]))
    a1 = 1.0 / (1.0 + math.exp(s[0] - s[1]))
    want = a0 * val(v[0, 0]) + a1 * val(v[0, 1])
    got = oracle.attn_decode(q, k, v, scale)[0, 0]
    assert np.allclose(got, want, rtol=1e-14, atol=1e-15)


def test_equal_keys_give_the_mean_of_the_values():
    depth = 37
    row = f16(rnd(4, 64))
    k = np.tile(row, (3, depth, 1))
    v = f16(rnd(5, (3, depth, 64)))
    q = rnd(6, (3, 2, 64)).astype(np.float32)
    out = oracle.attn_decode(q, k, v, 1 / 8)
    mean = val(v).sum(axis=1) / depth
    for g in range(2):
        assert np.allclose(out[:, g], mean, rtol=1e-14, atol=1e-15)


def test_a_dominant_key_selects_its_value_even_at_large_scores():
    # s_j - s_p >= 1000 for every other p: every other weight underflows to zero, and
    # without subtracting the maximum exp(s_j) would overflow
    depth, j = 50, 17
    k = np.zeros((1, depth, 32), np.float64)
    k[0, :, 0] = 1.0
    k[0, j, 0] = 64.0
    v = f16(rnd(7, (1, depth, 32)))
    q = np.zeros((1, 1, 32), np.float32)
    q[0, 0, 0] = 32.0
    out = oracle.attn_decode(q, f16(k), v, 1.0)  # s_j = 2048, others 32
    assert np.array_equal(out[0, 0], val(v[0, j]))


def test_permuting_positions_and_shifting_scores_change_nothing():
    depth = 300
    k = f16(rnd(8, (2, depth, 128)))
    v = f16(rnd(9, (2, depth, 128)))
    q = rnd(10, (2, 4, 128)).astype(np.float32)
    ref = oracle.attn_decode(q, k, v, 1 / math.sqrt(128))
    perm = np.random.default_rng(11).permutation(depth)
    got = oracle.attn_decode(q, k[:, perm], v[:, perm], 1 / math.sqrt(128))
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-14)
    # a dimension whose key value is the same at every position adds the same
    # constant to every score of a query
    k2 = k.copy()
    k2[:, :, 5] = f16(3.0)
    q2 = q.copy()
    q2[:, :, 5] = 0.0
    a = oracle.attn_decode(q2, k2, v, 0.1)
    q2[:, :, 5] = 7.0
    b = oracle.attn_decode(q2, k2, v, 0.1)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)


def test_linear_in_the_values():
    # small integers: v1 + v2 is exact in binary16
    g = np.random.default_rng(12)
    v1 = g.integers(-50, 50, (1, 40, 64)).astype(np.float64)
    v2 = g.integers(-50, 50, (1, 40, 64)).astype(np.float64)
    k = f16(rnd(13, (1, 40, 64)))
    q = rnd(14, (1, 2, 64)).astype(np.float32)
    o1 = oracle.attn_decode(q, k, f16(v1), 0.2)
    o2 = oracle.attn_decode(q, k, f16(v2), 0.2)
    o12 = oracle.attn_decode(q, k, f16(v1 + v2), 0.2)
    assert np.allclose(o12, o1 + o2, rtol=1e-12, atol=1e-12)


def test_position_major_layout_reads_the_same_rows():
    # the cache walks [position][head][dim] (row stride head_dim * heads), the scratch
    # [head][position][dim]; same values, same result bit for bit
    heads, depth = 4, 70
    k = f16(rnd(15, (heads, depth, 128)))
    v = f16(rnd(16, (heads, depth, 128)))
    q = rnd(17, (heads, 2, 128)).astype(np.float32)
    a = oracle.attn_decode(q, k, v, 0.09)
    b = oracle.attn_decode(q, np.ascontiguousarray(k.transpose(1, 0, 2)),
                           np.ascontiguousarray(v.transpose(1, 0, 2)), 0.09, layout="position_major")
    assert np.array_equal(a, b)
    # and every head reads its own rows: heads with swapped data swap their outputs
    c = oracle.attn_decode(q[[1, 0, 2, 3]], k[[1, 0, 2, 3]], v[[1, 0, 2, 3]], 0.09)
    assert np.array_equal(c, a[[1, 0, 2, 3]])


def test_query_heads_of_a_group_share_the_kv_head():
    heads, group, depth = 2, 3, 25
    k = f16(rnd(18, (heads, depth, 32)))
    v = f16(rnd(19, (heads, depth, 32)))
    q = rnd(20, (heads, group, 32)).astype(np.float32)
    out = oracle.attn_decode(q, k, v, 0.5)
    for h in range(heads):
        for g in range(group):
            one = oracle.attn_decode(q[h:h + 1, g:g + 1], k[h:h + 1], v[h:h + 1], 0.5)
            assert np.array_equal(out[h, g], one[0, 0])
