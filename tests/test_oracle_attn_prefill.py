"""Pins of the oracle's prefill attention: nq queries at the end of a cache of `depth`
positions, query i at position depth - nq + i seeing positions 0 .. depth - nq + i
("vulkan : dequant q8_0 KV once in coopmat1", Overview: the pp512 flash-attention
pass over the binary16 scratch; the stride discussion for the two layouts).

Each pin rests on something other than the function's own formula: a single query is
the decode attention (pinned in test_oracle_attn.py) bit for bit, every query equals
the decode attention over its visible prefix, the first query of a batch that fills
the cache sees one position, a dominant key placed just past a query's last visible
position changes nothing for that query and decides the next one, a permutation of
the prefix every query sees changes nothing, and the layouts and query-head grouping
agree."""
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


def _case(seed, heads=2, group=3, nq=5, depth=11, hd=32):
    q = f16(rnd(seed, (heads, group, nq, hd)))
    k = f16(rnd(seed + 1, (heads, depth, hd)))
    v = f16(rnd(seed + 2, (heads, depth, hd)))
    return q, k, v


def test_single_query_is_the_decode_attention():
    q, k, v = _case(0, nq=1, depth=9)
    out = oracle.attn_prefill(q, k, v, 0.17)
    qf = val(q[:, :, 0, :]).astype(np.float32)
    ref = oracle.attn_decode(qf, k, v, 0.17)
    assert np.array_equal(out[:, :, 0, :], ref)


def test_each_query_is_the_decode_attention_over_its_visible_prefix():
    heads, group, nq, depth = 2, 3, 6, 13
    q, k, v = _case(1, heads, group, nq, depth)
    out = oracle.attn_prefill(q, k, v, 0.2)
    for i in range(nq):
        vis = depth - nq + i + 1
        qf = val(q[:, :, i, :]).astype(np.float32)
        ref = oracle.attn_decode(qf, np.ascontiguousarray(k[:, :vis]), np.ascontiguousarray(v[:, :vis]), 0.2)
        assert np.array_equal(out[:, :, i, :], ref), i


def test_first_query_of_a_full_batch_sees_one_position():
    q, k, v = _case(2, nq=7, depth=7)
    out = oracle.attn_prefill(q, k, v, 0.5)
    for h in range(2):
        for g in range(3):
            assert np.array_equal(out[h, g, 0], val(v[h, 0]))


def test_a_key_past_the_last_visible_position_is_masked():
    """Query i's last visible position is depth - nq + i.  A key that dominates every
    score placed at depth - nq + i + 1 leaves query i unchanged and selects its value
    row for query i + 1."""
    heads, group, nq, depth, hd = 1, 1, 4, 10, 32
    q, k, v = _case(3, heads, group, nq, depth, hd)
    i = 1
    p = depth - nq + i + 1
    base = oracle.attn_prefill(q, k, v, 1.0)
    k2 = k.copy()
    qv = val(q[0, 0, i + 1])
    k2[0, p] = f16(np.sign(qv) * 60.0)  # score of about 60 * sum |q| against the rest
    out = oracle.attn_prefill(q, k2, v, 1.0)
    assert np.array_equal(out[0, 0, :i + 1], base[0, 0, :i + 1])
    assert np.allclose(out[0, 0, i + 1], val(v[0, p]), rtol=0, atol=1e-12)


def test_permuting_the_common_prefix_changes_nothing():
    heads, group, nq, depth = 2, 2, 4, 12
    q, k, v = _case(4, heads, group, nq, depth)
    out = oracle.attn_prefill(q, k, v, 0.3)
    perm = np.random.default_rng(5).permutation(depth - nq)  # positions every query sees
    k2, v2 = k.copy(), v.copy()
    k2[:, :depth - nq] = k[:, perm]
    v2[:, :depth - nq] = v[:, perm]
    out2 = oracle.attn_prefill(q, k2, v2, 0.3)
    assert np.allclose(out, out2, rtol=1e-12, atol=1e-14)


def test_position_major_layout_equals_per_head():
    q, k, v = _case(6)
    a = oracle.attn_prefill(q, k, v, 0.25)
    b = oracle.attn_prefill(q, np.ascontiguousarray(k.transpose(1, 0, 2)),
                            np.ascontiguousarray(v.transpose(1, 0, 2)), 0.25, layout="position_major")
    assert np.array_equal(a, b)


def test_each_query_head_of_a_group_equals_a_one_head_call():
    heads, group = 2, 4
    q, k, v = _case(7, heads, group)
    out = oracle.attn_prefill(q, k, v, 0.3)
    for g in range(group):
        one = oracle.attn_prefill(np.ascontiguousarray(q[:, g:g + 1]), k, v, 0.3)
        assert np.array_equal(out[:, g:g + 1], one)


def test_rejects_a_batch_longer_than_the_cache():
    q, k, v = _case(8, nq=5, depth=4)
    with pytest.raises(ValueError):
        oracle.attn_prefill(q, k, v, 0.3)
