"""Pins for the oracle's causal GQA attention and its cache flow (no GPU).

The attention is checked against torch's float64 scaled_dot_product_attention
(a library routine; grouped heads expanded with repeat_interleave), against
closed forms (the first row returns the first value row; identical keys give
the mean of the values; constant values come back unchanged; a two-key case
written out by hand), and the cache flow against the invariants the pages
state (a prompt cut into chunks gives the result of one pass; decoding at p
equals a one-row chunk at p).
"""

import math

import numpy as np
import pytest
import torch

from oracle.attention import attend
from oracle.cache import OracleCache


def sdpa_reference(q, positions, k, v):
    """torch float64 SDPA with the causal mask of absolute positions; K/V expanded per query head."""
    n_rows, n_head_q, d = q.shape
    n_head_kv, n = k.shape[0], k.shape[1]
    g = n_head_q // n_head_kv
    qt = torch.from_numpy(np.ascontiguousarray(q.transpose(1, 0, 2)))              # [H_q, R, D]
    kt = torch.from_numpy(k).repeat_interleave(g, dim=0)                            # [H_q, n, D]
    vt = torch.from_numpy(v).repeat_interleave(g, dim=0)
    mask = torch.from_numpy(np.arange(n)[None, :] <= np.asarray(positions)[:, None])  # [R, n]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
    return o.numpy().transpose(1, 0, 2)


@pytest.mark.parametrize("h_q,h_kv,d,n", [(4, 2, 64, 37), (40, 8, 128, 70), (3, 3, 32, 9), (8, 1, 96, 20)])
def test_matches_library_sdpa(h_q, h_kv, d, n):
    rng = np.random.default_rng(h_q * 100 + n)
    k = rng.standard_normal((h_kv, n, d))
    v = rng.standard_normal((h_kv, n, d))
    pos = np.sort(rng.choice(n, size=min(n, 11), replace=False))
    q = rng.standard_normal((pos.size, h_q, d)) * 2
    np.testing.assert_allclose(attend(q, pos, k, v), sdpa_reference(q, pos, k, v), rtol=1e-12, atol=1e-12)


def test_first_row_returns_first_value_row():
    rng = np.random.default_rng(1)
    k = rng.standard_normal((2, 10, 64))
    v = rng.standard_normal((2, 10, 64))
    q = rng.standard_normal((1, 6, 64)) * 5
    o = attend(q, [0], k, v)
    for h in range(6):
        assert (o[0, h] == v[h // 3, 0]).all()


def test_identical_keys_average_the_values():
    rng = np.random.default_rng(2)
    k = np.repeat(rng.standard_normal((1, 1, 32)), 12, axis=1)
    v = rng.standard_normal((1, 12, 32))
    q = rng.standard_normal((12, 2, 32))
    o = attend(q, np.arange(12), k, v)
    for t in range(12):
        np.testing.assert_allclose(o[t], np.broadcast_to(v[0, :t + 1].mean(0), (2, 32)), rtol=0, atol=1e-14)


def test_constant_values_come_back_unchanged():
    # softmax weights sum to one: with every value row equal to c, every output equals c
    rng = np.random.default_rng(3)
    k = rng.standard_normal((2, 50, 64)) * 3
    c = rng.standard_normal(64)
    v = np.broadcast_to(c, (2, 50, 64)).copy()
    q = rng.standard_normal((50, 4, 64)) * 3
    o = attend(q, np.arange(50), k, v)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-12)


def test_two_keys_written_out():
    # D = 32, query a*e0, keys b*e0 and 0: scores ab/sqrt(32) and 0
    a, b = 1.7, -2.3
    q = np.zeros((1, 1, 32)); q[0, 0, 0] = a
    k = np.zeros((1, 2, 32)); k[0, 0, 0] = b
    rng = np.random.default_rng(4)
    v = rng.standard_normal((1, 2, 32))
    e = math.exp(a * b / math.sqrt(32))
    expect = (e * v[0, 0] + v[0, 1]) / (e + 1)
    np.testing.assert_allclose(attend(q, [1], k, v)[0, 0], expect, rtol=1e-14, atol=1e-15)


def _prefill(cache, q, k, v, chunk):
    outs = []
    n = q.shape[0]
    for p in range(0, n, chunk):
        c = min(chunk, n - p)
        cache.append(0, p, k[p:p + c], v[p:p + c])
        outs.append(cache.prefill_chunk(0, p, q[p:p + c]))
    return np.concatenate(outs)


@pytest.mark.parametrize("cache_type", ["q8_0", "f16"])
def test_chunked_prefill_equals_one_pass(cache_type):
    rng = np.random.default_rng(5)
    n, h_q, h_kv, d = 150, 4, 2, 64
    q = rng.standard_normal((n, h_q, d)).astype(np.float32)
    k = rng.standard_normal((n, h_kv, d)).astype(np.float32)
    v = rng.standard_normal((n, h_kv, d)).astype(np.float32)
    ref_cache = OracleCache(1, 256, h_kv, d, cache_type)
    ref = _prefill(ref_cache, q, k, v, n)
    for chunk in (1, 7, 64, 100):
        c = OracleCache(1, 256, h_kv, d, cache_type)
        out = _prefill(c, q, k, v, chunk)
        np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)
        for a, b in zip(c.device_image("layer_major"), ref_cache.device_image("layer_major")):
            if a is not None:
                assert (a == b).all()


def test_decode_equals_one_row_chunk():
    rng = np.random.default_rng(6)
    h_q, h_kv, d = 4, 2, 64
    c = OracleCache(1, 64, h_kv, d, "q8_0")
    k = rng.standard_normal((40, h_kv, d)).astype(np.float32)
    v = rng.standard_normal((40, h_kv, d)).astype(np.float32)
    q = rng.standard_normal((40, h_q, d)).astype(np.float32)
    c.append(0, 0, k, v)
    for p in (0, 17, 39):
        np.testing.assert_array_equal(c.decode(0, p, q[p]), c.prefill_chunk(0, p, q[p:p + 1])[0])


def test_chunk_sees_its_own_keys_as_stored():
    # a chunk row attends over the dequantised cache, including the keys of its own chunk
    rng = np.random.default_rng(8)
    c = OracleCache(1, 16, 1, 32, "q8_0")
    k = rng.standard_normal((4, 1, 32)).astype(np.float32)
    v = rng.standard_normal((4, 1, 32)).astype(np.float32)
    q = rng.standard_normal((4, 1, 32)).astype(np.float32)
    c.append(0, 0, k, v)
    kh, vh = c.dequantized(0, 4)
    assert not np.array_equal(kh[0], k[:, 0].astype(np.float64))     # quantisation changed the keys
    np.testing.assert_array_equal(c.prefill_chunk(0, 0, q), attend(q, np.arange(4), kh, vh))
