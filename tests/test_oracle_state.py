"""Pins for the oracle's state pack/unpack and the cache layouts (no GPU).

The format is pinned by hand-written byte fixtures, the size rule by the state
sizes the pages print, the layouts by explicit index loops, and the round trip
and error behaviour by invariants.
"""

import itertools

import numpy as np
import pytest

from golden_io import read_hex
from oracle import state
from oracle.cache import OracleCache


def test_q8_0_fixture():
    c = OracleCache(1, 4, 1, 32, "q8_0")
    k0 = np.array([-127.0] + list(range(-15, 16)), np.float32)
    k1 = np.array([63.5] + [0.5 * i for i in range(-15, 16)], np.float32)
    v1 = np.zeros(32, np.float32)
    v1[:6] = [15.875, 0.0625, -0.0625, 0.1875, -0.3125, 0.03125]
    c.append(0, 0, np.stack([k0, k1])[:, None, :], np.stack([np.zeros(32, np.float32), v1])[:, None, :])
    assert (state.pack(c, 2) == read_hex("state_q8_0_tiny.txt")).all()


def test_f16_fixture():
    c = OracleCache(1, 4, 1, 32, "f16")
    k = np.zeros(32, np.float32)
    k[:10] = [1.0, -2.0, 0.5, 65504.0, 2.0 ** -24, np.float32(1.0) / np.float32(3.0), -0.0,
              np.float32(0.1), 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11]
    c.append(0, 0, k[None, None, :], np.full((1, 1, 32), 2.0, np.float32))
    assert (state.pack(c, 1) == read_hex("state_f16_tiny.txt")).all()


def test_fixture_restores_into_an_empty_cache():
    c = OracleCache(1, 4, 1, 32, "q8_0")
    blob = read_hex("state_q8_0_tiny.txt")
    assert state.unpack(blob, c) == 2
    assert c.k_q[0, 0, 0].tolist() == [-127] + list(range(-15, 16))
    assert c.v_q[0, 1, 0, :6].tolist() == [127, 1, -1, 2, -3, 0]
    assert (state.pack(c, 2) == blob).all()


@pytest.mark.parametrize("cache_type", ["q8_0", "f16"])
def test_round_trip_is_byte_identical(cache_type):
    rng = np.random.default_rng(11)
    L, n_ctx, H, D, n = 3, 40, 2, 64, 29
    a = OracleCache(L, n_ctx, H, D, cache_type)
    for layer in range(L):
        a.append(layer, 0, rng.standard_normal((n, H, D)).astype(np.float32) * 2,
                 rng.standard_normal((n, H, D)).astype(np.float32))
    blob = state.pack(a, n)
    assert blob.size == state.state_size(L, H, D, cache_type, n)
    b = OracleCache(L, n_ctx, H, D, cache_type)
    assert state.unpack(blob, b) == n
    assert (state.pack(b, n) == blob).all()
    for x, y in zip(a.device_image("head_major"), b.device_image("head_major")):
        if x is not None:
            assert (x[:, :, :n] == y[:, :, :n]).all()


def test_layout_images_index_the_logical_store():
    rng = np.random.default_rng(12)
    L, n_ctx, H, D = 2, 5, 3, 32
    c = OracleCache(L, n_ctx, H, D, "q8_0")
    for layer in range(L):
        c.append(layer, 0, rng.standard_normal((n_ctx, H, D)).astype(np.float32),
                 rng.standard_normal((n_ctx, H, D)).astype(np.float32))
    hk, hks, _, _ = c.device_image("head_major")
    lk, lks, _, _ = c.device_image("layer_major")
    for l, t, h in itertools.product(range(L), range(n_ctx), range(H)):
        for dim in (0, 7, 31):
            assert hk[h, l, t, dim] == c.k_q[l, t, h, dim] == lk[l, t, h, dim]
        assert hks[h, l, t, 0] == c.k_d[l, t, h, 0] == lks[l, t, h, 0]
    # flat offsets of the two layouts as documented
    flat_h, flat_l = hk.reshape(-1), lk.reshape(-1)
    l, t, h, dim = 1, 3, 2, 17
    assert flat_h[((h * L + l) * n_ctx + t) * D + dim] == flat_l[((l * n_ctx + t) * H + h) * D + dim]


def test_size_rule_reproduces_the_printed_state_sizes():
    # llama.cpp PR #58, section "Result": 2085 MiB of state for the 58.3k-token prompt (q8_0 cache);
    # llama.cpp PR #59, section "Why": 1216 MiB for 17055 tokens (f16 cache).  Both are linear in the
    # context (PR #58, section "Cost").  With 16 attention layers of 8 kv heads x 128 dims (an
    # inference: the pages do not print the model's shape), the per-token bytes leave the same
    # constant in both runs only with 34-byte q8_0 blocks and no padding to the context size.
    mib = 2.0 ** 20
    q8 = state.state_size(16, 8, 128, "q8_0", 58300) / mib
    f16 = state.state_size(16, 8, 128, "f16", 17055) / mib
    rest_q8, rest_f16 = 2085 - q8, 1216 - f16
    # "58.3k" is rounded to 100 tokens: +-50 tokens are +-1.7 MiB of q8_0 state
    assert abs(rest_q8 - rest_f16) < 1.7 + 0.5
    # a 36-byte block (fp32 scale) or padding to the context (65,536 / 20,480) would not agree
    per_tok_36 = 16 * 2 * 8 * 4 * 36
    assert abs((2085 - 58300 * per_tok_36 / mib) - rest_f16) > 50
    # padding to the context would need more bytes than were printed
    assert state.state_size(16, 8, 128, "q8_0", 65536) / mib > 2085
    assert state.state_size(16, 8, 128, "f16", 20480) / mib > 1216


@pytest.mark.parametrize("mutate", ["magic", "version", "shape", "type", "tokens", "size", "reserved", "short"])
def test_invalid_state_is_rejected_and_writes_nothing(mutate):
    rng = np.random.default_rng(13)
    a = OracleCache(1, 8, 1, 32, "q8_0")
    a.append(0, 0, rng.standard_normal((6, 1, 32)).astype(np.float32),
             rng.standard_normal((6, 1, 32)).astype(np.float32))
    blob = state.pack(a, 6).copy()
    words = blob[:32].view("<u4")
    if mutate == "magic":
        words[0] ^= 1
    elif mutate == "version":
        words[1] = 2
    elif mutate == "shape":
        words[4] = 64
    elif mutate == "type":
        words[5] = 0
    elif mutate == "tokens":
        words[6] = 9
    elif mutate == "reserved":
        words[7] = 1
    elif mutate == "size":
        blob = blob[:-1]
    elif mutate == "short":
        blob = blob[:20]
    b = OracleCache(1, 8, 1, 32, "q8_0")
    b.k_q[:] = 5
    with pytest.raises(ValueError):
        state.unpack(blob, b)
    assert (b.k_q == 5).all() and (b.v_q == 0).all()
