"""A cache split by head: its kv heads spread over several caches (as over several
devices).  A whole state restores into the parts (each part its head range, in either
layout), the parts pack back into the very same stream, and decode on the parts (each
with its query heads) gives the unsplit cache's attention."""

import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle import state as ostate
from oracle.cache import OracleCache
from parity_util import assert_close, np32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc(cuda_device):
    import decode_attention_kv_cache_gb300 as m
    return m


def whole_cache(kvc, cache, n_layer, n, hkv=8, d=128):
    w = si.small_workload("split-heads", 40, hkv, d, cache, "bf16", n_prompt=n, chunk=n, n_decode=0, seed=61,
                          n_layer=n_layer, k_outlier_frac=0.01)
    g = kvc.KVCache(n_layer, w.n_ctx, hkv, d, cache, "head_major")
    ins = []
    for layer in range(n_layer):
        q, k, v = si.layer_qkv(w, layer)
        kvc.kv_cache_append(g, layer, 0, k.cuda(), v.cuda())
        ins.append((q, k, v))
    return w, g, ins


def heads_of(cache_obj, kv, lo, hi, n):
    """Codes (and scales) of kv heads [lo, hi) as [head][layer][pos][...] for positions [0, n)."""
    c = cache_obj.codes(kv)
    s = cache_obj.scales(kv)
    if cache_obj.layout == "head_major":
        out = [c[lo:hi, :, :n]] + ([s[lo:hi, :, :n]] if s is not None else [])
    else:
        out = [c[:, :n, lo:hi].permute(2, 0, 1, 3)] + ([s[:, :n, lo:hi].permute(2, 0, 1, 3)] if s is not None else [])
    return out


@pytest.mark.parametrize("cache", ["q8_0", "f16"])
@pytest.mark.parametrize("ranges", [((0, 4), (4, 8)), ((0, 3), (3, 5), (5, 8))])
def test_restore_into_head_parts_and_pack_back(kvc, cache, ranges):
    n_layer, n = 2, 300
    w, g, ins = whole_cache(kvc, cache, n_layer, n)
    state = kvc.kv_state_get(g, n)
    parts = []
    for i, (lo, hi) in enumerate(ranges):
        p = kvc.KVCache(n_layer, w.n_ctx, hi - lo, w.head_dim, cache, "layer_major" if i % 2 else "head_major")
        assert kvc.kv_state_set_heads(p, lo, state) == n
        parts.append(p)
    torch.cuda.synchronize()
    for (lo, hi), p in zip(ranges, parts):
        for kv in (0, 1):
            for x, y in zip(heads_of(p, kv, 0, hi - lo, n), heads_of(g, kv, lo, hi, n)):
                assert torch.equal(x, y)
    packed = torch.full_like(state, 0xAB)
    for (lo, hi), p in zip(ranges, parts):
        kvc.kv_state_get_heads(p, lo, w.n_head_kv, n, dst=packed)
    torch.cuda.synchronize()
    assert torch.equal(packed, state)
    # the stream is the oracle's
    o = OracleCache(n_layer, w.n_ctx, w.n_head_kv, w.head_dim, cache)
    for layer, (q, k, v) in enumerate(ins):
        o.append(layer, 0, np32(k), np32(v))
    assert np.array_equal(packed.cpu().numpy(), ostate.pack(o, n))
    assert kvc.kvc_device_status() == 0


def test_decode_on_head_parts_matches_the_whole(kvc):
    n_layer, n = 1, 2000
    w, g, ins = whole_cache(kvc, "q8_0", n_layer, n)
    state = kvc.kv_state_get(g, n)
    a = kvc.KVCache(1, w.n_ctx, 4, w.head_dim, "q8_0", "layer_major")
    b = kvc.KVCache(1, w.n_ctx, 4, w.head_dim, "q8_0", "head_major")
    kvc.kv_state_set_heads(a, 0, state)
    kvc.kv_state_set_heads(b, 4, state)
    q, k, v = ins[0]
    pos = n - 1
    qd = q[pos].cuda()
    whole = kvc.decode_attn(g, 0, pos, qd)
    split = torch.cat([kvc.decode_attn(a, 0, pos, qd[:20]), kvc.decode_attn(b, 0, pos, qd[20:])])
    torch.cuda.synchronize()
    assert_close(split.cpu().numpy(), whole.cpu().numpy().astype(np.float64), "split vs whole")
    o = OracleCache(1, w.n_ctx, w.n_head_kv, w.head_dim, "q8_0")
    o.append(0, 0, np32(k), np32(v))
    assert_close(split.cpu().numpy(), o.decode(0, pos, np32(q[pos])), "split vs oracle")


def test_a_range_beyond_the_state_is_rejected_and_writes_nothing(kvc):
    w, g, _ = whole_cache(kvc, "q8_0", 1, 64, hkv=4)
    state = kvc.kv_state_get(g, 64)
    p = kvc.KVCache(1, w.n_ctx, 2, w.head_dim, "q8_0", "head_major")
    p.codes(0).fill_(7)
    with pytest.raises(kvc.KvcError):
        kvc.kv_state_set_heads(p, 3, state)        # heads 3..4 of a 4-head state
    torch.cuda.synchronize()
    assert bool((p.codes(0) == 7).all())
