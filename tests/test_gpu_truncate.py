"""kv_cache_truncate: a sequence that drops its last appends (speculative decode
tokens, or a trimmed excess) and appends other tokens in their place computes
exactly what a cache that never held the dropped tokens computes, and the dropped
positions read back as zero bytes."""

import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle.cache import OracleCache
from parity_util import assert_close, np32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc(cuda_device):
    import decode_attention_kv_cache_gb300 as m
    return m


@pytest.mark.parametrize("cache,layout", [("q8_0", "head_major"), ("f16", "layer_major"), ("q8_0", "layer_major")])
def test_rewind_then_append_equals_a_cache_without_the_dropped_tokens(kvc, cache, layout):
    n_layer, n0, drop, keep = 2, 700, 37, 5
    w = si.small_workload("trunc", 10, 2, 128, cache, "bf16", n_prompt=n0 + drop, chunk=256, n_decode=0, seed=7,
                          n_layer=n_layer)
    other = si.small_workload("trunc-other", 10, 2, 128, cache, "bf16", n_prompt=n0 + keep, chunk=256, n_decode=0,
                              seed=8, n_layer=n_layer)
    a = kvc.KVCache(n_layer, w.n_ctx, w.n_head_kv, w.head_dim, cache, layout)
    b = kvc.KVCache(n_layer, w.n_ctx, w.n_head_kv, w.head_dim, cache, layout)
    for kv in (0, 1):   # b starts zeroed, the state a rewound cache must reach past its appends
        b.codes(kv).zero_()
        if cache == "q8_0":
            b.scales(kv).zero_()
    ins, alt = [], []
    for layer in range(n_layer):
        q, k, v = (t.cuda() for t in si.layer_qkv(w, layer))
        q2, k2, v2 = (t.cuda() for t in si.layer_qkv(other, layer))
        ins.append((q, k, v))
        alt.append((q2, k2, v2))
        kvc.kv_cache_append(a, layer, 0, k, v)                     # n0 + drop tokens
        kvc.kv_cache_append(b, layer, 0, k[:n0], v[:n0])
    kvc.kv_cache_truncate(a, n0)
    for layer in range(n_layer):
        _, k2, v2 = alt[layer]
        for c in (a, b):
            kvc.kv_cache_append(c, layer, n0, k2[n0:n0 + keep], v2[n0:n0 + keep])
    torch.cuda.synchronize()
    for kv in (0, 1):
        assert torch.equal(a.codes(kv), b.codes(kv))
        if cache == "q8_0":
            assert torch.equal(a.scales(kv), b.scales(kv))
    # attention over the rewound cache: decode at the last kept position, bitwise equal to b and to the oracle
    for layer in range(n_layer):
        q2 = alt[layer][0]
        pos = n0 + keep - 1
        oa = kvc.decode_attn(a, layer, pos, q2[pos])
        ob = kvc.decode_attn(b, layer, pos, q2[pos])
        assert torch.equal(oa, ob)
        o = OracleCache(1, w.n_ctx, w.n_head_kv, w.head_dim, cache)
        _, k, v = (t.cpu() for t in ins[layer])
        _, k2, v2 = (t.cpu() for t in alt[layer])
        o.append(0, 0, np32(k[:n0]), np32(v[:n0]))
        o.append(0, n0, np32(k2[n0:n0 + keep]), np32(v2[n0:n0 + keep]))
        assert_close(oa.cpu().numpy(), o.decode(0, pos, np32(q2[pos].cpu())), "decode after rewind")
    # rewinding to zero clears everything
    kvc.kv_cache_truncate(a, 0)
    torch.cuda.synchronize()
    for kv in (0, 1):
        assert not a.codes(kv).view(torch.int16 if cache == "f16" else torch.int8).any()
    assert kvc.kvc_device_status() == 0
