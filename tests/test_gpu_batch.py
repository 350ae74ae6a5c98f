"""decode_attn_batch: several sequences, each with its own cache, length and layout,
decoded in one call.  Every sequence's output matches the oracle and the
single-sequence decode_attn within the attention tolerance (a batch may split the
key range differently); a batch of one equals decode_attn bit for bit."""

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


N_CTX = 4200
LENGTHS = [3000, 17, 1500, 700, 2, 4096, 900, 256]


def make_sequences(kvc, n_seq, hq, hkv, d, cache, dtype):
    seqs = []
    for i in range(n_seq):
        n = LENGTHS[i]
        w = si.small_workload("batch%d" % i, hq, hkv, d, cache, dtype, n_prompt=n, chunk=n, n_decode=0,
                              seed=500 + 7 * i, n_ctx=N_CTX, k_outlier_frac=0.01)
        q, k, v = si.layer_qkv(w, 0)
        g = kvc.KVCache(1, N_CTX, hkv, d, cache, "head_major" if i % 2 == 0 else "layer_major")
        kvc.kv_cache_append(g, 0, 0, k.cuda(), v.cuda())
        seqs.append((w, g, q, k, v, n - 1))
    return seqs


@pytest.mark.parametrize("n_seq,cache,d,dtype", [(2, "q8_0", 128, "bf16"), (5, "f16", 128, "bf16"),
                                                 (8, "q8_0", 128, "f16"), (8, "f16", 128, "f32"),
                                                 (3, "q8_0", 64, "bf16")])
def test_batch_matches_oracle_and_single_decode(kvc, n_seq, cache, d, dtype):
    hq, hkv = 10, 2
    seqs = make_sequences(kvc, n_seq, hq, hkv, d, cache, dtype)
    qb = torch.stack([q[p] for (_, _, q, _, _, p) in seqs]).cuda()
    out = kvc.decode_attn_batch([s[1] for s in seqs], 0, [s[5] for s in seqs], qb)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    for i, (w, g, q, k, v, p) in enumerate(seqs):
        single = kvc.decode_attn(g, 0, p, q[p].cuda())
        assert_close(out[i].cpu().numpy(), single.cpu().numpy().astype(np.float64), "seq %d vs single" % i)
        o = OracleCache(1, N_CTX, hkv, d, cache)
        o.append(0, 0, np32(k[:p + 1]), np32(v[:p + 1]))
        assert_close(out[i].cpu().numpy(), o.decode(0, p, np32(q[p])), "seq %d vs oracle" % i)


def test_batch_of_one_equals_decode_attn(kvc):
    (w, g, q, k, v, p), = make_sequences(kvc, 1, 40, 8, 128, "q8_0", "bf16")
    out = kvc.decode_attn_batch([g], 0, [p], q[p:p + 1].cuda())
    single = kvc.decode_attn(g, 0, p, q[p].cuda())
    assert torch.equal(out[0], single)


def test_batch_in_a_cuda_graph_replays(kvc):
    seqs = make_sequences(kvc, 4, 40, 8, 128, "q8_0", "bf16")
    caches, pos = [s[1] for s in seqs], [s[5] for s in seqs]
    qb = torch.stack([q[p] for (_, _, q, _, _, p) in seqs]).cuda()
    out = torch.empty(4, 40, 128, device="cuda")
    scratch = torch.empty(4 * caches[0].scratch_bytes(40), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        kvc.decode_attn_batch(caches, 0, pos, qb, out=out, scratch=scratch)
        torch.cuda.synchronize()
        ref = out.clone()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            kvc.decode_attn_batch(caches, 0, pos, qb, out=out, scratch=scratch)
    out.zero_()
    gr.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


@pytest.mark.parametrize("cache,dtype", [("q8_0", "bf16"), ("f16", "f32"), ("q8_0", "f16")])
def test_batched_append_equals_one_append_per_sequence(kvc, cache, dtype):
    n_seq, hkv, d = 6, 8, 128
    pos = [0, 4199, 17, 2048, 777, 3000]
    w = si.small_workload("bappend", 40, hkv, d, cache, dtype, n_prompt=n_seq, chunk=n_seq, n_decode=0, seed=77,
                          n_ctx=N_CTX, k_outlier_frac=0.01)
    _, k, v = si.layer_qkv(w, 0)
    k, v = k.cuda(), v.cuda()
    a = [kvc.KVCache(2, N_CTX, hkv, d, cache, "head_major" if i % 2 else "layer_major") for i in range(n_seq)]
    b = [kvc.KVCache(2, N_CTX, hkv, d, cache, "head_major" if i % 2 else "layer_major") for i in range(n_seq)]
    for x, y in zip(a, b):
        for kv in (0, 1):
            x.codes(kv).zero_(); y.codes(kv).zero_()
            if cache == "q8_0":
                x.scales(kv).zero_(); y.scales(kv).zero_()
    kvc.kv_cache_append_batch(a, 1, pos, k, v)
    for i in range(n_seq):
        kvc.kv_cache_append(b[i], 1, pos[i], k[i:i + 1], v[i:i + 1])
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        for kv in (0, 1):
            assert torch.equal(x.codes(kv), y.codes(kv))
            if cache == "q8_0":
                assert torch.equal(x.scales(kv), y.scales(kv))
    # and the appended rows are the oracle's bytes
    for i in range(n_seq):
        o = OracleCache(1, N_CTX, hkv, d, cache)
        o.append(0, pos[i], np32(k[i:i + 1].cpu()), np32(v[i:i + 1].cpu()))
        img = o.device_image("head_major")
        for kv in (0, 1):
            got = a[i].codes(kv)
            got = got[:, 1, pos[i]] if a[i].layout == "head_major" else got[1, pos[i]]
            ref = img[2 * kv][:, 0, pos[i]]
            if cache == "q8_0":
                assert np.array_equal(got.cpu().numpy(), ref)
            else:
                assert np.array_equal(got.cpu().view(torch.int16).numpy(), ref.view(np.int16))
