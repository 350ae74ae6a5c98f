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
