"""decode_step and decode_step_batch: the fused decode step (store the token, attend) against the two
calls it stands for.  The output equals append + decode_attn's bit for bit (the same split boundaries
and the same merge) and matches the oracle within the attention tolerance; the stored bytes equal the
oracle's, as kv_cache_append's do."""

import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle.cache import OracleCache
from parity_util import assert_cache_equal, assert_close, np32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc(cuda_device):
    import decode_attention_kv_cache_gb300 as m
    return m


CASES = [
    # H_q, H_kv, D, cache, dtype, prompt tokens, decode steps
    (40, 8, 128, "q8_0", "bf16", 250, 8),    # steps cross the tile edge at 256
    (40, 8, 128, "f16", "bf16", 124, 8),     # ... and at 128
    (8, 8, 128, "q8_0", "f32", 60, 5),       # G = 1
    (32, 2, 128, "f16", "f16", 300, 4),      # G = 16
    (32, 2, 128, "q8_0", "bf16", 200, 3),    # G = 16 with q8_0: 16 head slots, the token dequantised in place
    (12, 4, 128, "f16", "f32", 127, 3),      # f32 inputs into an f16 cache, the first step at a tile edge
    (24, 2, 128, "q8_0", "bf16", 0, 6),      # from an empty cache: the first step attends to itself
    (4, 2, 64, "q8_0", "f32", 100, 4),       # head_dim 64: append and decode_attn in turn
    (4, 2, 64, "f16", "bf16", 63, 3),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%d-%d-%d-%s-%s-%d" % c[:6])
def test_step_equals_append_then_decode(kvc, case):
    hq, hkv, d, cache, dt, n0, steps = case
    w = si.small_workload("step", hq, hkv, d, cache, dt, n_prompt=max(n0, 1), chunk=max(n0, 1), n_decode=steps,
                          seed=hq * 13 + d + n0, k_outlier_frac=0.01)
    q, k, v = si.layer_qkv(w, 0)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ga = kvc.KVCache(1, w.n_ctx, hkv, d, cache, "head_major")
    gb = kvc.KVCache(1, w.n_ctx, hkv, d, cache, "layer_major" if d == 128 else "head_major")
    o = OracleCache(1, w.n_ctx, hkv, d, cache)
    if n0 > 0:
        for g in (ga, gb):
            kvc.kv_cache_append(g, 0, 0, kd[:n0], vd[:n0])
        o.append(0, 0, np32(k[:n0]), np32(v[:n0]))
    sa = torch.empty(ga.scratch_bytes(hq), dtype=torch.uint8, device="cuda")
    sb = torch.empty(gb.scratch_bytes(hq), dtype=torch.uint8, device="cuda")
    for pos in range(n0, n0 + steps):
        kvc.kv_cache_append(ga, 0, pos, kd[pos:pos + 1], vd[pos:pos + 1])
        ref = kvc.decode_attn(ga, 0, pos, qd[pos], scratch=sa)
        out = kvc.decode_step(gb, 0, pos, qd[pos], kd[pos], vd[pos], scratch=sb)
        o.append(0, pos, np32(k[pos:pos + 1]), np32(v[pos:pos + 1]))
        torch.cuda.synchronize()
        assert kvc.kvc_device_status() == 0
        assert torch.equal(out, ref), "decode_step differs from append + decode_attn at pos %d" % pos
        assert_close(out.cpu().numpy(), o.decode(0, pos, np32(q[pos])), "pos %d" % pos)
    # the stored bytes, bit for bit (the append path is held to the same oracle bytes)
    assert_cache_equal(gb, o, n0 + steps)


def test_step_long_context_many_splits(kvc):
    # 9,000 keys: 19 splits of each of the 8 kv heads; the token lands in the last tile of the last split
    w = si.small_workload("steplong", 40, 8, 128, "q8_0", "bf16", n_prompt=8998, chunk=4096, n_decode=2, seed=21,
                          k_outlier_frac=0.01)
    q, k, v = si.layer_qkv(w, 0)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ga = kvc.KVCache(1, w.n_ctx, 8, 128, "q8_0", "head_major")
    gb = kvc.KVCache(1, w.n_ctx, 8, 128, "q8_0", "head_major")
    for g in (ga, gb):
        kvc.kv_cache_append(g, 0, 0, kd[:8998], vd[:8998])
    sb = torch.empty(gb.scratch_bytes(40), dtype=torch.uint8, device="cuda")
    o = OracleCache(1, w.n_ctx, 8, 128, "q8_0")
    o.append(0, 0, np32(k[:8998]), np32(v[:8998]))
    for pos in (8998, 8999):
        kvc.kv_cache_append(ga, 0, pos, kd[pos:pos + 1], vd[pos:pos + 1])
        ref = kvc.decode_attn(ga, 0, pos, qd[pos])
        out = kvc.decode_step(gb, 0, pos, qd[pos], kd[pos], vd[pos], scratch=sb)
        o.append(0, pos, np32(k[pos:pos + 1]), np32(v[pos:pos + 1]))
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        assert_close(out.cpu().numpy(), o.decode(0, pos, np32(q[pos])), "pos %d" % pos)
    assert_cache_equal(gb, o, 9000)


@pytest.mark.parametrize("n_seq,cache,d,dtype", [(3, "q8_0", 128, "bf16"), (8, "f16", 128, "f16"),
                                                 (2, "q8_0", 64, "bf16")])
def test_step_batch_equals_append_batch_then_decode_batch(kvc, n_seq, cache, d, dtype):
    hq, hkv, n_ctx = 10, 2, 3000
    lengths = [2000, 5, 900, 128, 127, 1, 2500, 640][:n_seq]
    ws = [si.small_workload("sb%d" % i, hq, hkv, d, cache, dtype, n_prompt=n, chunk=n, n_decode=3, seed=70 + i,
                            n_ctx=n_ctx) for i, n in enumerate(lengths)]
    qkv = [si.layer_qkv(w, 0) for w in ws]
    ga, gb = [], []
    for i, (w, (q, k, v)) in enumerate(zip(ws, qkv)):
        for lst in (ga, gb):
            g = kvc.KVCache(1, n_ctx, hkv, d, cache, "head_major" if i % 2 == 0 else "layer_major")
            kvc.kv_cache_append(g, 0, 0, k[:lengths[i]].cuda(), v[:lengths[i]].cuda())
            lst.append(g)
    sa = torch.empty(n_seq * ga[0].scratch_bytes(hq), dtype=torch.uint8, device="cuda")
    sb = torch.empty(n_seq * gb[0].scratch_bytes(hq), dtype=torch.uint8, device="cuda")
    for t in range(3):
        pos = [n + t for n in lengths]
        qb = torch.stack([q[p] for (q, _, _), p in zip(qkv, pos)]).cuda()
        kb = torch.stack([k[p] for (_, k, _), p in zip(qkv, pos)]).cuda()
        vb = torch.stack([v[p] for (_, _, v), p in zip(qkv, pos)]).cuda()
        kvc.kv_cache_append_batch(ga, 0, pos, kb, vb)
        ref = kvc.decode_attn_batch(ga, 0, pos, qb, scratch=sa)
        out = kvc.decode_step_batch(gb, 0, pos, qb, kb, vb, scratch=sb)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status() == 0
        assert torch.equal(out, ref), "step %d" % t
    for i in range(n_seq):
        q, k, v = qkv[i]
        p = lengths[i] + 2
        o = OracleCache(1, n_ctx, hkv, d, cache)
        o.append(0, 0, np32(k[:p + 1]), np32(v[:p + 1]))
        assert_cache_equal(gb[i], o, p + 1)
        assert_close(out[i].cpu().numpy(), o.decode(0, p, np32(q[p])), "seq %d vs oracle" % i)


@pytest.mark.parametrize("cache", ["q8_0", "f16"])
def test_step_loop_captured_in_a_cuda_graph(kvc, cache):
    # the decode loop as the bench runs it: steps captured once in a CUDA graph (programmatic launches
    # inside the graph), replayed; each step equals the eager step bit for bit, twice over
    w = si.small_workload("stepgraph", 40, 8, 128, cache, "bf16", n_prompt=3000, chunk=3000, n_decode=8, seed=44)
    q, k, v = (t.cuda() for t in si.layer_qkv(w, 0))
    g = kvc.KVCache(1, w.n_ctx, 8, 128, cache, "head_major")
    kvc.kv_cache_append(g, 0, 0, k[:3000], v[:3000])
    scratch = torch.empty(g.scratch_bytes(40), dtype=torch.uint8, device="cuda")
    eager = torch.empty(8, 40, 128, device="cuda")
    graph_out = torch.empty_like(eager)

    def loop(out):
        for i in range(8):
            p = 3000 + i
            kvc.decode_step(g, 0, p, q[p], k[p], v[p], out=out[i], scratch=scratch)

    loop(eager)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            loop(graph_out)
    for _ in range(2):
        graph_out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(graph_out, eager)
    assert kvc.kvc_device_status() == 0


@pytest.mark.parametrize("cache", ["q8_0", "f16"])
def test_step_up_to_the_last_cache_position(kvc, cache):
    # a cache filled to its last position: the final steps' tile reaches past n_ctx (zero-filled copies)
    n_ctx = 300
    w = si.small_workload("steplast", 40, 8, 128, cache, "bf16", n_prompt=296, chunk=296, n_decode=4, seed=52,
                          n_ctx=n_ctx)
    q, k, v = si.layer_qkv(w, 0)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    g = kvc.KVCache(1, n_ctx, 8, 128, cache, "layer_major")
    kvc.kv_cache_append(g, 0, 0, kd[:296], vd[:296])
    o = OracleCache(1, n_ctx, 8, 128, cache)
    o.append(0, 0, np32(k[:296]), np32(v[:296]))
    for pos in range(296, n_ctx):
        out = kvc.decode_step(g, 0, pos, qd[pos], kd[pos], vd[pos])
        o.append(0, pos, np32(k[pos:pos + 1]), np32(v[pos:pos + 1]))
        assert_close(out.cpu().numpy(), o.decode(0, pos, np32(q[pos])), "pos %d" % pos)
    assert_cache_equal(g, o, n_ctx)
    with pytest.raises(kvc.KvcError):
        kvc.decode_step(g, 0, n_ctx, qd[0], kd[0], vd[0])
    assert kvc.kvc_device_status() == 0
