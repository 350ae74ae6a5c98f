"""prefill_step: a prompt chunk's append and attention in one call, against the two calls it stands
for.  The output equals kv_cache_append + prefill_chunk_attn bit for bit (for q8_0 the fp16 copy of the
chunk is made from the codes just stored), the stored bytes equal the oracle's, sampled rows match the
oracle within the attention tolerance, and rows stay bitwise independent of the chunking."""

import ctypes

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


def partial_scratch(kvc, w, chunk):
    """A q8_0 scratch that holds the partials only (no fp16 copy): the in-kernel dequantiser path;
    its size is the f16 cache's."""
    d16 = kvc.make_desc(1, w.n_ctx, w.n_head_kv, w.head_dim, "f16", "head_major")
    n = ctypes.c_size_t()
    assert kvc.lib.kvc_prefill_scratch_bytes(ctypes.byref(d16), w.n_head_q, chunk, ctypes.byref(n)) == 0
    return torch.empty(n.value, dtype=torch.uint8, device="cuda")


def two_ways(kvc, w, chunk, qkv, scratch_kind="full"):
    """The prompt through append + prefill_chunk_attn (cache a) and through prefill_step (cache b)."""
    q, k, v = (t.cuda() for t in qkv)
    ga = kvc.KVCache(1, w.n_ctx, w.n_head_kv, w.head_dim, w.cache, "head_major")
    gb = kvc.KVCache(1, w.n_ctx, w.n_head_kv, w.head_dim, w.cache, "layer_major")
    sz = chunk if chunk > 0 else w.n_prompt
    if scratch_kind == "full":
        sa, sb = ga.prefill_scratch(w.n_head_q, sz), gb.prefill_scratch(w.n_head_q, sz).fill_(0xA5)
    else:
        sa, sb = partial_scratch(kvc, w, sz), partial_scratch(kvc, w, sz).fill_(0xA5)
    oa = torch.empty(w.n_prompt, w.n_head_q, w.head_dim, device="cuda")
    ob = torch.empty_like(oa)
    for p, c in w.chunks(chunk):
        kvc.kv_cache_append(ga, 0, p, k[p:p + c], v[p:p + c])
        kvc.prefill_chunk_attn(ga, 0, p, q[p:p + c], out=oa[p:p + c], scratch=sa)
        kvc.prefill_step(gb, 0, p, q[p:p + c], k[p:p + c], v[p:p + c], out=ob[p:p + c], scratch=sb)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    return gb, oa, ob


CASES = [
    # H_q, H_kv, D, cache, in dtype, prompt, chunk, scratch
    (8, 2, 128, "q8_0", "bf16", 333, 100, "full"),
    (8, 2, 128, "q8_0", "bf16", 333, 100, "partials"),
    (8, 2, 128, "f16", "bf16", 333, 128, "full"),
    (5, 1, 128, "q8_0", "f16", 260, 129, "full"),
    (4, 2, 64, "q8_0", "f32", 256, 64, "full"),
    (2, 2, 64, "f16", "f32", 140, 7, "full"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%d-%d-%d-%s-%s-%d-%d-%s" % c)
def test_step_equals_append_then_attention(kvc, case):
    hq, hkv, d, cache, dt, n, chunk, kind = case
    w = si.small_workload("pstep", hq, hkv, d, cache, dt, n_prompt=n, chunk=chunk, n_decode=0, seed=n + d + 3,
                          k_outlier_frac=0.01)
    qkv = si.layer_qkv(w, 0)
    gb, oa, ob = two_ways(kvc, w, chunk, qkv, kind)
    assert torch.equal(oa, ob)
    o = OracleCache(1, w.n_ctx, w.n_head_kv, w.head_dim, w.cache)
    q, k, v = qkv
    outs = []
    for p, c in w.chunks(chunk):
        o.append(0, p, np32(k[p:p + c]), np32(v[p:p + c]))
        outs.append(o.prefill_chunk(0, p, np32(q[p:p + c])))
    assert_cache_equal(gb, o, w.n_prompt)
    assert_close(ob.cpu().numpy(), np.concatenate(outs), "prefill_step vs oracle")


@pytest.mark.parametrize("cache,kind", [("q8_0", "full"), ("q8_0", "partials"), ("f16", "full")])
def test_step_with_key_splits(kvc, cache, kind):
    # 9,000 keys at this context size: splits of 4,096 keys, so the later chunks' rows span two or three
    # splits and are merged; the result must equal the separate calls' and stay the same whatever the
    # chunking
    w = si.small_workload("pstepsplit", 10, 2, 128, cache, "bf16", n_prompt=9000, chunk=1024, n_decode=0, seed=33,
                          k_outlier_frac=0.01)
    qkv = si.layer_qkv(w, 0)
    gb, oa, ob = two_ways(kvc, w, 1024, qkv, kind)
    assert torch.equal(oa, ob)
    _, _, oc = two_ways(kvc, w, 3000, qkv, kind)
    assert torch.equal(ob, oc), "chunk invariance"
    o = OracleCache(1, w.n_ctx, w.n_head_kv, w.head_dim, w.cache)
    q, k, v = qkv
    o.append(0, 0, np32(k[:w.n_prompt]), np32(v[:w.n_prompt]))
    assert_cache_equal(gb, o, w.n_prompt)
    rows = si.sample_rows(7, w.chunks(1024))
    kh, vh = o.dequantized(0, w.n_prompt)
    from oracle.attention import attend
    assert_close(ob[rows].cpu().numpy(), attend(np32(q[rows]), rows, kh, vh), "sampled rows")


def test_step_repeated_on_one_scratch(kvc):
    # calling the same chunk again on the same scratch (its copy and partials left by the first call)
    # gives the same bits
    w = si.small_workload("prep", 10, 2, 128, "q8_0", "bf16", n_prompt=6000, chunk=2000, n_decode=0, seed=5)
    q, k, v = (t.cuda() for t in si.layer_qkv(w, 0))
    g = kvc.KVCache(1, w.n_ctx, w.n_head_kv, w.head_dim, "q8_0", "head_major")
    s = g.prefill_scratch(w.n_head_q, 2000)
    kvc.prefill_step(g, 0, 0, q[:2000], k[:2000], v[:2000], scratch=s)
    kvc.prefill_step(g, 0, 2000, q[2000:4000], k[2000:4000], v[2000:4000], scratch=s)
    a = kvc.prefill_step(g, 0, 4000, q[4000:6000], k[4000:6000], v[4000:6000], scratch=s)
    b = kvc.prefill_step(g, 0, 4000, q[4000:6000], k[4000:6000], v[4000:6000], scratch=s)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert kvc.kvc_device_status() == 0


@pytest.mark.parametrize("cache", ["q8_0", "f16"])
def test_step_chunk_ending_at_the_cache_end(kvc, cache):
    # the last chunk fills the cache to n_ctx exactly (the largest copy and plan the scratch was sized for)
    n_ctx = 2600
    w = si.small_workload("pstepend", 10, 2, 128, cache, "bf16", n_prompt=n_ctx, chunk=1000, n_decode=0, seed=61,
                          n_ctx=n_ctx)
    qkv = si.layer_qkv(w, 0)
    gb, oa, ob = two_ways(kvc, w, 1000, qkv)
    assert torch.equal(oa, ob)
    o = OracleCache(1, n_ctx, w.n_head_kv, w.head_dim, cache)
    q, k, v = qkv
    o.append(0, 0, np32(k), np32(v))
    assert_cache_equal(gb, o, n_ctx)
    rows = np.array([0, 999, 1000, 1999, 2000, 2598, 2599])
    kh, vh = o.dequantized(0, n_ctx)
    from oracle.attention import attend
    assert_close(ob[rows].cpu().numpy(), attend(np32(q[rows]), rows, kh, vh), "rows at the end")


def chunked_steps(kvc, g, layer, qkv, chunks, scratch, out, valid):
    """The prompt's chunks through prefill_step; valid(pos0) gives each call's copy_valid."""
    q, k, v = qkv
    for p, c in chunks:
        kvc.prefill_step(g, layer, p, q[p:p + c], k[p:p + c], v[p:p + c], out=out[p:p + c], scratch=scratch,
                         copy_valid=valid(p))


@pytest.mark.parametrize("d,dt", [(128, "bf16"), (64, "f32")])
def test_incremental_copy_equals_the_full_copy(kvc, d, dt):
    # a q8_0 prompt whose chunks each convert only their own positions (copy_valid = pos0), or the
    # positions from part-way back, against calls that convert the whole prefix: the same bits; the
    # scratch starts as fp16 NaNs, so a position of the copy that no call wrote would show
    w = si.small_workload("pinc", 10, 2, d, "q8_0", dt, n_prompt=9000, chunk=1500, n_decode=0, seed=71 + d,
                          k_outlier_frac=0.01)
    qkv = tuple(t.cuda() for t in si.layer_qkv(w, 0))
    chunks = w.chunks(1500)
    outs, caches = [], []
    for valid in (lambda p: 0, lambda p: p, lambda p: max(0, p - 700)):
        g = kvc.KVCache(1, w.n_ctx, w.n_head_kv, d, "q8_0", "head_major")
        s = g.prefill_scratch(w.n_head_q, 1500).fill_(0xFF)
        o = torch.empty(w.n_prompt, w.n_head_q, d, device="cuda")
        chunked_steps(kvc, g, 0, qkv, chunks, s, o, valid)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status() == 0
        outs.append(o)
        caches.append(g)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert not torch.isnan(outs[1]).any()
    n = w.n_prompt
    for g in caches[1:]:
        for kv in (0, 1):
            assert torch.equal(g.codes(kv)[:, 0, :n], caches[0].codes(kv)[:, 0, :n])
            assert torch.equal(g.scales(kv)[:, 0, :n].view(torch.int16), caches[0].scales(kv)[:, 0, :n].view(torch.int16))


def test_incremental_copy_per_layer_with_chunks_through_all_layers(kvc):
    # the model's order: each chunk through every layer before the next chunk, one scratch (one fp16
    # copy) per layer; equals the same order converting the whole prefix every call
    L, n, chunk = 3, 5000, 1024
    w = si.small_workload("pincl", 8, 2, 128, "q8_0", "f16", n_prompt=n, chunk=chunk, n_decode=0, seed=81,
                          n_layer=L)
    qkv = [tuple(t.cuda() for t in si.layer_qkv(w, layer)) for layer in range(L)]
    res = []
    for incremental in (False, True):
        g = kvc.KVCache(L, w.n_ctx, w.n_head_kv, 128, "q8_0", "layer_major")
        scr = [g.prefill_scratch(w.n_head_q, chunk).fill_(0xFF) for _ in range(L)]
        outs = [torch.empty(n, w.n_head_q, 128, device="cuda") for _ in range(L)]
        for p, c in w.chunks(chunk):
            for layer in range(L):
                q, k, v = qkv[layer]
                kvc.prefill_step(g, layer, p, q[p:p + c], k[p:p + c], v[p:p + c], out=outs[layer][p:p + c],
                                 scratch=scr[layer], copy_valid=p if incremental else 0)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status() == 0
        res.append(outs)
    for layer in range(L):
        assert torch.equal(res[0][layer], res[1][layer]), "layer %d" % layer
    o = OracleCache(1, w.n_ctx, w.n_head_kv, 128, "q8_0")
    q, k, v = qkv[2]
    o.append(0, 0, np32(k[:n].cpu()), np32(v[:n].cpu()))
    rows = np.array([0, 1023, 1024, 3000, 4999])
    kh, vh = o.dequantized(0, n)
    from oracle.attention import attend
    assert_close(res[1][2][rows].cpu().numpy(), attend(np32(q[rows].cpu()), rows, kh, vh), "layer 2 rows")


def test_copy_left_by_prefill_chunk_attn(kvc):
    # prefill_chunk_attn's dequantising pass leaves the copy in the same layout: a following prefill_step
    # may take it as valid
    w = si.small_workload("pinca", 10, 2, 128, "q8_0", "bf16", n_prompt=4000, chunk=2000, n_decode=0, seed=91)
    q, k, v = (t.cuda() for t in si.layer_qkv(w, 0))
    ga = kvc.KVCache(1, w.n_ctx, 2, 128, "q8_0", "head_major")
    gb = kvc.KVCache(1, w.n_ctx, 2, 128, "q8_0", "head_major")
    sa = ga.prefill_scratch(10, 2000).fill_(0xFF)
    sb = gb.prefill_scratch(10, 2000)
    kvc.kv_cache_append(ga, 0, 0, k[:2000], v[:2000])
    kvc.prefill_chunk_attn(ga, 0, 0, q[:2000], scratch=sa)
    a = kvc.prefill_step(ga, 0, 2000, q[2000:], k[2000:], v[2000:], scratch=sa, copy_valid=2000)
    kvc.prefill_step(gb, 0, 0, q[:2000], k[:2000], v[:2000], scratch=sb)
    b = kvc.prefill_step(gb, 0, 2000, q[2000:], k[2000:], v[2000:], scratch=sb)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0
    assert torch.equal(a, b)


@pytest.mark.parametrize("cache", ["q8_0", "f16"])
def test_prompt_captured_in_a_cuda_graph(kvc, cache):
    # a whole prompt's prefill_step calls captured once and replayed: each replay's front kernels zero
    # the item counter again, and the outputs equal the eager calls' bit for bit
    w = si.small_workload("pgraph", 10, 2, 128, cache, "bf16", n_prompt=6000, chunk=1500, n_decode=0, seed=97)
    q, k, v = (t.cuda() for t in si.layer_qkv(w, 0))
    g = kvc.KVCache(1, w.n_ctx, 2, 128, cache, "head_major")
    s = g.prefill_scratch(10, 1500)
    eager = torch.empty(w.n_prompt, 10, 128, device="cuda")
    graph_out = torch.empty_like(eager)

    def prompt(out):
        for p, c in w.chunks(1500):
            kvc.prefill_step(g, 0, p, q[p:p + c], k[p:p + c], v[p:p + c], out=out[p:p + c], scratch=s, copy_valid=p)

    prompt(eager)
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            prompt(graph_out)
    for _ in range(2):
        graph_out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(graph_out, eager)
    assert kvc.kvc_device_status() == 0
