"""prefill_chunk_attn on the GPU: within tolerance of the oracle, and bitwise
independent of the chunking and of the cache layout."""

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


def gpu_prefill(kvc, w, layout, chunk, layer=0, qkv=None):
    g = kvc.KVCache(w.n_layer, w.n_ctx, w.n_head_kv, w.head_dim, w.cache, layout)
    q, k, v = qkv if qkv is not None else si.layer_qkv(w, layer)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty(w.n_prompt, w.n_head_q, w.head_dim, device="cuda")
    scratch = g.prefill_scratch(w.n_head_q, chunk if chunk > 0 else w.n_prompt)  # reused by every chunk
    for p, c in w.chunks(chunk):
        kvc.kv_cache_append(g, layer, p, kd[p:p + c], vd[p:p + c])
        kvc.prefill_chunk_attn(g, layer, p, qd[p:p + c], out=out[p:p + c], scratch=scratch)
    torch.cuda.synchronize()
    return g, out


def oracle_prefill(w, chunk, layer=0, qkv=None):
    o = OracleCache(w.n_layer, w.n_ctx, w.n_head_kv, w.head_dim, w.cache)
    q, k, v = qkv if qkv is not None else si.layer_qkv(w, layer)
    outs = []
    for p, c in w.chunks(chunk):
        o.append(layer, p, np32(k[p:p + c]), np32(v[p:p + c]))
        outs.append(o.prefill_chunk(layer, p, np32(q[p:p + c])))
    return o, np.concatenate(outs)


CASES = [
    # H_q, H_kv, D, cache, in dtype, prompt, chunk
    (4, 2, 64, "q8_0", "f32", 256, 64),
    (8, 2, 128, "q8_0", "bf16", 333, 100),
    (8, 2, 128, "f16", "bf16", 333, 128),
    (5, 1, 128, "q8_0", "f16", 260, 129),
    (2, 2, 64, "f16", "f32", 140, 7),
    (10, 2, 128, "q8_0", "bf16", 520, 520),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%d-%d-%d-%s-%s-%d-%d" % c)
def test_prefill_matches_oracle(kvc, case):
    hq, hkv, d, cache, dt, n, chunk = case
    w = si.small_workload("pf", hq, hkv, d, cache, dt, n_prompt=n, chunk=chunk, n_decode=0, seed=n + d,
                          k_outlier_frac=0.02)
    g, out = gpu_prefill(kvc, w, "head_major", chunk)
    o, ref = oracle_prefill(w, chunk)
    assert_cache_equal(g, o, n)
    assert_close(out.cpu().numpy(), ref, "prefill")


def test_prefill_chunk_and_layout_invariance(kvc):
    w = si.small_workload("inv", 10, 2, 128, "q8_0", "bf16", n_prompt=700, chunk=0, n_decode=0, seed=21)
    qkv = si.layer_qkv(w, 0)
    _, whole = gpu_prefill(kvc, w, "head_major", 0, qkv=qkv)
    for _ in range(3):  # repeat runs: the result must be deterministic
        assert torch.equal(gpu_prefill(kvc, w, "layer_major", 0, qkv=qkv)[1], whole)
    for chunk in (1, 37, 128, 300):
        for layout in ("head_major", "layer_major"):
            if chunk == 1 and layout == "layer_major":
                continue
            _, out = gpu_prefill(kvc, w, layout, chunk, qkv=qkv)
            assert torch.equal(out, whole), "chunk %d %s changed the result" % (chunk, layout)
    _, ref = oracle_prefill(w, 0, qkv=qkv)
    assert_close(whole.cpu().numpy(), ref)


def test_prefill_f16_cache_invariance(kvc):
    w = si.small_workload("inv16", 8, 8, 64, "f16", "bf16", n_prompt=400, chunk=0, n_decode=0, seed=22)
    qkv = si.layer_qkv(w, 0)
    _, whole = gpu_prefill(kvc, w, "layer_major", 0, qkv=qkv)
    _, out = gpu_prefill(kvc, w, "head_major", 96, qkv=qkv)
    assert torch.equal(out, whole)


def test_prefill_other_layer_and_repeatability(kvc):
    w = si.small_workload("lay", 8, 2, 128, "f16", "bf16", n_prompt=300, chunk=150, n_decode=0, seed=23, n_layer=2)
    qkv = si.layer_qkv(w, 1)
    _, a = gpu_prefill(kvc, w, "head_major", 150, layer=1, qkv=qkv)
    _, b = gpu_prefill(kvc, w, "head_major", 150, layer=1, qkv=qkv)
    assert torch.equal(a, b)
    _, ref = oracle_prefill(w, 150, layer=1, qkv=qkv)
    assert_close(a.cpu().numpy(), ref)
    assert kvc.kvc_device_status() == 0


def test_prefill_key_splits_merge_and_stay_chunk_invariant(kvc):
    # 9,000 keys: the splits (4,096 keys at this context size) are merged in split order; rows of one
    # chunking and another must agree bit for bit, and sampled rows must match the oracle
    w = si.small_workload("split", 10, 2, 128, "q8_0", "bf16", n_prompt=9000, chunk=1024, n_decode=0, seed=31,
                          k_outlier_frac=0.01)
    qkv = si.layer_qkv(w, 0)
    _, a = gpu_prefill(kvc, w, "head_major", 1024, qkv=qkv)
    for chunk, layout in ((3000, "layer_major"), (1024, "head_major"), (0, "head_major"), (257, "layer_major")):
        _, b = gpu_prefill(kvc, w, layout, chunk, qkv=qkv)
        assert torch.equal(a, b), "chunk %d %s" % (chunk, layout)
    o = OracleCache(1, w.n_ctx, w.n_head_kv, w.head_dim, w.cache)
    q, k, v = qkv
    o.append(0, 0, np32(k[:w.n_prompt]), np32(v[:w.n_prompt]))
    rows = si.sample_rows(5, w.chunks(1024))
    kh, vh = o.dequantized(0, w.n_prompt)
    from oracle.attention import attend
    ref = attend(np32(q[rows]), rows, kh, vh)
    assert_close(a[rows].cpu().numpy(), ref, "sampled rows")
    assert kvc.kvc_device_status() == 0


def test_scratch_reused_after_a_short_chunk(kvc):
    # a scratch buffer reused across calls with different work shapes (a short chunk, then long
    # chunks with key splits) gives the results of a fresh buffer filled with garbage
    w = si.small_workload("reuse", 10, 2, 128, "f16", "bf16", n_prompt=9000, chunk=1024, n_decode=0, seed=41)
    q, k, v = (t.cuda() for t in si.layer_qkv(w, 0))
    g = kvc.KVCache(1, w.n_ctx, w.n_head_kv, w.head_dim, w.cache, "head_major")
    kvc.kv_cache_append(g, 0, 0, k[:w.n_prompt], v[:w.n_prompt])
    shared = g.prefill_scratch(w.n_head_q, 1024)
    kvc.prefill_chunk_attn(g, 0, 8900, q[8900:9000], scratch=shared)          # short chunk, key splits
    for p in (6000, 7000, 7976):
        a = kvc.prefill_chunk_attn(g, 0, p, q[p:p + 1024], scratch=shared)
        fresh = g.prefill_scratch(w.n_head_q, 1024).fill_(0xA5)
        b = kvc.prefill_chunk_attn(g, 0, p, q[p:p + 1024], scratch=fresh)
        assert torch.equal(a, b), "chunk at %d" % p


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f32")])
def test_q8_0_dequantised_copy_and_in_kernel_dequant_agree_bitwise(kvc, d, dtype):
    # the full scratch dequantises the attended keys once and attends over that fp16 copy; a scratch
    # holding only the partials makes the attention kernel dequantise each tile in shared memory.
    # Both enter fp16(d * q) into the same products in the same order.
    w = si.small_workload("twopath", 10, 2, d, "q8_0", "bf16" if dtype == "bf16" else "f32", n_prompt=5000,
                          chunk=1000, n_decode=0, seed=91, k_outlier_frac=0.01)
    q, k, v = (t.cuda() for t in si.layer_qkv(w, 0))
    g = kvc.KVCache(1, w.n_ctx, w.n_head_kv, w.head_dim, "q8_0", "head_major")
    full = g.prefill_scratch(w.n_head_q, 1000)
    d16 = kvc.make_desc(1, w.n_ctx, w.n_head_kv, w.head_dim, "f16", "head_major")
    n = ctypes.c_size_t()
    assert kvc.lib.kvc_prefill_scratch_bytes(ctypes.byref(d16), w.n_head_q, 1000, ctypes.byref(n)) == 0
    small = torch.empty(n.value, dtype=torch.uint8, device="cuda")
    assert small.numel() < full.numel()
    outs = []
    for scratch in (full, small):
        out = torch.empty(w.n_prompt, w.n_head_q, w.head_dim, device="cuda")
        for p, c in w.chunks(1000):
            kvc.kv_cache_append(g, 0, p, k[p:p + c], v[p:p + c])
            kvc.prefill_chunk_attn(g, 0, p, q[p:p + c], out=out[p:p + c], scratch=scratch)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    assert kvc.kvc_device_status() == 0
