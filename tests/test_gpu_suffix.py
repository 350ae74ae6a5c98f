"""Suffix prefill from a restored state: the prompt's first n0 tokens are prefilled into
one cache, serialised, restored into a cache of the other layout, and only the remaining
tokens are then appended and prefilled there.  The rows of the suffix must equal, bit for
bit, the rows of one prefill of the whole prompt, and so must the cache (this is the
cache-hit path that a saved sequence state exists for: the restored prefix is never
recomputed)."""

import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle.attention import attend
from oracle.cache import OracleCache
from parity_util import assert_close, np32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc(cuda_device):
    import decode_attention_kv_cache_gb300 as m
    return m


def prefill(kvc, g, qkv, start, stop, chunk, out):
    qd, kd, vd = qkv
    scratch = g.prefill_scratch(qd.shape[1], chunk)
    for p in range(start, stop, chunk):
        c = min(chunk, stop - p)
        kvc.kv_cache_append(g, 0, p, kd[p:p + c], vd[p:p + c])
        kvc.prefill_chunk_attn(g, 0, p, qd[p:p + c], out=out[p:p + c], scratch=scratch)


# cache type, prompt, prefix length, chunk (the prefix ends inside a 256-key tile and a key split)
CASES = [("q8_0", 9000, 5003, 1024), ("f16", 6100, 4477, 512), ("q8_0", 700, 1, 256)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s-%d-%d-%d" % c)
def test_suffix_prefill_after_restore_equals_full_prefill(kvc, case):
    cache, n, n0, chunk = case
    w = si.small_workload("suffix", 10, 2, 128, cache, "bf16", n_prompt=n, chunk=chunk, n_decode=0, seed=n0,
                          k_outlier_frac=0.01)
    q, k, v = si.layer_qkv(w, 0)
    qkv = tuple(t.cuda() for t in (q, k, v))
    full = kvc.KVCache(1, w.n_ctx, w.n_head_kv, w.head_dim, cache, "head_major")
    out_full = torch.empty(n, w.n_head_q, w.head_dim, device="cuda")
    prefill(kvc, full, qkv, 0, n, chunk, out_full)

    # the prefix in its own cache, serialised after its last chunk
    first = kvc.KVCache(1, w.n_ctx, w.n_head_kv, w.head_dim, cache, "head_major")
    out_first = torch.empty(n, w.n_head_q, w.head_dim, device="cuda")
    prefill(kvc, first, qkv, 0, n0, chunk, out_first)
    state = kvc.kv_state_get(first, n0)
    restored = kvc.KVCache(1, w.n_ctx, w.n_head_kv, w.head_dim, cache, "layer_major")
    assert kvc.kv_state_set(restored, state) == n0
    out_suffix = torch.full((n, w.n_head_q, w.head_dim), float("nan"), device="cuda")
    prefill(kvc, restored, qkv, n0, n, chunk, out_suffix)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status() == 0

    assert torch.equal(out_suffix[n0:], out_full[n0:])
    assert torch.equal(out_first[:n0], out_full[:n0])
    for kv in (0, 1):
        assert torch.equal(restored.codes(kv)[:, :n].permute(2, 0, 1, 3), full.codes(kv)[:, :, :n])
        if cache == "q8_0":
            assert torch.equal(restored.scales(kv)[:, :n].permute(2, 0, 1, 3), full.scales(kv)[:, :, :n])

    # sampled suffix rows against the oracle
    o = OracleCache(1, w.n_ctx, w.n_head_kv, w.head_dim, cache)
    o.append(0, 0, np32(k[:n]), np32(v[:n]))
    kh, vh = o.dequantized(0, n)
    rng = np.random.default_rng(n0)
    rows = np.unique(np.concatenate([[n0, n0 + 1, n - 1], rng.integers(n0, n, 5)]))
    rows = rows[rows < n]
    assert_close(out_suffix[rows].cpu().numpy(), attend(np32(q[rows]), rows, kh, vh), "suffix rows")
