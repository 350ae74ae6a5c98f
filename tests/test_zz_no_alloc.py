"""decode_attn_noalloc: decode attention for callers that cannot allocate device
memory (for example code hosted by an engine that owns every device allocation,
or a path where cudaMalloc's implicit synchronisation is not allowed).  It keeps
its split-K partials in a fixed device array inside the library instead of a
caller-provided scratch buffer.

Checked through the C ABI on two calls in a row (the second reuses the array's
old contents): bit for bit against decode_attn, which runs the same kernels with
a caller scratch, and within the attention tolerance against the oracle.  The
file name sorts last so that a run stopping at its first failure has run every
other test first; the tests set up everything they use and pass when run alone.
"""

import ctypes

import numpy as np
import pytest
import torch

import seeded_inputs as si
from oracle.cache import OracleCache
from parity_util import assert_close, np32

pytestmark = pytest.mark.gpu


def _entry(kvc):
    lib = ctypes.CDLL(kvc.LIB_PATH)
    f = lib.decode_attn_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(kvc.kvc_cache), ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    return f


# (H_q, H_kv, head_dim, prompt tokens, positions decoded): head_dim 128 runs the tensor-core split
# pass, head_dim 64 the mma.sync one; both keep their partials in the library's array
CASES = [(40, 8, 128, 3000, (2999, 1234)), (4, 2, 64, 700, (699, 300))]


@pytest.mark.parametrize("cache_type", ["q8_0", "f16"])
@pytest.mark.parametrize("shape", CASES, ids=["d128", "d64"])
def test_noalloc_decode_matches_decode_attn_and_oracle(cuda_device, cache_type, shape):
    import decode_attention_kv_cache_gb300 as kvc
    f = _entry(kvc)
    n_head_q, n_head_kv, head_dim, n_prompt, positions = shape
    w = si.small_workload("na", n_head_q, n_head_kv, head_dim, cache_type, "bf16", n_prompt=n_prompt,
                          chunk=n_prompt, n_decode=0, seed=77)
    q, k, v = si.layer_qkv(w, 0)
    g = kvc.KVCache(1, w.n_ctx, w.n_head_kv, w.head_dim, cache_type, "head_major")
    kvc.kv_cache_append(g, 0, 0, k.cuda(), v.cuda())
    o = OracleCache(1, w.n_ctx, w.n_head_kv, w.head_dim, cache_type)
    o.append(0, 0, np32(k), np32(v))
    qd = q.cuda()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for pos in positions:
        out = torch.empty(w.n_head_q, w.head_dim, device="cuda")
        rc = f(ctypes.byref(g.c), 0, pos, ctypes.c_void_p(qd[pos].data_ptr()), 1, w.n_head_q,
               ctypes.c_void_p(out.data_ptr()), stream)
        assert rc == kvc.KVC_OK
        ref = kvc.decode_attn(g, 0, pos, qd[pos])
        torch.cuda.synchronize()
        assert torch.equal(out, ref), "noalloc differs from decode_attn at pos %d" % pos
        assert_close(out.cpu().numpy(), o.decode(0, pos, np32(q[pos])), "noalloc vs oracle, pos %d" % pos)
    assert kvc.kvc_device_status() == 0


def test_noalloc_rejects_more_heads_than_the_array_holds(cuda_device):
    import decode_attention_kv_cache_gb300 as kvc
    f = _entry(kvc)
    g = kvc.KVCache(1, 64, 64, 128, "q8_0", "head_major")   # 64 kv heads: 64 query heads need > 8 MiB
    q = torch.zeros(64, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(64, 128, device="cuda")
    rc = f(ctypes.byref(g.c), 0, 3, ctypes.c_void_p(q.data_ptr()), 1, 64, ctypes.c_void_p(out.data_ptr()),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == kvc.KVC_ENOSPC


def test_noalloc_rejects_an_output_in_host_memory(cuda_device):
    import decode_attention_kv_cache_gb300 as kvc
    f = _entry(kvc)
    g = kvc.KVCache(1, 64, 2, 64, "q8_0", "head_major")
    q = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.full((4, 64), 7.0).pin_memory()   # not memory of the current device (a known value: no NaN)
    before = out.clone()
    rc = f(ctypes.byref(g.c), 0, 3, ctypes.c_void_p(q.data_ptr()), 1, 4, ctypes.c_void_p(out.data_ptr()),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == kvc.KVC_EINVAL
    assert torch.equal(out, before)
