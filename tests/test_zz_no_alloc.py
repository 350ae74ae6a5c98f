"""decode_attn_noalloc: decode attention for callers that cannot allocate device
memory (for example code hosted by an engine that owns every device allocation,
or a path where cudaMalloc's implicit synchronisation is not allowed).  It keeps
its split-K partials in a fixed device array inside the library instead of a
caller-provided scratch buffer.  Checked through the C ABI against decode_attn
on two calls in a row; this file is collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

import seeded_inputs as si
from parity_util import assert_close

pytestmark = pytest.mark.gpu


def _entry(kvc):
    lib = ctypes.CDLL(kvc.LIB_PATH)
    f = lib.decode_attn_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(kvc.kvc_cache), ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    return f


def test_noalloc_decode_matches_decode_attn(cuda_device):
    import decode_attention_kv_cache_gb300 as kvc
    f = _entry(kvc)
    for cache_type in ("q8_0", "f16"):
        w = si.small_workload("na", 40, 8, 128, cache_type, "bf16", n_prompt=3000, chunk=3000, n_decode=0, seed=77)
        q, k, v = si.layer_qkv(w, 0)
        g = kvc.KVCache(1, w.n_ctx, w.n_head_kv, w.head_dim, cache_type, "head_major")
        kvc.kv_cache_append(g, 0, 0, k.cuda(), v.cuda())
        qd = q.cuda()
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        for pos in (2999, 1234):   # two calls in a row, the second reusing the array's old contents
            out = torch.empty(w.n_head_q, w.head_dim, device="cuda")
            rc = f(ctypes.byref(g.c), 0, pos, ctypes.c_void_p(qd[pos].data_ptr()), 1, w.n_head_q,
                   ctypes.c_void_p(out.data_ptr()), stream)
            assert rc == kvc.KVC_OK
            ref = kvc.decode_attn(g, 0, pos, qd[pos])
            torch.cuda.synchronize()
            assert_close(out.cpu().numpy(), ref.cpu().numpy(), "noalloc pos %d" % pos)
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
