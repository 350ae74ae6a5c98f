"""A bounded wait that gives up leaves a usable context.

The pages require that a failure must not lose the request and must leave the
caller a working context (llama.cpp PR #58 "completion : allow the prompt to be
processed under its own split mode", section "Memory"; llama.cpp PR #59 "llama :
switch the split mode of a live context", section "What this adds").  Every
mbarrier wait in the tensor-core kernels is bounded; these tests make one such
wait run out, without any fault: the test hook arms, for the next launch of a
kernel, a wait on a barrier nothing arrives at, with a 2 ms limit.  The kernel
unwinds (copies and MMAs in flight finish, tensor memory is freed), the device
status reports KVC_EDEVICE, and the next normal call on the same cache and
scratch matches the oracle.
"""

import ctypes

import pytest
import torch

import seeded_inputs as si
from oracle.cache import OracleCache
from parity_util import assert_close, np32

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000   # 2 ms


@pytest.fixture(scope="module")
def kvc(cuda_device):
    import decode_attention_kv_cache_gb300 as m
    return m


def _filled(kvc, cache_type, n_prompt):
    w = si.small_workload("fail", 40, 8, 128, cache_type, "bf16", n_prompt=n_prompt, chunk=n_prompt, n_decode=0,
                          seed=31)
    q, k, v = si.layer_qkv(w, 0)
    g = kvc.KVCache(1, w.n_ctx, w.n_head_kv, w.head_dim, cache_type, "head_major")
    kvc.kv_cache_append(g, 0, 0, k.cuda(), v.cuda())
    o = OracleCache(1, w.n_ctx, w.n_head_kv, w.head_dim, cache_type)
    o.append(0, 0, np32(k), np32(v))
    return w, q, g, o


def _status_code(kvc):
    s = ctypes.c_int32(0)
    rc = kvc.lib.kvc_device_status(ctypes.byref(s))
    return rc, s.value


@pytest.mark.parametrize("cache_type", ["q8_0", "f16"])
def test_decode_wait_that_gives_up_then_next_call_is_correct(kvc, cache_type):
    w, q, g, o = _filled(kvc, cache_type, 5000)
    assert kvc.kvc_device_status() == 0
    qd = q.cuda()
    scratch = torch.empty(g.scratch_bytes(w.n_head_q), dtype=torch.uint8, device="cuda")
    pos = w.n_prompt - 1
    kvc.arm_test_wait_timeout(kvc.TEST_DECODE, LIMIT_NS)
    kvc.decode_attn(g, 0, pos, qd[pos], scratch=scratch)
    rc, status = _status_code(kvc)
    assert rc == kvc.KVC_EDEVICE and status != 0, (rc, status)
    assert _status_code(kvc) == (kvc.KVC_OK, 0)          # read and cleared
    for p in (pos, 1234):                                  # the same cache and scratch, calls as usual
        out = kvc.decode_attn(g, 0, p, qd[p], scratch=scratch)
        assert_close(out.cpu().numpy(), o.decode(0, p, np32(q[p])), "decode after the abort, pos %d" % p)
    assert kvc.kvc_device_status() == 0


@pytest.mark.parametrize("cache_type", ["q8_0", "f16"])
def test_decode_step_wait_that_gives_up_then_next_step_is_correct(kvc, cache_type):
    # the fused step: the split pass gives up (after the token was stored); the next steps on the same
    # cache and scratch are correct
    w = si.small_workload("failstep", 40, 8, 128, cache_type, "bf16", n_prompt=5000, chunk=5000, n_decode=2, seed=37)
    q, k, v = si.layer_qkv(w, 0)
    g = kvc.KVCache(1, w.n_ctx, w.n_head_kv, w.head_dim, cache_type, "head_major")
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    kvc.kv_cache_append(g, 0, 0, kd[:5000], vd[:5000])
    o = OracleCache(1, w.n_ctx, w.n_head_kv, w.head_dim, cache_type)
    o.append(0, 0, np32(k[:5000]), np32(v[:5000]))
    scratch = torch.empty(g.scratch_bytes(w.n_head_q), dtype=torch.uint8, device="cuda")
    kvc.arm_test_wait_timeout(kvc.TEST_DECODE, LIMIT_NS)
    kvc.decode_step(g, 0, 5000, qd[5000], kd[5000], vd[5000], scratch=scratch)
    rc, status = _status_code(kvc)
    assert rc == kvc.KVC_EDEVICE and status != 0, (rc, status)
    for p in (5000, 5001):                                 # the aborted step again, then the next one
        out = kvc.decode_step(g, 0, p, qd[p], kd[p], vd[p], scratch=scratch)
        o.append(0, p, np32(k[p:p + 1]), np32(v[p:p + 1]))
        assert_close(out.cpu().numpy(), o.decode(0, p, np32(q[p])), "step after the abort, pos %d" % p)
    assert kvc.kvc_device_status() == 0


@pytest.mark.parametrize("cache_type", ["q8_0", "f16"])
def test_prefill_wait_that_gives_up_then_next_call_is_correct(kvc, cache_type):
    w, q, g, o = _filled(kvc, cache_type, 3000)
    assert kvc.kvc_device_status() == 0
    qd = q.cuda()
    pos0, c = 2000, 1000
    scratch = g.prefill_scratch(w.n_head_q, c)
    kvc.arm_test_wait_timeout(kvc.TEST_PREFILL, LIMIT_NS)
    kvc.prefill_chunk_attn(g, 0, pos0, qd[pos0:pos0 + c], scratch=scratch)
    rc, status = _status_code(kvc)
    assert rc == kvc.KVC_EDEVICE and status != 0, (rc, status)
    out = kvc.prefill_chunk_attn(g, 0, pos0, qd[pos0:pos0 + c], scratch=scratch)
    rows = [0, 1, 127, 128, 511, 998, 999]
    ref = o.prefill_chunk(0, pos0, np32(q[pos0:pos0 + c]), rows=rows)
    assert_close(out.cpu().numpy()[rows], ref, "prefill after the abort")
    assert kvc.kvc_device_status() == 0


@pytest.mark.parametrize("cache_type", ["q8_0", "f16"])
def test_prefill_step_wait_that_gives_up_then_next_call_is_correct(kvc, cache_type):
    # the fused step takes its attention items from a counter: after the aborted call the next one (the
    # same chunk again, then the next chunk, on the same scratch) is correct
    w, q, g, o = _filled(kvc, cache_type, 3000)
    _, k, v = si.layer_qkv(w, 0)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    c = 1000
    scratch = g.prefill_scratch(w.n_head_q, c)
    kvc.prefill_step(g, 0, 0, qd[:c], kd[:c], vd[:c], scratch=scratch)
    kvc.arm_test_wait_timeout(kvc.TEST_PREFILL, LIMIT_NS)
    kvc.prefill_step(g, 0, c, qd[c:2 * c], kd[c:2 * c], vd[c:2 * c], scratch=scratch, copy_valid=c)
    rc, status = _status_code(kvc)
    assert rc == kvc.KVC_EDEVICE and status != 0, (rc, status)
    rows = [0, 1, 127, 128, 511, 998, 999]
    for p0 in (c, 2 * c):
        out = kvc.prefill_step(g, 0, p0, qd[p0:p0 + c], kd[p0:p0 + c], vd[p0:p0 + c], scratch=scratch,
                               copy_valid=p0)
        ref = o.prefill_chunk(0, p0, np32(q[p0:p0 + c]), rows=rows)
        assert_close(out.cpu().numpy()[rows], ref, "prefill_step after the abort, pos0 %d" % p0)
    assert kvc.kvc_device_status() == 0


def test_arm_rejects_an_unknown_kernel(kvc):
    assert kvc.lib.kvc_test_arm_wait_timeout(7, LIMIT_NS) == kvc.KVC_EINVAL
