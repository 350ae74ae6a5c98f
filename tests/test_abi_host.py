"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, and its host-side checks and size queries behave as
documented (no call here reaches CUDA)."""

import ctypes
import os
import re

import pytest

from oracle import state as ostate

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvc.h")


@pytest.fixture(scope="module")
def kvc():
    from decode_attention_kv_cache_gb300 import build as b
    if not os.path.exists(b.LIB):
        b.build()
    import decode_attention_kv_cache_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\([^;{]*\)\s*;", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ["kv_cache_append", "prefill_chunk_attn", "decode_attn", "kv_state_get", "kv_state_set",
              "kv_state_size", "kvc_cache_bytes", "kvc_scratch_bytes", "kvc_prefill_scratch_bytes",
              "kvc_cache_init", "kvc_strerror", "kvc_device_status"]:
        assert n in names


def test_library_exports_every_declared_symbol(kvc):
    lib = ctypes.CDLL(kvc.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing


def test_cache_bytes(kvc):
    d = kvc.make_desc(64, 32768, 8, 128, "q8_0", "head_major")
    kq, ks, vq, vs = kvc.cache_bytes(d)
    n = 64 * 32768 * 8 * 128
    assert (kq, ks, vq, vs) == (n, n // 16, n, n // 16)
    d = kvc.make_desc(1, 20480, 8, 128, "f16", "layer_major")
    assert kvc.cache_bytes(d) == (2 * 20480 * 1024, 0, 2 * 20480 * 1024, 0)


@pytest.mark.parametrize("shape", [(1, 512, 2, 64, "q8_0"), (64, 32768, 8, 128, "q8_0"), (1, 20480, 8, 128, "f16"),
                                   (3, 40, 1, 32, "q8_0"), (2, 9, 3, 96, "f16")])
def test_state_size_agrees_with_the_oracle(kvc, shape):
    L, T, H, D, ct = shape
    d = kvc.make_desc(L, T, H, D, ct)
    for n in (0, 1, 7, T):
        assert kvc.lib.kv_state_size(ctypes.byref(d), n) == ostate.state_size(L, H, D, ct, n)
    assert kvc.lib.kv_state_size(ctypes.byref(d), T + 1) == 0
    assert kvc.lib.kv_state_size(ctypes.byref(d), -1) == 0


def test_invalid_descriptors(kvc):
    out = ctypes.c_size_t()
    for bad in [kvc.make_desc(1, 16, 2, 48), kvc.make_desc(0, 16, 2, 64), kvc.make_desc(1, 16, 0, 64),
                kvc.kvc_desc(1, 16, 2, 64, 7, 0), kvc.kvc_desc(1, 16, 2, 64, 1, 5)]:
        s = [ctypes.c_size_t() for _ in range(4)]
        assert kvc.lib.kvc_cache_bytes(ctypes.byref(bad), *[ctypes.byref(x) for x in s]) == kvc.KVC_EINVAL
    d = kvc.make_desc(1, 16, 2, 64)
    assert kvc.lib.kvc_scratch_bytes(ctypes.byref(d), 3, ctypes.byref(out)) == kvc.KVC_EINVAL
    assert kvc.lib.kvc_scratch_bytes(ctypes.byref(d), 4, ctypes.byref(out)) == kvc.KVC_OK
    assert out.value == 4 * 256 * 66 * 4


def _fake_cache(kvc, cache_type="q8_0", misalign=0):
    c = kvc.kvc_cache()
    d = kvc.make_desc(2, 64, 2, 64, cache_type)
    p = [ctypes.c_void_p(0x10000 * (i + 1) + misalign) for i in range(4)]
    rc = kvc.lib.kvc_cache_init(ctypes.byref(c), ctypes.byref(d), *p)
    return rc, c


def test_cache_init_checks(kvc):
    assert _fake_cache(kvc)[0] == kvc.KVC_OK
    assert _fake_cache(kvc, misalign=8)[0] == kvc.KVC_EINVAL
    c = kvc.kvc_cache()
    d = kvc.make_desc(2, 64, 2, 64, "q8_0")
    assert kvc.lib.kvc_cache_init(ctypes.byref(c), ctypes.byref(d), ctypes.c_void_p(0x10000), None,
                                  ctypes.c_void_p(0x20000), None) == kvc.KVC_EINVAL
    d = kvc.make_desc(2, 64, 2, 64, "f16")   # f16 needs no scale buffers
    assert kvc.lib.kvc_cache_init(ctypes.byref(c), ctypes.byref(d), ctypes.c_void_p(0x10000), None,
                                  ctypes.c_void_p(0x20000), None) == kvc.KVC_OK


def test_hot_path_checks_run_before_any_launch(kvc):
    _, c = _fake_cache(kvc)
    k = ctypes.c_void_p(0x40000)
    S = None
    assert kvc.lib.kv_cache_append(ctypes.byref(c), 2, 0, 4, k, k, 1, S) == kvc.KVC_ERANGE
    assert kvc.lib.kv_cache_append(ctypes.byref(c), 0, 62, 4, k, k, 1, S) == kvc.KVC_ERANGE
    assert kvc.lib.kv_cache_append(ctypes.byref(c), 0, -1, 4, k, k, 1, S) == kvc.KVC_ERANGE
    assert kvc.lib.kv_cache_append(ctypes.byref(c), 0, 0, 4, k, k, 9, S) == kvc.KVC_EINVAL
    assert kvc.lib.kv_cache_append(ctypes.byref(c), 0, 0, 4, None, k, 1, S) == kvc.KVC_EINVAL
    assert kvc.lib.kv_cache_append(ctypes.byref(c), 0, 10, 0, None, None, 1, S) == kvc.KVC_OK  # empty: no-op
    assert kvc.lib.prefill_chunk_attn(ctypes.byref(c), 0, 60, 5, k, 1, 4, k, k, 1 << 30, S) == kvc.KVC_ERANGE
    assert kvc.lib.prefill_chunk_attn(ctypes.byref(c), 0, 0, 5, k, 1, 3, k, k, 1 << 30, S) == kvc.KVC_EINVAL
    assert kvc.lib.prefill_chunk_attn(ctypes.byref(c), 0, 0, 5, k, 1, 4, k, None, 1 << 30, S) == kvc.KVC_EINVAL
    assert kvc.lib.prefill_chunk_attn(ctypes.byref(c), 0, 0, 5, k, 1, 4, k, k, 16, S) == kvc.KVC_ENOSPC
    assert kvc.lib.prefill_chunk_attn(ctypes.byref(c), 0, 3, 0, None, 1, 4, None, None, 0, S) == kvc.KVC_OK
    # the fused prefill step: prefill_chunk_attn's checks plus k and v
    assert kvc.lib.prefill_step(ctypes.byref(c), 0, 60, 5, k, k, k, 1, 4, k, k, 1 << 30, 0, S) == kvc.KVC_ERANGE
    assert kvc.lib.prefill_step(ctypes.byref(c), 0, 0, 5, k, None, k, 1, 4, k, k, 1 << 30, 0, S) == kvc.KVC_EINVAL
    assert kvc.lib.prefill_step(ctypes.byref(c), 0, 0, 5, k, k, ctypes.c_void_p(0x40004), 1, 4, k, k, 1 << 30, 0, S) == \
        kvc.KVC_EINVAL
    assert kvc.lib.prefill_step(ctypes.byref(c), 0, 0, 5, k, k, k, 1, 3, k, k, 1 << 30, 0, S) == kvc.KVC_EINVAL
    assert kvc.lib.prefill_step(ctypes.byref(c), 0, 0, 5, k, k, k, 1, 4, k, k, 16, 0, S) == kvc.KVC_ENOSPC
    assert kvc.lib.prefill_step(ctypes.byref(c), 0, 3, 0, None, None, None, 1, 4, None, None, 0, 0, S) == kvc.KVC_OK
    # copy_valid within [0, pos0]
    assert kvc.lib.prefill_step(ctypes.byref(c), 0, 8, 5, k, k, k, 1, 4, k, k, 1 << 30, 9, S) == kvc.KVC_ERANGE
    assert kvc.lib.prefill_step(ctypes.byref(c), 0, 8, 5, k, k, k, 1, 4, k, k, 1 << 30, -1, S) == kvc.KVC_ERANGE
    assert kvc.lib.decode_attn(ctypes.byref(c), 0, 64, k, 1, 4, k, k, 1 << 20, S) == kvc.KVC_ERANGE
    assert kvc.lib.decode_attn(ctypes.byref(c), 0, 5, k, 1, 4, k, k, 100, S) == kvc.KVC_ENOSPC
    assert kvc.lib.decode_attn(ctypes.byref(c), 0, 5, k, 1, 36, k, k, 1 << 24, S) == kvc.KVC_EINVAL  # G = 18 > 16
    assert kvc.lib.kv_state_get(ctypes.byref(c), 65, k, 1 << 20, S) == kvc.KVC_ERANGE
    assert kvc.lib.kv_state_get(ctypes.byref(c), 10, k, 100, S) == kvc.KVC_ENOSPC
    assert kvc.lib.kv_state_set(ctypes.byref(c), k, 16, ctypes.byref(ctypes.c_int32()), S) == kvc.KVC_EFORMAT
    assert kvc.lib.kv_cache_truncate(ctypes.byref(c), 65, S) == kvc.KVC_ERANGE
    assert kvc.lib.kv_cache_truncate(ctypes.byref(c), -1, S) == kvc.KVC_ERANGE
    assert kvc.lib.kv_cache_truncate(ctypes.byref(c), 64, S) == kvc.KVC_OK      # nothing past n_ctx: no-op
    assert kvc.lib.kv_cache_truncate(None, 0, S) == kvc.KVC_EINVAL
    # a head range of a split cache (c holds 2 kv heads)
    assert kvc.lib.kv_state_get_heads(ctypes.byref(c), 1, 2, 10, k, 1 << 20, S) == kvc.KVC_EINVAL   # 1 + 2 > 2
    assert kvc.lib.kv_state_get_heads(ctypes.byref(c), -1, 4, 10, k, 1 << 20, S) == kvc.KVC_EINVAL
    assert kvc.lib.kv_state_get_heads(ctypes.byref(c), 2, 4, 65, k, 1 << 20, S) == kvc.KVC_ERANGE
    assert kvc.lib.kv_state_get_heads(ctypes.byref(c), 2, 4, 10, k, 100, S) == kvc.KVC_ENOSPC
    assert kvc.lib.kv_state_set_heads(ctypes.byref(c), -1, k, 1 << 20, ctypes.byref(ctypes.c_int32()), S) == \
        kvc.KVC_EINVAL
    assert kvc.lib.kv_state_set_heads(ctypes.byref(c), 0, k, 16, ctypes.byref(ctypes.c_int32()), S) == kvc.KVC_EFORMAT
    # batched decode: the checks of decode_attn per sequence, plus the batch's own
    big = 1 << 30
    d128 = kvc.make_desc(2, 64, 2, 128, "q8_0")
    cb = kvc.kvc_cache()
    p4 = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(4)]
    assert kvc.lib.kvc_cache_init(ctypes.byref(cb), ctypes.byref(d128), *p4) == kvc.KVC_OK
    nine = (kvc.kvc_cache * 9)(*([cb] * 9))
    p9 = (ctypes.c_int32 * 9)(*([5] * 9))
    assert kvc.lib.decode_attn_batch(nine, 9, 0, p9, k, 1, 4, k, k, big, S) == kvc.KVC_EINVAL     # n_seq > 8
    assert kvc.lib.decode_attn_batch(nine, 0, 0, p9, k, 1, 4, k, k, big, S) == kvc.KVC_EINVAL     # n_seq < 1
    bad = (ctypes.c_int32 * 2)(5, 64)
    assert kvc.lib.decode_attn_batch(nine, 2, 0, bad, k, 1, 4, k, k, big, S) == kvc.KVC_ERANGE    # pos[1] = n_ctx
    assert kvc.lib.decode_attn_batch(nine, 2, 2, p9, k, 1, 4, k, k, big, S) == kvc.KVC_ERANGE     # layer
    assert kvc.lib.decode_attn_batch(nine, 2, 0, p9, k, 1, 3, k, k, big, S) == kvc.KVC_EINVAL     # n_head_q
    one = ctypes.c_size_t()
    assert kvc.lib.kvc_scratch_bytes(ctypes.byref(d128), 4, ctypes.byref(one)) == kvc.KVC_OK
    assert kvc.lib.decode_attn_batch(nine, 3, 0, p9, k, 1, 4, k, k, 3 * one.value - 16, S) == kvc.KVC_ENOSPC
    mixed = (kvc.kvc_cache * 2)(cb, c)                                                            # head_dim 128 and 64
    assert kvc.lib.decode_attn_batch(mixed, 2, 0, p9, k, 1, 4, k, k, big, S) == kvc.KVC_EINVAL
    # the fused step: decode_attn's checks plus k and v
    assert kvc.lib.decode_step(ctypes.byref(c), 0, 64, k, k, k, 1, 4, k, k, big, S) == kvc.KVC_ERANGE      # pos
    assert kvc.lib.decode_step(ctypes.byref(c), 2, 5, k, k, k, 1, 4, k, k, big, S) == kvc.KVC_ERANGE       # layer
    assert kvc.lib.decode_step(ctypes.byref(c), 0, 5, k, None, k, 1, 4, k, k, big, S) == kvc.KVC_EINVAL    # k
    assert kvc.lib.decode_step(ctypes.byref(c), 0, 5, k, k, ctypes.c_void_p(0x40008), 1, 4, k, k, big, S) == \
        kvc.KVC_EINVAL                                                                                    # unaligned v
    assert kvc.lib.decode_step(ctypes.byref(c), 0, 5, k, k, k, 1, 3, k, k, big, S) == kvc.KVC_EINVAL       # n_head_q
    assert kvc.lib.decode_step(ctypes.byref(c), 0, 5, k, k, k, 7, 4, k, k, big, S) == kvc.KVC_EINVAL       # dtype
    assert kvc.lib.decode_step(ctypes.byref(c), 0, 5, k, k, k, 1, 4, k, k, 100, S) == kvc.KVC_ENOSPC
    assert kvc.lib.decode_step_batch(nine, 9, 0, p9, k, k, k, 1, 4, k, k, big, S) == kvc.KVC_EINVAL    # n_seq > 8
    assert kvc.lib.decode_step_batch(nine, 2, 0, bad, k, k, k, 1, 4, k, k, big, S) == kvc.KVC_ERANGE   # pos[1]
    assert kvc.lib.decode_step_batch(mixed, 2, 0, p9, k, k, k, 1, 4, k, k, big, S) == kvc.KVC_EINVAL
    assert kvc.lib.decode_step_batch(nine, 2, 0, p9, k, None, k, 1, 4, k, k, big, S) == kvc.KVC_EINVAL
    assert kvc.lib.decode_step_batch(nine, 3, 0, p9, k, k, k, 1, 4, k, k, 3 * one.value - 16, S) == kvc.KVC_ENOSPC
    # batched append
    assert kvc.lib.kv_cache_append_batch(nine, 9, 0, p9, k, k, 1, S) == kvc.KVC_EINVAL           # n_seq > 8
    assert kvc.lib.kv_cache_append_batch(nine, 2, 0, bad, k, k, 1, S) == kvc.KVC_ERANGE          # pos[1] = n_ctx
    assert kvc.lib.kv_cache_append_batch(nine, 2, 2, p9, k, k, 1, S) == kvc.KVC_ERANGE           # layer
    assert kvc.lib.kv_cache_append_batch(mixed, 2, 0, p9, k, k, 1, S) == kvc.KVC_EINVAL
    assert kvc.lib.kv_cache_append_batch(nine, 2, 0, p9, None, k, 1, S) == kvc.KVC_EINVAL
    assert kvc.lib.kv_cache_append_batch(nine, 2, 0, p9, k, k, 7, S) == kvc.KVC_EINVAL           # dtype
    # unsupported head_dim for attention (append and state accept any multiple of 32)
    c96 = kvc.kvc_cache()
    d96 = kvc.make_desc(1, 64, 2, 96, "f16")
    assert kvc.lib.kvc_cache_init(ctypes.byref(c96), ctypes.byref(d96), k, None, k, None) == kvc.KVC_OK
    assert kvc.lib.prefill_chunk_attn(ctypes.byref(c96), 0, 0, 5, k, 1, 4, k, k, 1 << 30, S) == kvc.KVC_EINVAL


def test_prefill_scratch_query(kvc):
    out = ctypes.c_size_t()
    d = kvc.make_desc(1, 65536, 8, 128, "q8_0")
    assert kvc.lib.kvc_prefill_scratch_bytes(ctypes.byref(d), 40, 2048, ctypes.byref(out)) == kvc.KVC_OK
    big = out.value
    # 8 kv groups x 40 pairs x 4 splits x 2 tiles x 128 rows x 130 floats
    assert big >= 8 * 40 * 4 * 2 * 128 * 130 * 4
    assert kvc.lib.kvc_prefill_scratch_bytes(ctypes.byref(d), 40, 512, ctypes.byref(out)) == kvc.KVC_OK
    assert out.value < big
    small = kvc.make_desc(1, 512, 2, 64, "q8_0")
    assert kvc.lib.kvc_prefill_scratch_bytes(ctypes.byref(small), 4, 64, ctypes.byref(out)) == kvc.KVC_OK
    # one split: no partials, the minimum 256 bytes, behind the fp16 copy of K and V (2 * 2 * 512 * 64 * 2)
    assert out.value == 2 * 2 * 512 * 64 * 2 + 256
    small16 = kvc.make_desc(1, 512, 2, 64, "f16")
    assert kvc.lib.kvc_prefill_scratch_bytes(ctypes.byref(small16), 4, 64, ctypes.byref(out)) == kvc.KVC_OK
    assert out.value == 256
    assert kvc.lib.kvc_prefill_scratch_bytes(ctypes.byref(small), 4, 513, ctypes.byref(out)) == kvc.KVC_ERANGE
    assert kvc.lib.kvc_prefill_scratch_bytes(ctypes.byref(small), 3, 64, ctypes.byref(out)) == kvc.KVC_EINVAL


def test_strerror(kvc):
    for code in (0, -1, -2, -3, -4, -5, -6, 12):
        assert len(kvc.lib.kvc_strerror(code)) > 0


@pytest.mark.parametrize("n,chunk", [(2013, 1024), (3865, 1024), (10041, 2048), (28998, 3328)])
def test_pipeline_chunk_gives_the_printed_chunks(kvc, n, chunk):
    # strata #1441, "Prompt chunks sized for a layer split's pipeline": four stages, b/a = 1024
    assert kvc.pipeline_chunk(n, cap=8192, stages=4) == chunk


def test_pipeline_chunk_equals_the_oracle_rule(kvc):
    from oracle.chunking import pipeline_chunk
    for n in list(range(1, 3000, 37)) + list(range(3000, 200000, 1999)):
        for cap in (256, 512, 2048, 4096, 65536):
            for stages in (1, 2, 3, 4, 8):
                for ba in (64.0, 1024.0, 3000.5):
                    assert kvc.pipeline_chunk(n, cap, stages, ba) == pipeline_chunk(n, cap, stages, ba), \
                        (n, cap, stages, ba)


def test_pipeline_chunk_rejects_bad_arguments(kvc):
    for args in ((0, 8192, 4), (100, 0, 4), (100, 8192, 0), (-5, 8192, 4)):
        with pytest.raises(kvc.KvcError):
            kvc.pipeline_chunk(*args)
    for ba in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(kvc.KvcError):
            kvc.pipeline_chunk(1000, 8192, 4, ba)
