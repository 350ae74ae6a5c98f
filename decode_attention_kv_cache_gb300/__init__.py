"""Python binding of libkvc: attention over a device-resident q8_0/f16 KV cache on GB300.

Argument marshalling only.  Every step of the path (quantise-and-append,
chunked prefill attention, split-K decode attention, state pack/unpack) runs in
the library's CUDA kernels; torch supplies device memory and the current
stream.  The functions carry the names of the C ABI in include/kvc.h.

There is no fallback: the library is loaded on first use, which raises
ImportError if libkvc.so has not been built (python -m
decode_attention_kv_cache_gb300.build); every call raises KvcError when the
library reports an error.
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvc.so")

KVC_OK, KVC_EINVAL, KVC_ERANGE, KVC_ENOSPC, KVC_EFORMAT, KVC_ECUDA, KVC_EDEVICE = 0, -1, -2, -3, -4, -5, -6
CACHE_TYPES = {"f16": 0, "q8_0": 1}
LAYOUTS = {"head_major": 0, "layer_major": 1}
DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}


class KvcError(RuntimeError):
    def __init__(self, status, what):
        super().__init__("%s: %s (%d)" % (what, _lib().kvc_strerror(status).decode(), status))
        self.status = status


class kvc_desc(ctypes.Structure):
    _fields_ = [("n_layer", ctypes.c_int32), ("n_ctx", ctypes.c_int32), ("n_head_kv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("type", ctypes.c_int32), ("layout", ctypes.c_int32)]


class kvc_cache(ctypes.Structure):
    _fields_ = [("d", kvc_desc), ("k_q", ctypes.c_void_p), ("k_s", ctypes.c_void_p),
                ("v_q", ctypes.c_void_p), ("v_s", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libkvc.so is not built; run `python -m decode_attention_kv_cache_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    P, I32, SZ, VP = ctypes.POINTER, ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p
    sig = {
        "kvc_cache_bytes": (ctypes.c_int, [P(kvc_desc), P(SZ), P(SZ), P(SZ), P(SZ)]),
        "kvc_scratch_bytes": (ctypes.c_int, [P(kvc_desc), I32, P(SZ)]),
        "kv_state_size": (SZ, [P(kvc_desc), I32]),
        "kvc_cache_init": (ctypes.c_int, [P(kvc_cache), P(kvc_desc), VP, VP, VP, VP]),
        "kv_cache_append": (ctypes.c_int, [P(kvc_cache), I32, I32, I32, VP, VP, I32, VP]),
        "kvc_prefill_scratch_bytes": (ctypes.c_int, [P(kvc_desc), I32, I32, P(SZ)]),
        "prefill_chunk_attn": (ctypes.c_int, [P(kvc_cache), I32, I32, I32, VP, I32, I32, VP, VP, SZ, VP]),
        "decode_attn": (ctypes.c_int, [P(kvc_cache), I32, I32, VP, I32, I32, VP, VP, SZ, VP]),
        "prefill_step": (ctypes.c_int, [P(kvc_cache), I32, I32, I32, VP, VP, VP, I32, I32, VP, VP, SZ, I32, VP]),
        "kv_state_get": (ctypes.c_int, [P(kvc_cache), I32, VP, SZ, VP]),
        "kv_state_set": (ctypes.c_int, [P(kvc_cache), VP, SZ, P(I32), VP]),
        "kvc_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "kvc_device_status": (ctypes.c_int, [P(I32)]),
        "kvc_pipeline_chunk": (ctypes.c_int, [I32, I32, I32, ctypes.c_double, P(I32)]),
        "kv_cache_truncate": (ctypes.c_int, [P(kvc_cache), I32, VP]),
        "decode_attn_batch": (ctypes.c_int, [P(kvc_cache), I32, I32, P(I32), VP, I32, I32, VP, VP, SZ, VP]),
        "decode_step": (ctypes.c_int, [P(kvc_cache), I32, I32, VP, VP, VP, I32, I32, VP, VP, SZ, VP]),
        "decode_step_batch": (ctypes.c_int, [P(kvc_cache), I32, I32, P(I32), VP, VP, VP, I32, I32, VP, VP, SZ, VP]),
        "kv_cache_append_batch": (ctypes.c_int, [P(kvc_cache), I32, I32, P(I32), VP, VP, I32, VP]),
        "kv_state_get_heads": (ctypes.c_int, [P(kvc_cache), I32, I32, I32, VP, SZ, VP]),
        "kv_state_set_heads": (ctypes.c_int, [P(kvc_cache), I32, VP, SZ, P(I32), VP]),
        "kvc_test_arm_wait_timeout": (ctypes.c_int, [I32, ctypes.c_uint64]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    return L


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def __getattr__(name):
    if name == "lib":
        return _lib()
    raise AttributeError(name)


def _check(status, what):
    if status != KVC_OK:
        raise KvcError(status, what)


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(t, what, dtype=None):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA tensor" % what)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s" % (what, dtype))


def make_desc(n_layer, n_ctx, n_head_kv, head_dim, cache_type="q8_0", layout="head_major"):
    return kvc_desc(n_layer, n_ctx, n_head_kv, head_dim, CACHE_TYPES[cache_type], LAYOUTS[layout])


def cache_bytes(desc):
    s = [ctypes.c_size_t() for _ in range(4)]
    _check(_lib().kvc_cache_bytes(ctypes.byref(desc), *[ctypes.byref(x) for x in s]), "kvc_cache_bytes")
    return tuple(x.value for x in s)


class KVCache:
    """A cache whose four buffers are torch allocations on `device`.

    Codes/values: k_q, v_q; scales (q8_0 only): k_s, v_s.  The buffers are
    exposed as typed views in the layout of the descriptor.
    """

    def __init__(self, n_layer, n_ctx, n_head_kv, head_dim, cache_type="q8_0", layout="head_major",
                 device="cuda"):
        self.desc = make_desc(n_layer, n_ctx, n_head_kv, head_dim, cache_type, layout)
        self.n_layer, self.n_ctx, self.n_head_kv, self.head_dim = n_layer, n_ctx, n_head_kv, head_dim
        self.cache_type, self.layout = cache_type, layout
        self.device = torch.device(device)
        kq, ks, vq, vs = cache_bytes(self.desc)
        self._bufs = [torch.empty(max(n, 16), dtype=torch.uint8, device=self.device) for n in (kq, ks, vq, vs)]
        self._sizes = (kq, ks, vq, vs)
        self.c = kvc_cache()
        scales = cache_type == "q8_0"
        _check(_lib().kvc_cache_init(ctypes.byref(self.c), ctypes.byref(self.desc), _ptr(self._bufs[0]),
                                  _ptr(self._bufs[1]) if scales else ctypes.c_void_p(0), _ptr(self._bufs[2]),
                                  _ptr(self._bufs[3]) if scales else ctypes.c_void_p(0)), "kvc_cache_init")

    def _shape(self, last):
        if self.layout == "head_major":
            return (self.n_head_kv, self.n_layer, self.n_ctx, last)
        return (self.n_layer, self.n_ctx, self.n_head_kv, last)

    def codes(self, kv):
        """K (kv=0) or V (kv=1) codes (int8) or values (float16), in layout order."""
        b = self._bufs[2 * kv][: self._sizes[2 * kv]]
        dt = torch.int8 if self.cache_type == "q8_0" else torch.float16
        return b.view(dt).view(self._shape(self.head_dim))

    def scales(self, kv):
        if self.cache_type != "q8_0":
            return None
        b = self._bufs[2 * kv + 1][: self._sizes[2 * kv + 1]]
        return b.view(torch.float16).view(self._shape(self.head_dim // 32))

    def scratch_bytes(self, n_head_q):
        n = ctypes.c_size_t()
        _check(_lib().kvc_scratch_bytes(ctypes.byref(self.desc), n_head_q, ctypes.byref(n)), "kvc_scratch_bytes")
        return n.value

    def prefill_scratch_bytes(self, n_head_q, max_tokens):
        n = ctypes.c_size_t()
        _check(_lib().kvc_prefill_scratch_bytes(ctypes.byref(self.desc), n_head_q, max_tokens, ctypes.byref(n)),
               "kvc_prefill_scratch_bytes")
        return n.value

    def prefill_scratch(self, n_head_q, max_tokens):
        """A prefill scratch buffer for chunks of up to max_tokens rows (needs no initialisation)."""
        return torch.empty(max(self.prefill_scratch_bytes(n_head_q, max_tokens), 16), dtype=torch.uint8,
                           device=self.device)

    def state_size(self, n_tokens):
        return _lib().kv_state_size(ctypes.byref(self.desc), n_tokens)


def pipeline_chunk(n_tokens, cap, stages, b_over_a=1024.0):
    """Prompt chunk size for prefill over `stages` layer-split pipeline stages (host only)."""
    c = ctypes.c_int32(0)
    _check(_lib().kvc_pipeline_chunk(int(n_tokens), int(cap), int(stages), ctypes.c_double(b_over_a),
                                     ctypes.byref(c)), "kvc_pipeline_chunk")
    return c.value


def kv_cache_append(cache, layer, pos0, k, v, stream=None):
    """Quantise/round and store K, V [n, H_kv, D] at positions [pos0, pos0 + n) of `layer`."""
    _need(k, "k"); _need(v, "v", k.dtype)
    st = _lib().kv_cache_append(ctypes.byref(cache.c), layer, pos0, k.shape[0], _ptr(k), _ptr(v), DTYPES[k.dtype],
                             _stream(stream, k.device))
    _check(st, "kv_cache_append")


def prefill_chunk_attn(cache, layer, pos0, q, out=None, scratch=None, stream=None):
    """Causal attention of chunk rows q [C, H_q, D] at positions [pos0, pos0 + C); returns out [C, H_q, D] f32.

    scratch: a uint8 CUDA buffer (KVCache.prefill_scratch); one is made when None.
    """
    _need(q, "q")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if scratch is None:
        scratch = cache.prefill_scratch(q.shape[1], max(q.shape[0], 1))
    _need(out, "out", torch.float32); _need(scratch, "scratch")
    st = _lib().prefill_chunk_attn(ctypes.byref(cache.c), layer, pos0, q.shape[0], _ptr(q), DTYPES[q.dtype],
                                q.shape[1], _ptr(out), _ptr(scratch), scratch.numel() * scratch.element_size(),
                                _stream(stream, q.device))
    _check(st, "prefill_chunk_attn")
    return out


def prefill_step(cache, layer, pos0, q, k, v, out=None, scratch=None, stream=None, copy_valid=0):
    """One prompt chunk: store k, v [C, H_kv, D] at positions [pos0, pos0 + C) (as kv_cache_append) and
    attend with q [C, H_q, D] (as prefill_chunk_attn); returns out [C, H_q, D] f32.  copy_valid: leading
    positions of the scratch's fp16 copy (q8_0) already holding this layer's values from earlier calls
    with this scratch (pos0 when the previous chunk of this layer went through it)."""
    _need(q, "q"); _need(k, "k", q.dtype); _need(v, "v", q.dtype)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if scratch is None:
        scratch = cache.prefill_scratch(q.shape[1], max(q.shape[0], 1))
    _need(out, "out", torch.float32); _need(scratch, "scratch")
    st = _lib().prefill_step(ctypes.byref(cache.c), layer, pos0, q.shape[0], _ptr(q), _ptr(k), _ptr(v), DTYPES[q.dtype],
                             q.shape[1], _ptr(out), _ptr(scratch), scratch.numel() * scratch.element_size(),
                             copy_valid, _stream(stream, q.device))
    _check(st, "prefill_step")
    return out


def decode_attn(cache, layer, pos, q, out=None, scratch=None, stream=None):
    """Attention of one query token q [H_q, D] at position pos; returns out [H_q, D] f32."""
    _need(q, "q")
    n_head_q = q.shape[0]
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if scratch is None:
        scratch = torch.empty(cache.scratch_bytes(n_head_q), dtype=torch.uint8, device=q.device)
    _need(out, "out", torch.float32); _need(scratch, "scratch")
    st = _lib().decode_attn(ctypes.byref(cache.c), layer, pos, _ptr(q), DTYPES[q.dtype], n_head_q, _ptr(out),
                         _ptr(scratch), scratch.numel() * scratch.element_size(), _stream(stream, q.device))
    _check(st, "decode_attn")
    return out


def decode_step(cache, layer, pos, q, k, v, out=None, scratch=None, stream=None):
    """One decode step: store k, v [H_kv, D] at position pos (as kv_cache_append) and attend with
    q [H_q, D] over positions [0, pos] (as decode_attn); returns out [H_q, D] f32."""
    _need(q, "q"); _need(k, "k", q.dtype); _need(v, "v", q.dtype)
    n_head_q = q.shape[0]
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if scratch is None:
        scratch = torch.empty(cache.scratch_bytes(n_head_q), dtype=torch.uint8, device=q.device)
    _need(out, "out", torch.float32); _need(scratch, "scratch")
    st = _lib().decode_step(ctypes.byref(cache.c), layer, pos, _ptr(q), _ptr(k), _ptr(v), DTYPES[q.dtype], n_head_q,
                            _ptr(out), _ptr(scratch), scratch.numel() * scratch.element_size(),
                            _stream(stream, q.device))
    _check(st, "decode_step")
    return out


def decode_step_batch(caches, layer, pos, q, k, v, out=None, scratch=None, stream=None):
    """decode_step for len(caches) sequences in one call: q [n_seq][H_q][D], k and v [n_seq][H_kv][D]
    (CUDA), pos a list; returns out [n_seq][H_q][D] f32."""
    n = len(caches)
    if n != len(pos) or q.dim() != 3 or q.shape[0] != n or k.shape[0] != n or v.shape != k.shape:
        raise ValueError("one position, one query and one K/V row block per sequence")
    _need(q, "q"); _need(k, "k", q.dtype); _need(v, "v", q.dtype)
    c0 = caches[0]
    n_head_q = q.shape[1]
    if out is None:
        out = torch.empty(n, n_head_q, c0.head_dim, dtype=torch.float32, device=c0.device)
    _need(out, "out", torch.float32)
    if scratch is None:
        scratch = torch.empty(n * c0.scratch_bytes(n_head_q), dtype=torch.uint8, device=c0.device)
    _need(scratch, "scratch")
    arr = (kvc_cache * n)(*[c.c for c in caches])
    ps = (ctypes.c_int32 * n)(*[int(p) for p in pos])
    st = _lib().decode_step_batch(arr, n, layer, ps, _ptr(q), _ptr(k), _ptr(v), DTYPES[q.dtype], n_head_q, _ptr(out),
                                  _ptr(scratch), scratch.numel() * scratch.element_size(), _stream(stream, c0.device))
    _check(st, "decode_step_batch")
    return out


def kv_cache_append_batch(caches, layer, pos, k, v, stream=None):
    """Append one token per sequence: row i of k and v ([n_seq][H_kv][D], CUDA) to caches[i] at pos[i]."""
    n = len(caches)
    if n != len(pos) or k.shape[0] != n or v.shape != k.shape or k.dtype != v.dtype:
        raise ValueError("one position and one K/V row block per sequence")
    _need(k, "k"); _need(v, "v")
    arr = (kvc_cache * n)(*[c.c for c in caches])
    ps = (ctypes.c_int32 * n)(*[int(p) for p in pos])
    st = _lib().kv_cache_append_batch(arr, n, layer, ps, _ptr(k), _ptr(v), DTYPES[k.dtype],
                                   _stream(stream, caches[0].device))
    _check(st, "kv_cache_append_batch")


def decode_attn_batch(caches, layer, pos, q, out=None, scratch=None, stream=None):
    """Decode one token for each of len(caches) sequences in one call: q [n_seq][n_head_q][head_dim]
    (CUDA), pos a list of positions; returns out [n_seq][n_head_q][head_dim] float32."""
    n = len(caches)
    if n != len(pos) or q.dim() != 3 or q.shape[0] != n:
        raise ValueError("one position and one query row block per sequence")
    _need(q, "q")
    c0 = caches[0]
    n_head_q = q.shape[1]
    if out is None:
        out = torch.empty(n, n_head_q, c0.head_dim, dtype=torch.float32, device=c0.device)
    _need(out, "out", torch.float32)
    if scratch is None:
        scratch = torch.empty(n * c0.scratch_bytes(n_head_q), dtype=torch.uint8, device=c0.device)
    _need(scratch, "scratch")
    arr = (kvc_cache * n)(*[c.c for c in caches])
    ps = (ctypes.c_int32 * n)(*[int(p) for p in pos])
    st = _lib().decode_attn_batch(arr, n, layer, ps, _ptr(q), DTYPES[q.dtype], n_head_q, _ptr(out), _ptr(scratch),
                               scratch.numel() * scratch.element_size(), _stream(stream, c0.device))
    _check(st, "decode_attn_batch")
    return out


def kv_state_get(cache, n_tokens, dst=None, stream=None):
    """Serialise positions [0, n_tokens) into dst (uint8 CUDA tensor); returns dst."""
    n = cache.state_size(n_tokens)
    if dst is None:
        dst = torch.empty(max(n, 16), dtype=torch.uint8, device=cache.device)
    _need(dst, "dst")
    st = _lib().kv_state_get(ctypes.byref(cache.c), n_tokens, _ptr(dst), dst.numel() * dst.element_size(),
                          _stream(stream, cache.device))
    _check(st, "kv_state_get")
    return dst[:n]


def kv_state_set(cache, src, stream=None):
    """Restore a state (uint8 CUDA tensor of exactly the state's size); returns n_tokens."""
    _need(src, "src")
    n = ctypes.c_int32(-1)
    st = _lib().kv_state_set(ctypes.byref(cache.c), _ptr(src), src.numel() * src.element_size(), ctypes.byref(n),
                          _stream(stream, cache.device))
    _check(st, "kv_state_set")
    return n.value


def kv_state_get_heads(cache, head0, n_head_total, n_tokens, dst=None, stream=None):
    """Write the part of the whole state (n_head_total kv heads) that `cache`, holding kv heads
    [head0, head0 + cache.n_head_kv), owns, plus the header, into dst; returns dst."""
    whole = make_desc(cache.n_layer, cache.n_ctx, n_head_total, cache.head_dim, cache.cache_type, cache.layout)
    n = _lib().kv_state_size(ctypes.byref(whole), n_tokens)
    if dst is None:
        dst = torch.zeros(max(n, 16), dtype=torch.uint8, device=cache.device)
    _need(dst, "dst")
    st = _lib().kv_state_get_heads(ctypes.byref(cache.c), head0, n_head_total, n_tokens, _ptr(dst),
                                dst.numel() * dst.element_size(), _stream(stream, cache.device))
    _check(st, "kv_state_get_heads")
    return dst[:n]


def kv_state_set_heads(cache, head0, src, stream=None):
    """Restore kv heads [head0, head0 + cache.n_head_kv) of a whole state into `cache`; returns n_tokens."""
    _need(src, "src")
    n = ctypes.c_int32(-1)
    st = _lib().kv_state_set_heads(ctypes.byref(cache.c), head0, _ptr(src), src.numel() * src.element_size(),
                                ctypes.byref(n), _stream(stream, cache.device))
    _check(st, "kv_state_set_heads")
    return n.value


def kv_cache_truncate(cache, n_tokens, stream=None):
    """Rewind `cache` to its first n_tokens positions (later positions cleared to zero bytes)."""
    _check(_lib().kv_cache_truncate(ctypes.byref(cache.c), int(n_tokens), _stream(stream, cache.device)),
           "kv_cache_truncate")


def kvc_device_status():
    """Synchronise and read/clear the device status word (non-zero: a kernel gave up a bounded wait,
    which the C call reports as KVC_EDEVICE)."""
    s = ctypes.c_int32(0)
    rc = _lib().kvc_device_status(ctypes.byref(s))
    if rc != KVC_EDEVICE:
        _check(rc, "kvc_device_status")
    return s.value


TEST_PREFILL, TEST_DECODE = 0, 1


def arm_test_wait_timeout(which, limit_ns):
    """Test hook: the next launch of the prefill (TEST_PREFILL) or head_dim-128 decode (TEST_DECODE)
    tensor-core kernel waits on a barrier nothing arrives at, gives up after limit_ns and unwinds."""
    _check(_lib().kvc_test_arm_wait_timeout(which, limit_ns), "kvc_test_arm_wait_timeout")
