"""The layout-independent serialised cache state: pack and unpack.

Source: the sequence state the pages carry across a change of split mode.  It
is written in a layout-independent form, so the same bytes restore into a
cache split by layer or split by head and restore byte-identical (llama.cpp
PR #58, "completion : allow the prompt to be processed under its own split
mode", section "What this does"; llama.cpp PR #59, "llama : switch the split
mode of a live context", section "What this adds", step 1).  It is held as one
buffer whose size is linear in the context (PR #58, section "Cost").  The
pages fix no byte format; this one is the project's own:

    header, 32 bytes: eight little-endian uint32
        magic 'KVC1', version 1, n_layer, n_head_kv, head_dim,
        cache type (0 = f16, 1 = q8_0), n_tokens, 0
    body: for layer l in 0..n_layer-1, for position t in 0..n_tokens-1:
        the K record of (l, t), then the V record of (l, t);
        a record holds the kv heads in order; per head
          q8_0: head_dim/32 blocks of [fp16 scale, little-endian][32 int8 codes]
          f16:  head_dim float16 values, little-endian

Only positions [0, n_tokens) are written: no padding to the context size.
"""

import struct

import numpy as np

from .cache import F16, Q8_0, OracleCache

MAGIC = 0x3143564B          # the bytes 'K' 'V' 'C' '1' read as a little-endian uint32
VERSION = 1
HEADER_BYTES = 32
TYPE_CODE = {F16: 0, Q8_0: 1}


def record_bytes(n_head_kv, head_dim, cache_type):
    """Bytes of one K (or V) record of one (layer, position)."""
    if cache_type == Q8_0:
        return n_head_kv * (head_dim // 32) * 34
    return n_head_kv * head_dim * 2


def state_size(n_layer, n_head_kv, head_dim, cache_type, n_tokens):
    return HEADER_BYTES + n_layer * n_tokens * 2 * record_bytes(n_head_kv, head_dim, cache_type)


def header(cache, n_tokens):
    return struct.pack("<8I", MAGIC, VERSION, cache.n_layer, cache.n_head_kv, cache.head_dim,
                       TYPE_CODE[cache.cache_type], n_tokens, 0)


def pack(cache: OracleCache, n_tokens):
    """The state bytes (numpy uint8) of positions [0, n_tokens) of every layer."""
    if not 0 <= n_tokens <= cache.n_ctx:
        raise ValueError("n_tokens outside the cache")
    n = n_tokens
    L, H, D = cache.n_layer, cache.n_head_kv, cache.head_dim
    if cache.cache_type == Q8_0:
        nb = D // 32
        # body[l, t, kv, h, b, :] = one 34-byte block
        body = np.empty((L, n, 2, H, nb, 34), np.uint8)
        for kv, (d, q) in enumerate(((cache.k_d, cache.k_q), (cache.v_d, cache.v_q))):
            scale_bytes = d[:, :n].astype("<f2").view(np.uint8).reshape(L, n, H, nb, 2)
            code_bytes = q[:, :n].view(np.uint8).reshape(L, n, H, nb, 32)
            body[:, :, kv, :, :, 0:2] = scale_bytes
            body[:, :, kv, :, :, 2:34] = code_bytes
    else:
        body = np.empty((L, n, 2, H, D * 2), np.uint8)
        body[:, :, 0] = cache.k_f[:, :n].astype("<f2").view(np.uint8).reshape(L, n, H, D * 2)
        body[:, :, 1] = cache.v_f[:, :n].astype("<f2").view(np.uint8).reshape(L, n, H, D * 2)
    head = np.frombuffer(header(cache, n), np.uint8)
    return np.concatenate([head, body.reshape(-1)])


def check_header(stream, cache: OracleCache):
    """Validate a state against a destination cache; returns n_tokens or raises ValueError."""
    stream = np.asarray(stream, dtype=np.uint8)
    if stream.size < HEADER_BYTES:
        raise ValueError("state shorter than its header")
    magic, version, n_layer, n_head_kv, head_dim, tcode, n_tokens, reserved = struct.unpack(
        "<8I", stream[:HEADER_BYTES].tobytes())
    if magic != MAGIC or version != VERSION:
        raise ValueError("bad magic or version")
    if (n_layer, n_head_kv, head_dim, tcode) != (cache.n_layer, cache.n_head_kv, cache.head_dim,
                                                 TYPE_CODE[cache.cache_type]):
        raise ValueError("state was written from a cache of another shape or type")
    if reserved != 0:
        raise ValueError("reserved header field is not zero")
    if n_tokens > cache.n_ctx:
        raise ValueError("state holds more positions than the cache")
    if stream.size != state_size(n_layer, n_head_kv, head_dim, cache.cache_type, n_tokens):
        raise ValueError("state size does not match its header")
    return n_tokens


def unpack(stream, cache: OracleCache):
    """Restore a state into `cache`; returns n_tokens.  On any error nothing is written."""
    n = check_header(stream, cache)
    stream = np.asarray(stream, dtype=np.uint8)
    L, H, D = cache.n_layer, cache.n_head_kv, cache.head_dim
    if cache.cache_type == Q8_0:
        nb = D // 32
        body = stream[HEADER_BYTES:].reshape(L, n, 2, H, nb, 34)
        for kv, (d, q) in enumerate(((cache.k_d, cache.k_q), (cache.v_d, cache.v_q))):
            d[:, :n] = np.ascontiguousarray(body[:, :, kv, :, :, 0:2]).view("<f2").reshape(L, n, H, nb)
            q[:, :n] = np.ascontiguousarray(body[:, :, kv, :, :, 2:34]).view(np.int8).reshape(L, n, H, D)
    else:
        body = stream[HEADER_BYTES:].reshape(L, n, 2, H, D * 2)
        cache.k_f[:, :n] = np.ascontiguousarray(body[:, :, 0]).view("<f2").reshape(L, n, H, D)
        cache.v_f[:, :n] = np.ascontiguousarray(body[:, :, 1]).view("<f2").reshape(L, n, H, D)
    return n
