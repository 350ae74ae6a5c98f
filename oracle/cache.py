"""A logical KV cache: append, chunked prompt prefill and single-token decode.

Source: the request flow of the pages.  A prompt is processed in ubatches of C
tokens against the growing cache (llama.cpp PR #17, "--split-overlap",
section "How"; strata #1441, "Prompt chunks sized for a layer split's
pipeline", section "Summary"); generation then decodes one token at a time
(llama.cpp PR #58, "completion : allow the prompt to be processed under its
own split mode", section "Why").  The cache is "device-resident q8_0" or f16
(same page, section "Why"; llama.cpp PR #59, section "Why").

Reading taken for the order of steps: a chunk's K/V rows are appended
(quantised) first, then its query rows attend to cache positions
[0, pos0 + C) with causality, so a row sees the stored (dequantised) values of
every key, including the keys of its own chunk.  With this order the result of
a row never depends on how the prompt was cut into chunks.

The logical store is indexed [layer][position][kv head][dim].  The two device
layouts are byte images of it:
    head-major   [kv head][layer][position][dim]   (a cache split by head)
    layer-major  [layer][position][kv head][dim]   (a cache split by layer)
with the q8_0 codes and the fp16 scales in separate arrays ([..][dim/32] for
the scales), and the f16 values in the code array.
"""

import numpy as np

from . import q8_0
from .attention import attend

Q8_0 = "q8_0"
F16 = "f16"
HEAD_MAJOR = "head_major"
LAYER_MAJOR = "layer_major"


class OracleCache:
    def __init__(self, n_layer, n_ctx, n_head_kv, head_dim, cache_type):
        if head_dim % q8_0.BLOCK:
            raise ValueError("head_dim must be a multiple of 32")
        if cache_type not in (Q8_0, F16):
            raise ValueError(cache_type)
        self.n_layer, self.n_ctx = n_layer, n_ctx
        self.n_head_kv, self.head_dim = n_head_kv, head_dim
        self.cache_type = cache_type
        shape = (n_layer, n_ctx, n_head_kv, head_dim)
        if cache_type == Q8_0:
            sshape = (n_layer, n_ctx, n_head_kv, head_dim // q8_0.BLOCK)
            self.k_q = np.zeros(shape, np.int8)
            self.v_q = np.zeros(shape, np.int8)
            self.k_d = np.zeros(sshape, np.float16)
            self.v_d = np.zeros(sshape, np.float16)
        else:
            self.k_f = np.zeros(shape, np.float16)
            self.v_f = np.zeros(shape, np.float16)

    # ---- append -----------------------------------------------------------
    def append(self, layer, pos0, k, v):
        """Store K/V rows [C, H_kv, D] (float32 values) at positions [pos0, pos0 + C)."""
        k = np.asarray(k, dtype=np.float32)
        v = np.asarray(v, dtype=np.float32)
        n = k.shape[0]
        if not (0 <= layer < self.n_layer and 0 <= pos0 and pos0 + n <= self.n_ctx):
            raise IndexError("append outside the cache")
        sl = slice(pos0, pos0 + n)
        if self.cache_type == Q8_0:
            self.k_d[layer, sl], self.k_q[layer, sl] = q8_0.quantize_blocks(k)
            self.v_d[layer, sl], self.v_q[layer, sl] = q8_0.quantize_blocks(v)
        else:
            self.k_f[layer, sl] = q8_0.to_f16(k)
            self.v_f[layer, sl] = q8_0.to_f16(v)

    # ---- reads ------------------------------------------------------------
    def dequantized(self, layer, n):
        """(khat, vhat) of positions [0, n), float64 [H_kv, n, D]."""
        if self.cache_type == Q8_0:
            kh = q8_0.dequantize_blocks(self.k_d[layer, :n], self.k_q[layer, :n])
            vh = q8_0.dequantize_blocks(self.v_d[layer, :n], self.v_q[layer, :n])
        else:
            kh = self.k_f[layer, :n].astype(np.float32)
            vh = self.v_f[layer, :n].astype(np.float32)
        return (np.ascontiguousarray(kh.transpose(1, 0, 2), dtype=np.float64),
                np.ascontiguousarray(vh.transpose(1, 0, 2), dtype=np.float64))

    def prefill_chunk(self, layer, pos0, q, rows=None):
        """Outputs of a chunk's query rows q [C, H_q, D] at positions [pos0, pos0 + C).

        Assumes the chunk's K/V were appended.  `rows` (indices into the chunk)
        restricts the computation to a subset of rows.
        """
        q = np.asarray(q)
        idx = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
        kh, vh = self.dequantized(layer, pos0 + q.shape[0])
        return attend(q[idx], pos0 + idx, kh, vh)

    def decode(self, layer, pos, q):
        """Output of one query token q [H_q, D] at position pos (its K/V appended)."""
        kh, vh = self.dequantized(layer, pos + 1)
        return attend(np.asarray(q)[None], [pos], kh, vh)[0]

    # ---- device byte images -----------------------------------------------
    def device_image(self, layout):
        """Arrays in the order a device cache of `layout` holds them.

        Returns (k_codes, k_scales, v_codes, v_scales); the scale arrays are None
        for the f16 cache, whose values sit in the code arrays as float16.
        """
        if self.cache_type == Q8_0:
            arrs = (self.k_q, self.k_d, self.v_q, self.v_d)
        else:
            arrs = (self.k_f, None, self.v_f, None)
        if layout == LAYER_MAJOR:
            return arrs
        if layout == HEAD_MAJOR:
            return tuple(None if a is None else np.ascontiguousarray(a.transpose(2, 0, 1, 3))
                         for a in arrs)
        raise ValueError(layout)
