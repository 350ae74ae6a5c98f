"""Causal grouped-query softmax attention over the dequantised cache, in float64.

Source: the flash attention the pages run over the KV cache during prompt
processing and generation (llama.cpp PR #17, "--split-overlap", section
"Results": "native FA"; prompt chunks attend to the growing cache in
llama.cpp PR #58, section "Why", and in strata #1441, "Prompt chunks sized for
a layer split's pipeline", section "Summary").  The pages do not print the
formula; this is the textbook one:

    O[t, h] = sum_{j <= t} w_j * vhat[j, g(h)] / sum_{j <= t} w_j
    w_j     = exp(s_j - max_j s_j),  s_j = (q[t, h] . khat[j, g(h)]) / sqrt(D)

with strict causality (query position t sees keys 0..t), the 1/sqrt(D) scale,
no window, soft-cap or bias, and grouped-query heads g(h) = h // (H_q / H_kv)
(contiguous groups of query heads share one KV head).  khat and vhat are the
values the cache holds after appending (dequantised q8_0 or f16), so a query
row in a chunk sees the chunk's own keys as stored in the cache.

Each query row is independent: the result of a row depends only on that row,
its position and the cache, never on which other rows are computed with it.
"""

import numpy as np


def attend(q_rows, positions, k_hat, v_hat):
    """Attention outputs for a set of query rows.

    q_rows    [R, H_q, D]   query rows (any float dtype; widened to float64)
    positions [R]           absolute position t of each query row
    k_hat     [H_kv, n, D]  dequantised keys of cache positions 0..n-1 (n > max position)
    v_hat     [H_kv, n, D]  dequantised values
    returns   [R, H_q, D]   float64
    """
    q = np.asarray(q_rows, dtype=np.float64)
    pos = np.asarray(positions, dtype=np.int64)
    n_rows, n_head_q, head_dim = q.shape
    n_head_kv, n_keys = k_hat.shape[0], k_hat.shape[1]
    if n_head_q % n_head_kv:
        raise ValueError("H_q must be a multiple of H_kv")
    if n_rows == 0:
        return np.zeros((0, n_head_q, head_dim))
    if pos.max() >= n_keys:
        raise ValueError("a query position lies beyond the cache contents")
    group = n_head_q // n_head_kv
    n_used = int(pos.max()) + 1
    key_index = np.arange(n_used)
    visible = key_index[None, :] <= pos[:, None]                   # [R, n_used]
    out = np.empty((n_rows, n_head_q, head_dim))
    for g in range(n_head_kv):
        kg = np.asarray(k_hat[g, :n_used], dtype=np.float64)      # [n_used, D]
        vg = np.asarray(v_hat[g, :n_used], dtype=np.float64)
        qg = q[:, g * group:(g + 1) * group, :]                    # [R, G, D]
        s = (qg @ kg.T) / np.sqrt(head_dim)                        # [R, G, n_used]
        s = np.where(visible[:, None, :], s, -np.inf)
        w = np.exp(s - s.max(axis=-1, keepdims=True))
        out[:, g * group:(g + 1) * group, :] = (w @ vg) / w.sum(axis=-1, keepdims=True)
    return out
