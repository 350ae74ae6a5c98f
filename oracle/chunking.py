"""The pipeline chunk-size rule for prefill under a layer split.

Source: strata #1441, "Prompt chunks sized for a layer split's pipeline",
sections "Summary" and "What changed".  A prompt of n tokens read in chunks of
C over S pipeline stages takes (S - 1 + n/C) stage-chunks of (b + a*C), which
is smallest at C = sqrt(n * (b/a) / (S - 1)); b is a layer's fixed cost per
chunk and a its cost per token (b/a defaults to 1024 tokens).  The chunk is then
rounded up to the 256-token grid, kept at least 512 and at most the buffers'
chunk, and evened out over the chunks it takes so that there is no short last
chunk.  A prompt the rule would read in one chunk is read whole.

Reading taken for "evened out": with k = ceil(n / C) chunks, the chunk becomes
ceil(n / k) rounded up to the 256-token grid.
"""

import math

GRID = 256
MIN_CHUNK = 512


def _round_up(x, m):
    return -(-x // m) * m


def pipeline_chunk(n_tokens, cap, stages, b_over_a=1024.0):
    """Chunk size for n_tokens over `stages` pipeline stages; cap is the largest chunk allowed."""
    if n_tokens <= 0:
        raise ValueError("empty prompt")
    if stages <= 1:
        return min(n_tokens, cap)
    c = math.sqrt(n_tokens * b_over_a / (stages - 1))
    c = _round_up(math.ceil(c), GRID)
    c = max(c, MIN_CHUNK)
    c = min(c, cap)
    if c >= n_tokens:
        return n_tokens
    k = -(-n_tokens // c)
    even = _round_up(-(-n_tokens // k), GRID)
    return min(max(even, MIN_CHUNK), cap)
