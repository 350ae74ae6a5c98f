"""CPU oracle for the attention-over-KV-cache path.  TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the path computes, used
to check the CUDA path.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import it; the library itself never does, and the two
share no code (the only common module is the seeded input generator, which
holds none of the method's arithmetic).

Modules:
  q8_0       block quantisation to 32-value int8 blocks with an fp16 scale, and
             the f16 cache rounding
  attention  causal grouped-query softmax attention in float64 over the
             dequantised cache
  cache      a logical KV cache (append, chunk prefill, decode) and the byte
             images of the two device layouts
  state      the layout-independent serialised cache state (pack / unpack)
  chunking   the pipeline chunk-size rule for a layer-split prefill

Every function is pinned by tests that do not re-run its own formula:
brute force over all int8 codes, hand-computed fp16 constants, hand-written
byte fixtures of the state format, torch's float64 scaled-dot-product
attention as a library special case, closed-form special cases (first row,
identical keys, constant values), the printed state sizes and the printed
chunk sizes of the pages.  No function is left with parity unpinned.
"""
