/*
 * kvc.h - C ABI of libkvc: one transformer attention layer's hot path over a
 * device-resident KV cache on NVIDIA GB300 (sm_103a).
 *
 * The path, as the source pages describe it:
 *   - a prompt is processed in ubatches ("chunks") of C tokens against the
 *     growing KV cache, then generation decodes one token at a time
 *     (llama.cpp PR #58 "completion : allow the prompt to be processed under
 *     its own split mode", section "Why"; llama.cpp PR #17 "--split-overlap",
 *     section "How"; strata #1441 "Prompt chunks sized for a layer split's
 *     pipeline", section "Summary");
 *   - the cache is device-resident and stored as q8_0 or f16 (PR #58,
 *     section "Why"; llama.cpp PR #59 "llama : switch the split mode of a live
 *     context", section "Why");
 *   - the cache state is serialised in a layout-independent form that restores
 *     byte-identical into a cache split by layer or by head (PR #58, section
 *     "What this does"; PR #59, section "What this adds", step 1).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers unless stated otherwise.  The
 *     caller allocates and owns every buffer (cache, inputs, outputs, scratch,
 *     state) and the stream; the library allocates no device memory.
 *   - Work is asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  Only kv_state_set synchronises (once, to read the
 *     32-byte header before anything is written).
 *   - Q, K, V and the outputs are token-major and contiguous:
 *       q   [n_tokens][n_head_q ][head_dim]   in kvc_dtype
 *       k,v [n_tokens][n_head_kv][head_dim]   in kvc_dtype
 *       out [n_tokens][n_head_q ][head_dim]   float32
 *   - Every argument is checked before anything is launched.  A call that
 *     returns an error has launched nothing and written nothing: the cache
 *     stays as it was and usable (the pages' rule that a failure must leave a
 *     working context, PR #58 section "Memory"; PR #59 section "What this
 *     adds").  Errors of asynchronous work surface at the caller's next
 *     synchronisation; the kernels contain no unbounded waits.
 *   - The append, prefill attention (and its split merge), prefill_step's
 *     first kernel and the decode kernels are launched with programmatic
 *     dependent launch: one may be scheduled while the kernel before it on
 *     `stream` is finishing, and it waits on the device (griddepcontrol.wait)
 *     for that kernel to complete before it reads or writes memory (the decode
 *     split pass only hints, before that wait, that L2 fetch its first tiles,
 *     which moves no data it reads).  Stream order therefore holds exactly as
 *     for ordinary launches, also inside a captured CUDA graph.  The state
 *     kernels and prefill_chunk_attn's q8_0 dequantising pass are ordinary
 *     launches.
 *
 * Cache contents.  A cache holds n_layer layers of n_ctx positions of
 * n_head_kv heads of head_dim values, for K and for V.  Cache types:
 *   KVC_Q8_0: blocks of 32 consecutive values along head_dim; each block has
 *             one fp16 scale d = fp16(amax/127) and 32 int8 codes
 *             q = round(x / (amax/127)) (float32 division, ties away from zero),
 *             all codes and d zero for an all-zero block.  The stored value is
 *             d * q.  Codes and scales live in separate arrays.
 *   KVC_F16:  fp16(x), round to nearest even.  The scale arrays are unused.
 * Layouts (element offsets; nb = head_dim/32; codes use head_dim, scales nb):
 *   KVC_HEAD_MAJOR  [n_head_kv][n_layer][n_ctx][head_dim]   (split by head)
 *   KVC_LAYER_MAJOR [n_layer][n_ctx][n_head_kv][head_dim]   (split by layer)
 *
 * Supported shapes: head_dim a multiple of 32 for append and state calls;
 * head_dim 64 or 128 for the attention calls; n_head_q a multiple of
 * n_head_kv; n_head_q / n_head_kv <= 16 for the decode calls.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kvc_stream_t; /* a cudaStream_t */

/* Status codes: 0 on success, negative on error. */
#define KVC_OK       0
#define KVC_EINVAL  -1 /* null pointer, unsupported shape, dtype or type, bad alignment */
#define KVC_ERANGE  -2 /* layer or positions outside the cache */
#define KVC_ENOSPC  -3 /* a destination or scratch buffer is too small */
#define KVC_EFORMAT -4 /* a state stream that does not match its header or the cache */
#define KVC_ECUDA   -5 /* a CUDA call or launch failed */
#define KVC_EDEVICE -6 /* a kernel gave up a bounded wait (see kvc_device_status) */

typedef enum { KVC_F16 = 0, KVC_Q8_0 = 1 } kvc_cache_type;
typedef enum { KVC_IN_F32 = 0, KVC_IN_BF16 = 1, KVC_IN_F16 = 2 } kvc_dtype;
typedef enum { KVC_HEAD_MAJOR = 0, KVC_LAYER_MAJOR = 1 } kvc_layout;

/* Shape, type and layout of a cache.  Plain data. */
typedef struct {
    int32_t n_layer;
    int32_t n_ctx;
    int32_t n_head_kv;
    int32_t head_dim;
    int32_t type;    /* kvc_cache_type */
    int32_t layout;  /* kvc_layout */
} kvc_desc;

/* A cache: its descriptor and four caller-owned device buffers.  For q8_0,
 * k_q/v_q hold int8 codes and k_s/v_s fp16 scales; for f16, k_q/v_q hold the
 * fp16 values and k_s/v_s are NULL.  Buffers must be 16-byte aligned and at
 * least as large as kvc_cache_bytes reports.  Plain data, copied by value. */
typedef struct {
    kvc_desc d;
    void *k_q;
    void *k_s;
    void *v_q;
    void *v_s;
} kvc_cache;

/* ---- size queries and set-up (host only, no CUDA call) -------------------- */

/* Bytes of each of the four cache buffers (scale sizes are 0 for f16).
 * Returns KVC_EINVAL for an invalid descriptor. */
int kvc_cache_bytes(const kvc_desc *desc, size_t *k_q, size_t *k_s, size_t *v_q, size_t *v_s);

/* Bytes of the scratch buffer decode_attn and decode_step need for this cache
 * and n_head_q: float32 partial results of the split-K pass,
 * [n_head_q][max_split][head_dim + 2]. */
int kvc_scratch_bytes(const kvc_desc *desc, int32_t n_head_q, size_t *bytes);

/* Bytes of the serialised state of n_tokens positions: 32 + n_layer * n_tokens *
 * 2 * record, record = n_head_kv * head_dim/32 * 34 (q8_0) or n_head_kv *
 * head_dim * 2 (f16).  Returns 0 for an invalid descriptor or n_tokens. */
size_t kv_state_size(const kvc_desc *desc, int32_t n_tokens);

/* Fill *out from a descriptor and four device buffers after checking them
 * (shape, non-null, 16-byte alignment).  Writes *out only on success. */
int kvc_cache_init(kvc_cache *out, const kvc_desc *desc, void *k_q, void *k_s, void *v_q, void *v_s);

/* The prompt chunk size for prefill when the layers are split over `stages`
 * pipeline stages (strata PR #1441 "Prompt chunks sized for a layer split's
 * pipeline", sections "Summary" and "What changed"): C = sqrt(n_tokens *
 * b_over_a / (stages - 1)), where b_over_a is a layer's fixed cost per chunk
 * over its cost per token (the page uses 1024), rounded up to the 256-token grid,
 * kept within [512, cap] and evened out over the ceil(n_tokens / C) chunks it
 * needs (ceil(n_tokens / chunks), rounded up to the grid, within [512, cap]).  A
 * prompt that fits in one chunk is read whole; one stage gives min(n_tokens,
 * cap).  Host only.  Writes *chunk on success; KVC_EINVAL for n_tokens, cap or
 * stages <= 0, a b_over_a that is not finite and positive, or a null chunk. */
int kvc_pipeline_chunk(int32_t n_tokens, int32_t cap, int32_t stages, double b_over_a, int32_t *chunk);

/* ---- hot path ---------------------------------------------------------------- */

/* Append (quantise and store) the K/V rows of n_tokens tokens at cache
 * positions [pos0, pos0 + n_tokens) of `layer`.  k, v: [n_tokens][n_head_kv]
 * [head_dim] in `dtype`, values finite.  q8_0 blocks and f16 values exactly as
 * defined above (bit-exact: float32 IEEE division, round half away from zero,
 * fp16 round to nearest even).  n_tokens == 0 is a no-op.
 * Errors: KVC_EINVAL (null, dtype), KVC_ERANGE (layer, pos0 + n_tokens > n_ctx). */
int kv_cache_append(const kvc_cache *cache, int32_t layer, int32_t pos0, int32_t n_tokens,
                    const void *k, const void *v, int32_t dtype, kvc_stream_t stream);

/* Append one token to each of n_seq caches (1 <= n_seq <= 8) in one launch:
 * row i of k and v ([n_seq][n_head_kv][head_dim] in `dtype`) goes to position
 * pos[i] of `layer` of caches[i], quantised exactly as kv_cache_append does.
 * This is the append half of a decode step of several sequences together (see
 * decode_attn_batch).  caches: host array whose descriptors agree in n_head_kv,
 * head_dim and type; pos: host array.  Errors: KVC_EINVAL (null, dtype, n_seq
 * outside [1, 8], caches that disagree), KVC_ERANGE (layer or any pos[i] outside
 * its cache). */
int kv_cache_append_batch(const kvc_cache *caches, int32_t n_seq, int32_t layer, const int32_t *pos, const void *k,
                          const void *v, int32_t dtype, kvc_stream_t stream);

/* Bytes of the scratch buffer prefill_chunk_attn and prefill_step need for
 * chunks of up to max_tokens rows anywhere in this cache: a 256-byte header
 * (prefill_step's work counter) and the float32 partial results (output row,
 * running max, sum) of the key splits, and for a q8_0 cache in front of them
 * room for an fp16 copy of one layer's
 * keys and values (2 * n_head_kv * n_ctx * head_dim * 2 bytes, laid out
 * [K|V][head][position][head_dim]).  The contents need no initialisation:
 * every call writes what it reads, except the part of the copy that
 * prefill_step's copy_valid says is already there. */
int kvc_prefill_scratch_bytes(const kvc_desc *desc, int32_t n_head_q, int32_t max_tokens, size_t *bytes);

/* Causal attention of a chunk's query rows over the cache:
 *   out[i][h] = sum_{j <= pos0+i} softmax_j(q[i][h] . khat[j][h/G] / sqrt(head_dim)) vhat[j][h/G]
 * for i in [0, n_tokens), G = n_head_q / n_head_kv, khat/vhat the values the
 * cache holds for `layer` at positions [0, pos0 + n_tokens).  The chunk's own
 * K/V must have been appended (kv_cache_append earlier on the same stream).
 * Keys are processed in tiles of 256 and splits whose boundaries sit at
 * absolute positions (a size fixed by n_ctx); partial results of a row are
 * merged in split order, so a row's output is bitwise independent of how the
 * prompt is cut into chunks.  Computed with fp16 tensor-core products and
 * float32 accumulation and softmax.  A q8_0 cache's keys and values enter the
 * products as fp16(d * q): with the full scratch of kvc_prefill_scratch_bytes,
 * positions [0, pos0 + n_tokens) are first dequantised once into the scratch's
 * copy (one more kernel), and the attention reads that copy; with a scratch that
 * holds only the partials, the attention kernel dequantises each tile in
 * shared memory instead (slower: once per 128-row query tile).  Both give the
 * same bits.
 * q: [n_tokens][n_head_q][head_dim] in dtype (f32, bf16 or f16); out float32.
 * Kernels on `stream`: for q8_0 with the full scratch the dequantising pass,
 * then the attention (partials of rows whose keys span several splits go to
 * scratch) and, when any row has several splits, the merge.  scratch: device buffer of scratch_bytes >=
 * kvc_prefill_scratch_bytes(desc, n_head_q, n_tokens); calls on one scratch
 * buffer must not overlap on the GPU.
 * Errors: KVC_EINVAL (null, dtype, head_dim not 64/128, heads), KVC_ERANGE,
 * KVC_ENOSPC (scratch too small). */
int prefill_chunk_attn(const kvc_cache *cache, int32_t layer, int32_t pos0, int32_t n_tokens,
                       const void *q, int32_t dtype, int32_t n_head_q, float *out, void *scratch,
                       size_t scratch_bytes, kvc_stream_t stream);

/* One prompt chunk in one call: store its K/V at positions [pos0, pos0 +
 * n_tokens) of `layer`, exactly as kv_cache_append does (the same bytes), then
 * attend with its query rows exactly as prefill_chunk_attn does (the same bits
 * of out): the ubatch step of prompt processing (llama.cpp PR #17
 * "--split-overlap", section "How"; strata #1441 "Prompt chunks sized for a
 * layer split's pipeline", "Summary").  q: [n_tokens][n_head_q][head_dim], k and
 * v: [n_tokens][n_head_kv][head_dim], device memory in `dtype`, 16-byte
 * aligned; out float32.  Kernels: the first stores the chunk (for q8_0 with
 * the full scratch it also completes the fp16 copy of positions [0, pos0 +
 * n_tokens) that the attention reads, so no separate dequantising pass runs),
 * then the attention and, when rows span several key splits, the merge - two
 * launches, or three with the merge, where the separate calls take three or
 * four.  The attention's CTAs take their work items in order from a counter
 * in the scratch header, which the first kernel sets to zero; the result does
 * not depend on which CTA takes which item.  scratch: as for
 * prefill_chunk_attn (kvc_prefill_scratch_bytes); calls on one scratch buffer
 * must not overlap on the GPU.
 * copy_valid (0 <= copy_valid <= pos0): how many leading positions of the
 * scratch's fp16 copy already hold this layer's values, left there by earlier
 * calls of prefill_step or prefill_chunk_attn with this scratch on this cache
 * and layer, the cache's positions [0, copy_valid) unchanged since.  The call
 * converts [copy_valid, pos0) from the cache and the chunk from the codes it
 * stores, so a prompt processed chunk after chunk on one scratch with
 * copy_valid = pos0 converts each position once (an fp16 copy per layer when
 * chunks go through all layers in turn).  0 for a fresh scratch; a
 * copy_valid that overstates the copy gives wrong outputs, not an error.
 * Ignored for an f16 cache and for a scratch without the copy.
 * Errors as prefill_chunk_attn, KVC_EINVAL for a null or unaligned k or v,
 * KVC_ERANGE for copy_valid outside [0, pos0]. */
int prefill_step(const kvc_cache *cache, int32_t layer, int32_t pos0, int32_t n_tokens, const void *q, const void *k,
                 const void *v, int32_t dtype, int32_t n_head_q, float *out, void *scratch, size_t scratch_bytes,
                 int32_t copy_valid, kvc_stream_t stream);

/* Single-token decode attention at position pos: the formula above with one
 * query row at pos, keys [0, pos].  The token's K/V must have been appended.
 * Split-K over the key range into float32 partials in `scratch` (size from
 * kvc_scratch_bytes), then a combine pass.  q: [n_head_q][head_dim] in dtype;
 * out: [n_head_q][head_dim] float32.
 * Errors: KVC_EINVAL, KVC_ERANGE, KVC_ENOSPC (scratch too small). */
int decode_attn(const kvc_cache *cache, int32_t layer, int32_t pos, const void *q, int32_t dtype,
                int32_t n_head_q, float *out, void *scratch, size_t scratch_bytes,
                kvc_stream_t stream);

/* Decode attention for n_seq sequences in one call (1 <= n_seq <= 8): sequence i
 * attends with its query at position pos[i] over positions [0, pos[i]] of its
 * own cache caches[i], exactly as decode_attn would.  This is decoding several
 * sequences together, one token each per step, as llama-batched-bench's npl
 * parallel sequences do (llama.cpp PR #58 "completion : allow the prompt to be
 * processed under its own split mode", section "Why -np 1", the npl
 * table; llama.cpp PR #59 "llama : switch the split mode of a live context",
 * section "Several sequences at once").  caches: host array of n_seq caches
 * whose descriptors agree in n_layer, n_ctx, n_head_kv, head_dim and type (the
 * layouts may differ).  pos: host array of n_seq positions.  q: device,
 * [n_seq][n_head_q][head_dim] in `dtype`; out: device, [n_seq][n_head_q]
 * [head_dim] float32.  scratch: device, at least n_seq * kvc_scratch_bytes(desc,
 * n_head_q) bytes, sequence i using the i-th slice.  With head_dim 128 the split
 * pass of all sequences is one launch over (split, kv head, sequence), the SMs
 * shared evenly among the sequences, followed by one combine launch; with
 * head_dim 64 (or n_seq == 1) each sequence is its own launch pair.  A batched
 * call may choose other split boundaries than decode_attn for the same
 * sequence, so results agree within rounding, not bit for bit.  Errors as
 * decode_attn; KVC_EINVAL also for n_seq outside [1, 8] or caches that disagree,
 * KVC_ERANGE for any pos[i] out of range, KVC_ENOSPC for a scratch below n_seq
 * slices. */
int decode_attn_batch(const kvc_cache *caches, int32_t n_seq, int32_t layer, const int32_t *pos, const void *q,
                      int32_t dtype, int32_t n_head_q, float *out, void *scratch, size_t scratch_bytes,
                      kvc_stream_t stream);

/* One decode step in one call: store the token's K/V at position pos, exactly
 * as kv_cache_append(cache, layer, pos, 1, k, v, dtype) does (the same bytes),
 * then attend with its query over positions [0, pos] exactly as decode_attn
 * does (the same bits of out).  This is the per-token work of generation, which
 * the pages time as "generation t/s" (llama.cpp PR #58 "completion : allow the
 * prompt to be processed under its own split mode", section "Why"; llama.cpp
 * PR #59 "llama : switch the split mode of a live context", section "Why").
 * q: [n_head_q][head_dim], k and v: [n_head_kv][head_dim], all device memory
 * in `dtype`, 16-byte aligned; out: [n_head_q][head_dim] float32.
 * It is two kernels: the split pass, in which the CTA whose key range holds
 * pos quantises and stores the token before it copies that tile, then
 * decode_attn's combine.  scratch: as for decode_attn
 * (kvc_scratch_bytes, no initialisation); calls on one scratch buffer must not
 * overlap on the GPU.  Errors: KVC_EINVAL (null or unaligned pointers, dtype,
 * head_dim, heads), KVC_ERANGE (layer, pos), KVC_ENOSPC (scratch too small). */
int decode_step(const kvc_cache *cache, int32_t layer, int32_t pos, const void *q, const void *k, const void *v,
                int32_t dtype, int32_t n_head_q, float *out, void *scratch, size_t scratch_bytes, kvc_stream_t stream);

/* decode_step for n_seq sequences in one call (1 <= n_seq <= 8): sequence i
 * stores row i of k and v at position pos[i] of caches[i] and attends with row
 * i of q, as decode_step would.  caches, pos: host arrays as for
 * decode_attn_batch.  q: [n_seq][n_head_q][head_dim]; k, v: [n_seq][n_head_kv]
 * [head_dim]; out: [n_seq][n_head_q][head_dim] float32.  scratch: as for
 * decode_attn_batch.  With head_dim 128 the sequences share one split pass and
 * one combine (decode_attn_batch's kernels, whose split boundaries it shares,
 * so out matches decode_attn_batch bit for bit); otherwise each sequence is its
 * own decode_step.  Errors as decode_attn_batch. */
int decode_step_batch(const kvc_cache *caches, int32_t n_seq, int32_t layer, const int32_t *pos, const void *q,
                      const void *k, const void *v, int32_t dtype, int32_t n_head_q, float *out, void *scratch,
                      size_t scratch_bytes, kvc_stream_t stream);

/* decode_attn without a scratch argument, for callers that cannot allocate
 * device memory themselves (code hosted by an engine that owns every device
 * allocation, or a path where cudaMalloc's implicit synchronisation is not
 * allowed).  The source pages have no counterpart of this call; it is a
 * convenience of this library.  The split-K partials go to a fixed 8 MiB
 * device array inside the library (held on every device that loads it, until
 * the process exits): calls whose kvc_scratch_bytes(desc, n_head_q) exceeds
 * 8 MiB (n_head_q * 256 * (head_dim + 2) * 4 bytes, i.e. n_head_q > 63 at
 * head_dim 128) are rejected with KVC_ENOSPC before anything is launched.
 * The call allocates nothing.  Its first call in a device's context looks up
 * that array's device address (cudaGetSymbolAddress) with the device current
 * and caches it under the context's id, so a context created again after a
 * device reset gets a fresh lookup; make that first call before capturing a
 * stream into a CUDA graph.  The cache, q, out and the stream must belong to
 * the current device: a cache or output on another device is rejected with
 * KVC_EINVAL.  All calls share the one array: calls that overlap on the GPU
 * (other streams, other threads) race and must be serialised by the caller.
 * When kvc_device_status() reports a non-zero status after a call, that
 * call's out is undefined.  Arguments, result and errors otherwise as
 * decode_attn. */
int decode_attn_noalloc(const kvc_cache *cache, int32_t layer, int32_t pos, const void *q, int32_t dtype,
                        int32_t n_head_q, float *out, kvc_stream_t stream);

/* Serialise positions [0, n_tokens) of every layer into dst (device memory,
 * dst_bytes >= kv_state_size).  The stream does not depend on the layout.
 * Format: 32-byte header of eight little-endian uint32 (magic 'KVC1',
 * version 1, n_layer, n_head_kv, head_dim, type, n_tokens, 0); then for each
 * layer, for each position, the K record then the V record; a record holds
 * the kv heads in order, each as head_dim/32 blocks of [fp16 scale LE][32
 * int8 codes] (q8_0) or head_dim fp16 values LE (f16).
 * Errors: KVC_EINVAL, KVC_ERANGE (n_tokens > n_ctx), KVC_ENOSPC. */
int kv_state_get(const kvc_cache *cache, int32_t n_tokens, void *dst, size_t dst_bytes,
                 kvc_stream_t stream);

/* Restore a state written by kv_state_get (from a cache of any layout) into
 * `cache`.  src: device memory of src_bytes.  Synchronises `stream` once to
 * read the header, validates it (magic, version, shape and type equal to the
 * cache's, n_tokens <= n_ctx, src_bytes equal to the size the header implies)
 * and only then writes.  *n_tokens_out receives n_tokens on success.
 * Errors: KVC_EINVAL (null), KVC_EFORMAT (any header mismatch), KVC_ECUDA. */
int kv_state_set(kvc_cache *cache, const void *src, size_t src_bytes, int32_t *n_tokens_out,
                 kvc_stream_t stream);

/* A cache split by head: its kv heads spread over several caches (as over several
 * devices), each holding a contiguous range.  kv_state_get_heads writes the part
 * of the stream that `cache`, holding kv heads [head0, head0 + its n_head_kv) of
 * n_head_total, owns: those heads' blocks (or values) of every record, plus the
 * header of the whole state (n_head_total heads), which every part writes
 * identically.  Calls for parts that cover all heads, on one dst, produce the
 * stream kv_state_get writes for the unsplit cache, byte for byte.
 * kv_state_set_heads restores that range from a whole stream, however it was
 * written (llama.cpp PR #59 "llama : switch the split mode of a live context",
 * section "What this adds", step 1: a state restores into a cache split by
 * layer or by head; llama.cpp PR #58 "completion : allow the prompt to be
 * processed under its own split mode", section "The library version, for
 * later", item 2).  dst/src: device memory sized for the whole state.
 * Errors as kv_state_get / kv_state_set; KVC_EINVAL for a head range outside
 * n_head_total; kv_state_set_heads gives KVC_EFORMAT when the header's head
 * count does not cover the range. */
int kv_state_get_heads(const kvc_cache *cache, int32_t head0, int32_t n_head_total, int32_t n_tokens, void *dst,
                       size_t dst_bytes, kvc_stream_t stream);
int kv_state_set_heads(kvc_cache *cache, int32_t head0, const void *src, size_t src_bytes, int32_t *n_tokens_out,
                       kvc_stream_t stream);

/* Rewind the cache to its first n_tokens positions: positions [n_tokens, n_ctx)
 * of every layer, codes and scales, are cleared to zero bytes, as in a zeroed
 * cache; earlier positions are untouched.  This is the undo of appends past
 * n_tokens that a sequence needs when it drops speculative decode appends or
 * trims excess state (mlxcel issue #2170 "refactor: one prefill planner and one
 * pad-trim hook for CLI and server", sections "Current Behavior", the hook that
 * unwinds decode appends exactly, and "Proposed Solution", item 2, one trim hook
 * with an excess count).  Appends and attention address positions, so a cache
 * rewound to n and appended again computes exactly what a cache that never held
 * the dropped tokens computes.  Asynchronous on `stream` (strided memsets).
 * Errors: KVC_EINVAL (invalid cache), KVC_ERANGE (n_tokens < 0 or > n_ctx),
 * KVC_ECUDA. */
int kv_cache_truncate(const kvc_cache *cache, int32_t n_tokens, kvc_stream_t stream);

/* ---- diagnostics ------------------------------------------------------------- */

/* A short static description of a status code. */
const char *kvc_strerror(int status);

/* Synchronise the current device, then read and clear the device-side status
 * word that kernels set when a bounded wait gives up (0 = none) into *status.
 * Returns KVC_OK when the word was 0, KVC_EDEVICE when a kernel gave up a wait
 * since the last read (the outputs of that call are undefined; the cache, the
 * context and later calls stay usable), KVC_ECUDA if the synchronisation
 * fails. */
int kvc_device_status(int32_t *status);

/* Test hook for the failure path.  Arms one bounded wait that nothing will
 * satisfy in the next launch of the chosen tensor-core kernel on any device:
 * which = KVC_TEST_PREFILL (the prefill attention pass, head_dim 64 or 128) or
 * KVC_TEST_DECODE (the decode split pass for head_dim 128).  In that launch the
 * thread that issues the MMAs waits on a barrier nothing arrives at, in place
 * of its first wait for a softmax tile; after limit_ns the wait gives up, as
 * any bounded wait does, and every CTA unwinds: the TMA copies and MMAs in
 * flight are let finish, tensor memory is freed, the kernel returns and
 * kvc_device_status reports KVC_EDEVICE.  limit_ns = 0 disarms.  One launch
 * consumes the arm.  The pages define no such call: it exists so that a test
 * can show a wait that gives up leaves a usable context. */
#define KVC_TEST_PREFILL 0
#define KVC_TEST_DECODE 1
int kvc_test_arm_wait_timeout(int32_t which, uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
