// The C ABI (include/kvc.h): argument checks, size queries and dispatch.
//
// Every check runs before anything is launched, so a call that fails leaves
// the cache untouched and usable - the error contract of the pages' state
// switch (llama.cpp PR #58 "completion : allow the prompt to be processed
// under its own split mode", section "Memory": a mode that does not fit must
// not lose the request; llama.cpp PR #59 "llama : switch the split mode of a
// live context", section "What this adds": the call returns false and the
// caller keeps a working context).
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>

#include "kvc_internal.h"

using namespace kvc;

namespace kvc {
namespace {
std::atomic<uint64_t> g_test_stall[2];   // per kernel kind: wait limit of the armed stall, 0 = none
}  // namespace
void arm_test_stall(int which, uint64_t limit_ns) { g_test_stall[which].store(limit_ns); }
uint64_t take_test_stall(int which) { return g_test_stall[which].exchange(0); }
}  // namespace kvc

namespace {

constexpr uint32_t STATE_MAGIC = 0x3143564Bu;  // 'K' 'V' 'C' '1' little-endian
constexpr uint32_t STATE_VERSION = 1u;
constexpr size_t STATE_HEADER = 32;

bool desc_ok(const kvc_desc *d) {
    if (!d) return false;
    if (d->n_layer <= 0 || d->n_ctx <= 0 || d->n_head_kv <= 0 || d->head_dim <= 0) return false;
    if (d->head_dim % 32 != 0 || d->head_dim > 1024) return false;
    if (d->type != KVC_F16 && d->type != KVC_Q8_0) return false;
    if (d->layout != KVC_HEAD_MAJOR && d->layout != KVC_LAYER_MAJOR) return false;
    return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// True when p is device memory of the current device (or managed memory the runtime attributes to it).
bool on_current_device(const void *p) {
    int dev = -1;
    cudaPointerAttributes at;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();   // a failed query leaves no sticky error behind
        return false;
    }
    return (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) && at.device == dev;
}

bool cache_ok(const kvc_cache *c) {
    if (!c || !desc_ok(&c->d)) return false;
    if (!c->k_q || !c->v_q || !aligned16(c->k_q) || !aligned16(c->v_q)) return false;
    if (c->d.type == KVC_Q8_0 && (!c->k_s || !c->v_s || !aligned16(c->k_s) || !aligned16(c->v_s)))
        return false;
    return true;
}

size_t elems(const kvc_desc &d) { return (size_t)d.n_layer * d.n_ctx * d.n_head_kv * d.head_dim; }

size_t record_bytes(const kvc_desc &d) {
    return d.type == KVC_Q8_0 ? (size_t)d.n_head_kv * (d.head_dim / 32) * 34
                              : (size_t)d.n_head_kv * d.head_dim * 2;
}

bool dtype_ok(int dtype) { return dtype == KVC_IN_F32 || dtype == KVC_IN_BF16 || dtype == KVC_IN_F16; }

}  // namespace

extern "C" {

int kvc_cache_bytes(const kvc_desc *desc, size_t *k_q, size_t *k_s, size_t *v_q, size_t *v_s) {
    if (!desc_ok(desc) || !k_q || !k_s || !v_q || !v_s) return KVC_EINVAL;
    const size_t n = elems(*desc);
    if (desc->type == KVC_Q8_0) {
        *k_q = *v_q = n;
        *k_s = *v_s = n / 32 * 2;
    } else {
        *k_q = *v_q = n * 2;
        *k_s = *v_s = 0;
    }
    return KVC_OK;
}

int kvc_scratch_bytes(const kvc_desc *desc, int32_t n_head_q, size_t *bytes) {
    if (!desc_ok(desc) || !bytes || n_head_q <= 0 || n_head_q % desc->n_head_kv) return KVC_EINVAL;
    *bytes = (size_t)n_head_q * decode_max_split() * (desc->head_dim + 2) * sizeof(float);
    return KVC_OK;
}

size_t kv_state_size(const kvc_desc *desc, int32_t n_tokens) {
    if (!desc_ok(desc) || n_tokens < 0 || n_tokens > desc->n_ctx) return 0;
    return STATE_HEADER + (size_t)desc->n_layer * n_tokens * 2 * record_bytes(*desc);
}

int kvc_cache_init(kvc_cache *out, const kvc_desc *desc, void *k_q, void *k_s, void *v_q, void *v_s) {
    if (!out || !desc_ok(desc)) return KVC_EINVAL;
    kvc_cache c;
    c.d = *desc;
    c.k_q = k_q;
    c.k_s = desc->type == KVC_Q8_0 ? k_s : nullptr;
    c.v_q = v_q;
    c.v_s = desc->type == KVC_Q8_0 ? v_s : nullptr;
    if (!cache_ok(&c)) return KVC_EINVAL;
    *out = c;
    return KVC_OK;
}

int kv_cache_append(const kvc_cache *cache, int32_t layer, int32_t pos0, int32_t n_tokens,
                    const void *k, const void *v, int32_t dtype, kvc_stream_t stream) {
    if (!cache_ok(cache) || !dtype_ok(dtype)) return KVC_EINVAL;
    if (n_tokens < 0) return KVC_EINVAL;
    if (layer < 0 || layer >= cache->d.n_layer || pos0 < 0 || (int64_t)pos0 + n_tokens > cache->d.n_ctx)
        return KVC_ERANGE;
    if (n_tokens == 0) return KVC_OK;
    if (!k || !v || !aligned16(k) || !aligned16(v)) return KVC_EINVAL;
    return launch_append(*cache, layer, pos0, n_tokens, k, v, dtype, (cudaStream_t)stream);
}

int kv_cache_append_batch(const kvc_cache *caches, int32_t n_seq, int32_t layer, const int32_t *pos, const void *k,
                          const void *v, int32_t dtype, kvc_stream_t stream) {
    if (!caches || !pos || n_seq < 1 || n_seq > append_max_batch() || !dtype_ok(dtype)) return KVC_EINVAL;
    const kvc_desc &d = caches[0].d;
    for (int i = 0; i < n_seq; ++i) {
        const kvc_desc &e = caches[i].d;
        if (!cache_ok(&caches[i]) || e.n_head_kv != d.n_head_kv || e.head_dim != d.head_dim || e.type != d.type)
            return KVC_EINVAL;
    }
    for (int i = 0; i < n_seq; ++i)
        if (layer < 0 || layer >= caches[i].d.n_layer || pos[i] < 0 || pos[i] >= caches[i].d.n_ctx) return KVC_ERANGE;
    if (!k || !v || !aligned16(k) || !aligned16(v)) return KVC_EINVAL;
    return launch_append_batch(caches, n_seq, layer, pos, k, v, dtype, (cudaStream_t)stream);
}

int kvc_prefill_scratch_bytes(const kvc_desc *desc, int32_t n_head_q, int32_t max_tokens, size_t *bytes) {
    if (!desc_ok(desc) || !bytes || n_head_q <= 0 || n_head_q % desc->n_head_kv) return KVC_EINVAL;
    if (max_tokens <= 0 || max_tokens > desc->n_ctx) return KVC_ERANGE;
    const size_t b = prefill_scratch_bytes(*desc, n_head_q, max_tokens);
    if (b == 0) return KVC_EINVAL;
    *bytes = b;
    return KVC_OK;
}

int prefill_chunk_attn(const kvc_cache *cache, int32_t layer, int32_t pos0, int32_t n_tokens,
                       const void *q, int32_t dtype, int32_t n_head_q, float *out, void *scratch,
                       size_t scratch_bytes, kvc_stream_t stream) {
    if (!cache_ok(cache) || !dtype_ok(dtype)) return KVC_EINVAL;
    if (cache->d.head_dim != 64 && cache->d.head_dim != 128) return KVC_EINVAL;
    if (n_head_q <= 0 || n_head_q % cache->d.n_head_kv || n_head_q > 65535 || n_tokens < 0) return KVC_EINVAL;
    if (layer < 0 || layer >= cache->d.n_layer || pos0 < 0 || (int64_t)pos0 + n_tokens > cache->d.n_ctx)
        return KVC_ERANGE;
    if (n_tokens == 0) return KVC_OK;
    if (!q || !out || !scratch || !aligned16(q) || !aligned16(out) || !aligned16(scratch)) return KVC_EINVAL;
    return launch_prefill(*cache, layer, pos0, n_tokens, q, dtype, n_head_q, out, scratch, scratch_bytes,
                          (cudaStream_t)stream);
}

int prefill_step(const kvc_cache *cache, int32_t layer, int32_t pos0, int32_t n_tokens, const void *q, const void *k,
                 const void *v, int32_t dtype, int32_t n_head_q, float *out, void *scratch, size_t scratch_bytes,
                 int32_t copy_valid, kvc_stream_t stream) {
    if (!cache_ok(cache) || !dtype_ok(dtype)) return KVC_EINVAL;
    if (cache->d.head_dim != 64 && cache->d.head_dim != 128) return KVC_EINVAL;
    if (n_head_q <= 0 || n_head_q % cache->d.n_head_kv || n_head_q > 65535 || n_tokens < 0) return KVC_EINVAL;
    if (layer < 0 || layer >= cache->d.n_layer || pos0 < 0 || (int64_t)pos0 + n_tokens > cache->d.n_ctx ||
        copy_valid < 0 || copy_valid > pos0)
        return KVC_ERANGE;
    if (n_tokens == 0) return KVC_OK;
    if (!q || !k || !v || !out || !scratch || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
        !aligned16(scratch))
        return KVC_EINVAL;
    return launch_prefill_step(*cache, layer, pos0, n_tokens, q, k, v, dtype, n_head_q, out, scratch, scratch_bytes,
                               copy_valid, (cudaStream_t)stream);
}

int decode_attn(const kvc_cache *cache, int32_t layer, int32_t pos, const void *q, int32_t dtype,
                int32_t n_head_q, float *out, void *scratch, size_t scratch_bytes, kvc_stream_t stream) {
    if (!cache_ok(cache) || !dtype_ok(dtype)) return KVC_EINVAL;
    if (cache->d.head_dim != 64 && cache->d.head_dim != 128) return KVC_EINVAL;
    if (n_head_q <= 0 || n_head_q % cache->d.n_head_kv || n_head_q / cache->d.n_head_kv > 16)
        return KVC_EINVAL;
    if (layer < 0 || layer >= cache->d.n_layer || pos < 0 || pos >= cache->d.n_ctx) return KVC_ERANGE;
    if (!q || !out || !scratch || !aligned16(q) || !aligned16(out) || !aligned16(scratch)) return KVC_EINVAL;
    size_t need = 0;
    kvc_scratch_bytes(&cache->d, n_head_q, &need);
    if (scratch_bytes < need) return KVC_ENOSPC;
    return launch_decode(*cache, layer, pos, q, dtype, n_head_q, out, static_cast<float *>(scratch),
                         (cudaStream_t)stream);
}

int decode_step(const kvc_cache *cache, int32_t layer, int32_t pos, const void *q, const void *k, const void *v,
                int32_t dtype, int32_t n_head_q, float *out, void *scratch, size_t scratch_bytes, kvc_stream_t stream) {
    if (!cache_ok(cache) || !dtype_ok(dtype)) return KVC_EINVAL;
    if (cache->d.head_dim != 64 && cache->d.head_dim != 128) return KVC_EINVAL;
    if (n_head_q <= 0 || n_head_q % cache->d.n_head_kv || n_head_q / cache->d.n_head_kv > 16)
        return KVC_EINVAL;
    if (layer < 0 || layer >= cache->d.n_layer || pos < 0 || pos >= cache->d.n_ctx) return KVC_ERANGE;
    if (!q || !k || !v || !out || !scratch || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
        !aligned16(scratch))
        return KVC_EINVAL;
    size_t need = 0;
    kvc_scratch_bytes(&cache->d, n_head_q, &need);
    if (scratch_bytes < need) return KVC_ENOSPC;
    return launch_decode_step(*cache, layer, pos, q, k, v, dtype, n_head_q, out, static_cast<float *>(scratch),
                              (cudaStream_t)stream);
}

int decode_step_batch(const kvc_cache *caches, int32_t n_seq, int32_t layer, const int32_t *pos, const void *q,
                      const void *k, const void *v, int32_t dtype, int32_t n_head_q, float *out, void *scratch,
                      size_t scratch_bytes, kvc_stream_t stream) {
    if (!caches || !pos || n_seq < 1 || n_seq > decode_max_batch() || !dtype_ok(dtype)) return KVC_EINVAL;
    const kvc_desc &d = caches[0].d;
    for (int i = 0; i < n_seq; ++i) {
        const kvc_desc &e = caches[i].d;
        if (!cache_ok(&caches[i]) || e.n_layer != d.n_layer || e.n_ctx != d.n_ctx || e.n_head_kv != d.n_head_kv ||
            e.head_dim != d.head_dim || e.type != d.type)
            return KVC_EINVAL;
    }
    if (d.head_dim != 64 && d.head_dim != 128) return KVC_EINVAL;
    if (n_head_q <= 0 || n_head_q % d.n_head_kv || n_head_q / d.n_head_kv > 16) return KVC_EINVAL;
    for (int i = 0; i < n_seq; ++i)
        if (layer < 0 || layer >= d.n_layer || pos[i] < 0 || pos[i] >= d.n_ctx) return KVC_ERANGE;
    if (!q || !k || !v || !out || !scratch || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
        !aligned16(scratch))
        return KVC_EINVAL;
    size_t need = 0;
    kvc_scratch_bytes(&d, n_head_q, &need);
    if (scratch_bytes / (size_t)n_seq < need) return KVC_ENOSPC;
    return launch_decode_step_batch(caches, n_seq, layer, pos, q, k, v, dtype, n_head_q, out,
                                    static_cast<float *>(scratch), need, (cudaStream_t)stream);
}

int decode_attn_noalloc(const kvc_cache *cache, int32_t layer, int32_t pos, const void *q, int32_t dtype,
                        int32_t n_head_q, float *out, kvc_stream_t stream) {
    if (!cache_ok(cache) || !dtype_ok(dtype)) return KVC_EINVAL;
    if (cache->d.head_dim != 64 && cache->d.head_dim != 128) return KVC_EINVAL;
    if (n_head_q <= 0 || n_head_q % cache->d.n_head_kv || n_head_q / cache->d.n_head_kv > 16)
        return KVC_EINVAL;
    if (layer < 0 || layer >= cache->d.n_layer || pos < 0 || pos >= cache->d.n_ctx) return KVC_ERANGE;
    if (!q || !out || !aligned16(q) || !aligned16(out)) return KVC_EINVAL;
    size_t need = 0;
    kvc_scratch_bytes(&cache->d, n_head_q, &need);
    if (need > decode_noalloc_capacity()) return KVC_ENOSPC;  // more partials than the fixed array holds
    // the partials go to the current device's array: the cache and the output must live there too
    if (!on_current_device(cache->k_q) || !on_current_device(out)) return KVC_EINVAL;
    return launch_decode_noalloc(*cache, layer, pos, q, dtype, n_head_q, out, (cudaStream_t)stream);
}

int decode_attn_batch(const kvc_cache *caches, int32_t n_seq, int32_t layer, const int32_t *pos, const void *q,
                      int32_t dtype, int32_t n_head_q, float *out, void *scratch, size_t scratch_bytes,
                      kvc_stream_t stream) {
    if (!caches || !pos || n_seq < 1 || n_seq > decode_max_batch() || !dtype_ok(dtype)) return KVC_EINVAL;
    const kvc_desc &d = caches[0].d;
    for (int i = 0; i < n_seq; ++i) {
        const kvc_desc &e = caches[i].d;
        if (!cache_ok(&caches[i]) || e.n_layer != d.n_layer || e.n_ctx != d.n_ctx || e.n_head_kv != d.n_head_kv ||
            e.head_dim != d.head_dim || e.type != d.type)
            return KVC_EINVAL;
    }
    if (d.head_dim != 64 && d.head_dim != 128) return KVC_EINVAL;
    if (n_head_q <= 0 || n_head_q % d.n_head_kv || n_head_q / d.n_head_kv > 16) return KVC_EINVAL;
    if (layer < 0 || layer >= d.n_layer) return KVC_ERANGE;
    for (int i = 0; i < n_seq; ++i)
        if (pos[i] < 0 || pos[i] >= d.n_ctx) return KVC_ERANGE;
    if (!q || !out || !scratch || !aligned16(q) || !aligned16(out) || !aligned16(scratch)) return KVC_EINVAL;
    size_t need = 0;
    kvc_scratch_bytes(&d, n_head_q, &need);
    if (scratch_bytes / (size_t)n_seq < need) return KVC_ENOSPC;
    return launch_decode_batch(caches, n_seq, layer, pos, q, dtype, n_head_q, out, static_cast<float *>(scratch),
                               need, (cudaStream_t)stream);
}

int kv_state_get(const kvc_cache *cache, int32_t n_tokens, void *dst, size_t dst_bytes, kvc_stream_t stream) {
    if (!cache_ok(cache) || !dst || !aligned16(dst) || n_tokens < 0) return KVC_EINVAL;
    if (n_tokens > cache->d.n_ctx) return KVC_ERANGE;
    if (dst_bytes < kv_state_size(&cache->d, n_tokens)) return KVC_ENOSPC;
    return launch_state_pack(*cache, n_tokens, static_cast<uint8_t *>(dst), (cudaStream_t)stream);
}

int kv_state_set(kvc_cache *cache, const void *src, size_t src_bytes, int32_t *n_tokens_out,
                 kvc_stream_t stream) {
    if (!cache_ok(cache) || !src || !aligned16(src) || !n_tokens_out) return KVC_EINVAL;
    if (src_bytes < STATE_HEADER) return KVC_EFORMAT;
    uint32_t h[8];
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(h, src, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return KVC_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVC_ECUDA;
    const kvc_desc &d = cache->d;
    if (h[0] != STATE_MAGIC || h[1] != STATE_VERSION) return KVC_EFORMAT;
    if (h[2] != (uint32_t)d.n_layer || h[3] != (uint32_t)d.n_head_kv || h[4] != (uint32_t)d.head_dim ||
        h[5] != (uint32_t)d.type || h[7] != 0u)
        return KVC_EFORMAT;
    if (h[6] > (uint32_t)d.n_ctx) return KVC_EFORMAT;
    const int32_t n = (int32_t)h[6];
    if (src_bytes != kv_state_size(&d, n)) return KVC_EFORMAT;
    const int rc = launch_state_unpack(*cache, n, static_cast<const uint8_t *>(src), s);
    if (rc == KVC_OK) *n_tokens_out = n;
    return rc;
}

int kv_state_get_heads(const kvc_cache *cache, int32_t head0, int32_t n_head_total, int32_t n_tokens, void *dst,
                       size_t dst_bytes, kvc_stream_t stream) {
    if (!cache_ok(cache) || !dst || !aligned16(dst) || n_tokens < 0) return KVC_EINVAL;
    if (head0 < 0 || n_head_total <= 0 || (int64_t)head0 + cache->d.n_head_kv > n_head_total) return KVC_EINVAL;
    if (n_tokens > cache->d.n_ctx) return KVC_ERANGE;
    kvc_desc whole = cache->d;
    whole.n_head_kv = n_head_total;
    if (dst_bytes < kv_state_size(&whole, n_tokens)) return KVC_ENOSPC;
    return launch_state_pack_heads(*cache, head0, n_head_total, n_tokens, static_cast<uint8_t *>(dst),
                                   (cudaStream_t)stream);
}

int kv_state_set_heads(kvc_cache *cache, int32_t head0, const void *src, size_t src_bytes, int32_t *n_tokens_out,
                       kvc_stream_t stream) {
    if (!cache_ok(cache) || !src || !aligned16(src) || !n_tokens_out || head0 < 0) return KVC_EINVAL;
    if (src_bytes < STATE_HEADER) return KVC_EFORMAT;
    uint32_t h[8];
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(h, src, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return KVC_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVC_ECUDA;
    const kvc_desc &d = cache->d;
    if (h[0] != STATE_MAGIC || h[1] != STATE_VERSION) return KVC_EFORMAT;
    if (h[2] != (uint32_t)d.n_layer || h[4] != (uint32_t)d.head_dim || h[5] != (uint32_t)d.type || h[7] != 0u)
        return KVC_EFORMAT;
    if (h[3] == 0u || h[3] > 65536u || (uint64_t)head0 + d.n_head_kv > h[3]) return KVC_EFORMAT;
    if (h[6] > (uint32_t)d.n_ctx) return KVC_EFORMAT;
    const int32_t n = (int32_t)h[6];
    kvc_desc whole = d;
    whole.n_head_kv = (int32_t)h[3];
    if (src_bytes != kv_state_size(&whole, n)) return KVC_EFORMAT;
    const int rc = launch_state_unpack_heads(*cache, head0, (int)h[3], n, static_cast<const uint8_t *>(src), s);
    if (rc == KVC_OK) *n_tokens_out = n;
    return rc;
}

int kv_cache_truncate(const kvc_cache *cache, int32_t n_tokens, kvc_stream_t stream) {
    if (!cache_ok(cache)) return KVC_EINVAL;
    const kvc_desc &d = cache->d;
    if (n_tokens < 0 || n_tokens > d.n_ctx) return KVC_ERANGE;
    if (n_tokens == d.n_ctx) return KVC_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t T = d.n_ctx, n = n_tokens, H = d.n_head_kv, L = d.n_layer;
    // one strided fill per buffer: rows of positions [0, n_ctx), their tail [n_tokens, n_ctx) cleared
    auto clear = [&](void *buf, size_t row_bytes) -> bool {  // row_bytes: one position of one row
        const bool hm = d.layout == KVC_HEAD_MAJOR;
        const size_t per_pos = hm ? row_bytes : row_bytes * H;   // bytes of one position in a row
        const size_t rows = hm ? H * L : L;
        return cudaMemset2DAsync(static_cast<uint8_t *>(buf) + n * per_pos, T * per_pos, 0, (T - n) * per_pos, rows,
                                 s) == cudaSuccess;
    };
    const size_t code_bytes = (size_t)d.head_dim * (d.type == KVC_Q8_0 ? 1 : 2);
    if (!clear(cache->k_q, code_bytes) || !clear(cache->v_q, code_bytes)) return KVC_ECUDA;
    if (d.type == KVC_Q8_0) {
        const size_t scale_bytes = (size_t)(d.head_dim / 32) * 2;
        if (!clear(cache->k_s, scale_bytes) || !clear(cache->v_s, scale_bytes)) return KVC_ECUDA;
    }
    return KVC_OK;
}

const char *kvc_strerror(int status) {
    switch (status) {
        case KVC_OK: return "ok";
        case KVC_EINVAL: return "invalid argument";
        case KVC_ERANGE: return "layer or position outside the cache";
        case KVC_ENOSPC: return "destination or scratch buffer too small";
        case KVC_EFORMAT: return "state stream does not match its header or the cache";
        case KVC_ECUDA: return "CUDA call or launch failed";
        case KVC_EDEVICE: return "a kernel gave up a bounded wait";
        default: return "unknown status";
    }
}

int kvc_device_status(int32_t *status) {
    if (!status) return KVC_EINVAL;
    const int rc = read_and_clear_device_status(status);
    if (rc != KVC_OK) return rc;
    return *status != 0 ? KVC_EDEVICE : KVC_OK;
}

int kvc_test_arm_wait_timeout(int32_t which, uint64_t limit_ns) {
    if (which != KVC_TEST_PREFILL && which != KVC_TEST_DECODE) return KVC_EINVAL;
    arm_test_stall(which, limit_ns);
    return KVC_OK;
}

}  // extern "C"
