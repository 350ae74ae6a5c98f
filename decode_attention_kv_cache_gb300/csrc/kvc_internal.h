// Internal declarations shared by the C-ABI layer and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

// Element strides of one cache buffer family.  Element (layer, pos, head, i)
// of the codes sits at layer*c_layer + pos*c_tok + head*c_head + i; the scale
// of block b at layer*s_layer + pos*s_tok + head*s_head + b.
struct Geom {
    int64_t c_layer, c_tok, c_head;
    int64_t s_layer, s_tok, s_head;
};

inline Geom geom_of(const kvc_desc &d) {
    const int64_t D = d.head_dim, nb = d.head_dim / 32, H = d.n_head_kv, L = d.n_layer, T = d.n_ctx;
    Geom g;
    if (d.layout == KVC_HEAD_MAJOR) {
        g.c_head = L * T * D; g.c_layer = T * D; g.c_tok = D;
        g.s_head = L * T * nb; g.s_layer = T * nb; g.s_tok = nb;
    } else {
        g.c_layer = T * H * D; g.c_tok = H * D; g.c_head = D;
        g.s_layer = T * H * nb; g.s_tok = H * nb; g.s_head = nb;
    }
    return g;
}

inline int dtype_bytes(int dtype) { return dtype == KVC_IN_F32 ? 4 : 2; }


// A 3-D tiled TMA tensor map (dims innermost first, strides of dims 1 and 2 in bytes); false when
// the driver entry point is missing or the encoding is rejected.
bool make_map_3d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t d0, uint64_t d1,
                 uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1,
                 uint32_t b2, CUtensorMapSwizzle sw);
// Streaming multiprocessors of the current device (cached per device).
int sm_count();
// Raise `kernel`'s dynamic shared memory limit to `bytes` on the current device, once per device (the
// attribute belongs to the device's context).  KVC_OK or KVC_ECUDA.
int allow_dynamic_smem(const void *kernel, int bytes);

// Launchers: arguments are already validated; return KVC_OK or KVC_ECUDA.
int launch_append(const kvc_cache &c, int layer, int pos0, int n_tokens, const void *k,
                  const void *v, int dtype, cudaStream_t s);
int append_max_batch();
int launch_append_batch(const kvc_cache *caches, int n_seq, int layer, const int *pos, const void *k, const void *v,
                        int dtype, cudaStream_t s);
size_t prefill_scratch_bytes(const kvc_desc &d, int n_head_q, int max_tokens);
int launch_prefill(const kvc_cache &c, int layer, int pos0, int n_tokens, const void *q, int dtype,
                   int n_head_q, float *out, void *scratch, size_t scratch_bytes, cudaStream_t s);
int launch_prefill_step(const kvc_cache &c, int layer, int pos0, int n_tokens, const void *q, const void *k,
                        const void *v, int dtype, int n_head_q, float *out, void *scratch, size_t scratch_bytes,
                        int copy_valid, cudaStream_t s);
int decode_max_split();
int launch_decode(const kvc_cache &c, int layer, int pos, const void *q, int dtype, int n_head_q,
                  float *out, float *scratch, cudaStream_t s);
int launch_decode_step(const kvc_cache &c, int layer, int pos, const void *q, const void *k, const void *v, int dtype,
                       int n_head_q, float *out, float *scratch, cudaStream_t s);
int launch_decode_step_batch(const kvc_cache *caches, int n_seq, int layer, const int *pos, const void *q, const void *k,
                             const void *v, int dtype, int n_head_q, float *out, float *scratch,
                             size_t seq_scratch_bytes, cudaStream_t s);
int decode_max_batch();
int launch_decode_batch(const kvc_cache *caches, int n_seq, int layer, const int *pos, const void *q, int dtype,
                        int n_head_q, float *out, float *scratch, size_t seq_scratch_bytes, cudaStream_t s);
size_t decode_noalloc_capacity();
int launch_decode_noalloc(const kvc_cache &c, int layer, int pos, const void *q, int dtype, int n_head_q,
                          float *out, cudaStream_t s);
int launch_state_pack(const kvc_cache &c, int n_tokens, uint8_t *dst, cudaStream_t s);
int launch_state_unpack(const kvc_cache &c, int n_tokens, const uint8_t *src, cudaStream_t s);
int launch_state_pack_heads(const kvc_cache &c, int head0, int H_total, int n_tokens, uint8_t *dst, cudaStream_t s);
int launch_state_unpack_heads(const kvc_cache &c, int head0, int H_total, int n_tokens, const uint8_t *src,
                              cudaStream_t s);

// Test hook of the failure path: the wait limit (ns) of a stall armed for the next launch of a kernel
// kind (KVC_TEST_PREFILL / KVC_TEST_DECODE), 0 when none; take_ consumes it.
void arm_test_stall(int which, uint64_t limit_ns);
uint64_t take_test_stall(int which);

// Device status word set by kernels that give up a bounded wait (all kernels' words, read and cleared).
int read_and_clear_device_status(int32_t *status);
int read_and_clear_decode_status(int32_t *status);

}  // namespace kvc
