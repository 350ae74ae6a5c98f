// State pack / unpack: the cache (either device layout) <-> the
// layout-independent byte stream.
//
// The pages carry a sequence's cache across a change of split mode through a
// serialised state that restores byte-identical into a cache split by layer or
// split by head (llama.cpp PR #58 "completion : allow the prompt to be
// processed under its own split mode", section "What this does"; llama.cpp
// PR #59 "llama : switch the split mode of a live context", section "What
// this adds", step 1).  Stream format (the project's own; the pages fix none):
// a 32-byte header, then per layer, per position, the K record and the V
// record; a record lists the kv heads in order, each as head_dim/32 blocks of
// [fp16 scale][32 int8 codes] (q8_0) or head_dim fp16 values (f16).
//
// Every unit of the stream is a 2-byte halfword (a 34-byte q8_0 block is 17
// halfwords: the scale, then 16 code pairs).  A CTA takes RPC consecutive
// records (RPC a multiple of 8, so its share of the stream starts on a 16-byte
// boundary): pack loads the records' codes and scales with 16-byte loads into
// shared memory, then assembles 16-byte output chunks from halfwords; unpack
// does the reverse.  Both are HBM-bound copies with a permutation.
#include <cuda_runtime.h>

#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int THREADS = 256;

struct StateArgs {
    const uint8_t *kq, *vq;        // codes (q8_0) or values (f16)
    const uint16_t *ks, *vs;       // scales (q8_0)
    uint8_t *kq_w, *vq_w;          // same, writable (unpack)
    uint16_t *ks_w, *vs_w;
    Geom g;
    int n_tokens, H, D, nb, n_records, rpc;
    int rec_hw;                    // halfwords per record
    uint8_t *out;                  // stream body (pack)
    const uint8_t *in;             // stream body (unpack)
};

// Record rho = (layer * n_tokens + t) * 2 + kv.
__device__ __forceinline__ void record_coords(int rho, int n_tokens, int &layer, int &t, int &kv) {
    kv = rho & 1;
    const int lt = rho >> 1;
    layer = lt / n_tokens;
    t = lt - layer * n_tokens;
}

template <bool Q8>
__global__ void __launch_bounds__(THREADS) pack_kernel(const StateArgs a) {
    extern __shared__ uint4 smem4[];
    uint8_t *s_codes = reinterpret_cast<uint8_t *>(smem4);
    const int esz = Q8 ? 1 : 2;
    const int row_bytes = a.D * esz;                // one head's codes of one record
    const int rec_code_bytes = a.H * row_bytes;
    uint16_t *s_scales = reinterpret_cast<uint16_t *>(s_codes + a.rpc * rec_code_bytes);
    const int rec0 = blockIdx.x * a.rpc;
    const int nrec = min(a.rpc, a.n_records - rec0);

    // 1. gather codes (16-byte chunks) and scales into shared memory, record by record
    const int chunks_per_row = row_bytes / 16;
    const int chunks_per_rec = a.H * chunks_per_row;
    for (int i = threadIdx.x; i < nrec * chunks_per_rec; i += THREADS) {
        const int r = i / chunks_per_rec, rem = i - r * chunks_per_rec;
        const int h = rem / chunks_per_row, c = rem - h * chunks_per_row;
        int layer, t, kv;
        record_coords(rec0 + r, a.n_tokens, layer, t, kv);
        const uint8_t *src = (kv ? a.vq : a.kq) +
                             (layer * a.g.c_layer + (int64_t)t * a.g.c_tok + h * a.g.c_head) * esz + c * 16;
        *reinterpret_cast<uint4 *>(s_codes + r * rec_code_bytes + h * row_bytes + c * 16) =
            __ldg(reinterpret_cast<const uint4 *>(src));
    }
    if (Q8) {
        const int per_rec = a.H * a.nb;
        for (int i = threadIdx.x; i < nrec * per_rec; i += THREADS) {
            const int r = i / per_rec, rem = i - r * per_rec;
            const int h = rem / a.nb, b = rem - h * a.nb;
            int layer, t, kv;
            record_coords(rec0 + r, a.n_tokens, layer, t, kv);
            s_scales[i] = __ldg((kv ? a.vs : a.ks) + layer * a.g.s_layer + (int64_t)t * a.g.s_tok +
                                h * a.g.s_head + b);
        }
    }
    __syncthreads();

    // 2. assemble the stream: halfword x of record r is
    //    q8_0: block k = x / 17, m = x % 17 -> m == 0 ? scale k : code pair (m - 1) of block k
    //    f16:  value x of the record (heads in order)
    const uint16_t *s_hw = reinterpret_cast<const uint16_t *>(s_codes);
    const int total_hw = nrec * a.rec_hw;
    uint8_t *dst = a.out + (int64_t)rec0 * a.rec_hw * 2;
    auto hw_at = [&](int u) -> uint32_t {
        const int r = u / a.rec_hw, x = u - r * a.rec_hw;
        if (Q8) {
            const int k = x / 17, m = x - k * 17;
            return m == 0 ? s_scales[r * a.H * a.nb + k]
                          : s_hw[(r * rec_code_bytes + k * 32) / 2 + (m - 1)];
        }
        return s_hw[r * (rec_code_bytes / 2) + x];
    };
    const int n_vec = total_hw / 8;
    for (int i = threadIdx.x; i < n_vec; i += THREADS) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = hw_at(8 * i + 2 * j) | (hw_at(8 * i + 2 * j + 1) << 16);
        *reinterpret_cast<uint4 *>(dst + 16 * i) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    for (int u = n_vec * 8 + threadIdx.x; u < total_hw; u += THREADS)
        reinterpret_cast<uint16_t *>(dst)[u] = (uint16_t)hw_at(u);
}

template <bool Q8>
__global__ void __launch_bounds__(THREADS) unpack_kernel(const StateArgs a) {
    extern __shared__ uint4 smem4[];
    uint16_t *s_hw = reinterpret_cast<uint16_t *>(smem4);
    const int rec0 = blockIdx.x * a.rpc;
    const int nrec = min(a.rpc, a.n_records - rec0);
    const int total_hw = nrec * a.rec_hw;
    const uint8_t *src = a.in + (int64_t)rec0 * a.rec_hw * 2;

    // 1. stage the records' stream bytes
    const int n_vec = total_hw / 8;
    for (int i = threadIdx.x; i < n_vec; i += THREADS)
        smem4[i] = __ldg(reinterpret_cast<const uint4 *>(src) + i);
    for (int u = n_vec * 8 + threadIdx.x; u < total_hw; u += THREADS)
        s_hw[u] = __ldg(reinterpret_cast<const uint16_t *>(src) + u);
    __syncthreads();

    // 2. scatter: 16 bytes of one head's codes (or values) per thread
    const int esz = Q8 ? 1 : 2;
    const int row_bytes = a.D * esz;
    const int chunks_per_row = row_bytes / 16;
    const int chunks_per_rec = a.H * chunks_per_row;
    for (int i = threadIdx.x; i < nrec * chunks_per_rec; i += THREADS) {
        const int r = i / chunks_per_rec, rem = i - r * chunks_per_rec;
        const int h = rem / chunks_per_row, c = rem - h * chunks_per_row;
        int layer, t, kv;
        record_coords(rec0 + r, a.n_tokens, layer, t, kv);
        int x0;  // first stream halfword of these 16 bytes within the record
        if (Q8) {
            const int k = h * a.nb + (c * 16) / 32;          // block
            x0 = k * 17 + 1 + ((c * 16) % 32) / 2;
        } else {
            x0 = h * a.D + c * 8;
        }
        const uint16_t *p = s_hw + r * a.rec_hw + x0;
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = (uint32_t)p[2 * j] | ((uint32_t)p[2 * j + 1] << 16);
        uint8_t *dst = (kv ? a.vq_w : a.kq_w) +
                       (layer * a.g.c_layer + (int64_t)t * a.g.c_tok + h * a.g.c_head) * esz + c * 16;
        *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (Q8) {
        const int per_rec = a.H * a.nb;
        for (int i = threadIdx.x; i < nrec * per_rec; i += THREADS) {
            const int r = i / per_rec, k = i - r * per_rec;
            const int h = k / a.nb, b = k - h * a.nb;
            int layer, t, kv;
            record_coords(rec0 + r, a.n_tokens, layer, t, kv);
            (kv ? a.vs_w : a.ks_w)[layer * a.g.s_layer + (int64_t)t * a.g.s_tok + h * a.g.s_head + b] =
                s_hw[r * a.rec_hw + k * 17];
        }
    }
}

StateArgs make_args(const kvc_cache &c, int n_tokens) {
    StateArgs a = {};
    a.kq = static_cast<const uint8_t *>(c.k_q);
    a.vq = static_cast<const uint8_t *>(c.v_q);
    a.ks = static_cast<const uint16_t *>(c.k_s);
    a.vs = static_cast<const uint16_t *>(c.v_s);
    a.kq_w = static_cast<uint8_t *>(c.k_q);
    a.vq_w = static_cast<uint8_t *>(c.v_q);
    a.ks_w = static_cast<uint16_t *>(c.k_s);
    a.vs_w = static_cast<uint16_t *>(c.v_s);
    a.g = geom_of(c.d);
    a.n_tokens = n_tokens;
    a.H = c.d.n_head_kv;
    a.D = c.d.head_dim;
    a.nb = c.d.head_dim / 32;
    a.n_records = c.d.n_layer * n_tokens * 2;
    const bool q8 = c.d.type == KVC_Q8_0;
    const int rec_bytes = q8 ? a.H * a.nb * 34 : a.H * a.D * 2;
    a.rec_hw = rec_bytes / 2;
    // records per CTA: a multiple of 8 (16-byte aligned CTA boundaries), about 16 KB of stream
    int rpc = (16384 / rec_bytes) / 8 * 8;
    a.rpc = rpc < 8 ? 8 : rpc;
    return a;
}

size_t pack_smem(const StateArgs &a, bool q8) {
    const size_t codes = (size_t)a.rpc * a.H * a.D * (q8 ? 1 : 2);
    return codes + (q8 ? (size_t)a.rpc * a.H * a.nb * 2 : 0);
}

__global__ void write_header(uint8_t *dst, uint32_t n_layer, uint32_t H, uint32_t D, uint32_t type,
                             uint32_t n_tokens) {
    uint32_t *w = reinterpret_cast<uint32_t *>(dst);
    w[0] = 0x3143564Bu;  // 'K' 'V' 'C' '1'
    w[1] = 1u;
    w[2] = n_layer;
    w[3] = H;
    w[4] = D;
    w[5] = type;
    w[6] = n_tokens;
    w[7] = 0u;
}

}  // namespace

int launch_state_pack(const kvc_cache &c, int n_tokens, uint8_t *dst, cudaStream_t s) {
    const bool q8 = c.d.type == KVC_Q8_0;
    write_header<<<1, 1, 0, s>>>(dst, c.d.n_layer, c.d.n_head_kv, c.d.head_dim, q8 ? 1u : 0u, n_tokens);
    StateArgs a = make_args(c, n_tokens);
    a.out = dst + 32;
    if (a.n_records > 0) {
        const size_t smem = pack_smem(a, q8);
        const int grid = (a.n_records + a.rpc - 1) / a.rpc;
        if (q8) {
            if (smem > 48 * 1024 && cudaFuncSetAttribute(pack_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         (int)smem) != cudaSuccess)
                return KVC_ECUDA;
            pack_kernel<true><<<grid, THREADS, smem, s>>>(a);
        } else {
            if (smem > 48 * 1024 && cudaFuncSetAttribute(pack_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         (int)smem) != cudaSuccess)
                return KVC_ECUDA;
            pack_kernel<false><<<grid, THREADS, smem, s>>>(a);
        }
    }
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
}

int launch_state_unpack(const kvc_cache &c, int n_tokens, const uint8_t *src, cudaStream_t s) {
    const bool q8 = c.d.type == KVC_Q8_0;
    StateArgs a = make_args(c, n_tokens);
    a.in = src + 32;
    if (a.n_records > 0) {
        const size_t smem = ((size_t)a.rpc * a.rec_hw * 2 + 15) / 16 * 16;
        const int grid = (a.n_records + a.rpc - 1) / a.rpc;
        if (q8) {
            if (smem > 48 * 1024 && cudaFuncSetAttribute(unpack_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         (int)smem) != cudaSuccess)
                return KVC_ECUDA;
            unpack_kernel<true><<<grid, THREADS, smem, s>>>(a);
        } else {
            if (smem > 48 * 1024 && cudaFuncSetAttribute(unpack_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                         (int)smem) != cudaSuccess)
                return KVC_ECUDA;
            unpack_kernel<false><<<grid, THREADS, smem, s>>>(a);
        }
    }
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
}

}  // namespace kvc
