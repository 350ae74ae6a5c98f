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
// q8_0: the body is a sequence of 34-byte blocks.  Eight consecutive blocks
// are a 272-byte unit that starts on a 16-byte boundary (32 + 272u), so one
// thread moves one unit: pack loads the eight blocks' 32-byte code runs and
// 2-byte scales and assembles the 17 16-byte output chunks with byte permutes
// (a block pair is 17 words: scale + codes shifted by two bytes, then the
// second scale, then the second block's codes word-aligned); unpack is the
// mirror image.  A last unit with fewer than eight blocks moves halfword by
// halfword.  f16: records are runs of 16-byte chunks; one thread moves four.
// Both are HBM-bound copies with a permutation.
#include <cuda_runtime.h>

#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int THREADS = 256;
constexpr int F16_CHUNKS = 4;   // 16-byte chunks per thread (f16)

struct StateArgs {
    uint8_t *kq, *vq;              // codes (q8_0) or values (f16)
    uint16_t *ks, *vs;             // scales (q8_0)
    Geom g;
    int n_tokens, H, D, nb;
    int64_t n_blocks;              // q8_0: 34-byte blocks in the body
    int64_t n_chunks;              // f16: 16-byte chunks in the body
    uint8_t *body;                 // stream body (after the header)
};

// Coordinates of block `beta` of the body: record (layer, t, kv), head h, block b within the head.
struct BlockPos {
    int layer, t, kv, h, b;
};

__device__ __forceinline__ BlockPos block_pos(const StateArgs &a, int64_t beta) {
    const int bpr = a.H * a.nb;                 // blocks per record
    const int64_t rec = beta / bpr;
    const int within = (int)(beta - rec * bpr);
    BlockPos p;
    p.kv = (int)(rec & 1);
    const int64_t lt = rec >> 1;
    p.layer = (int)(lt / a.n_tokens);
    p.t = (int)(lt - (int64_t)p.layer * a.n_tokens);
    p.h = within / a.nb;
    p.b = within - p.h * a.nb;
    return p;
}

__device__ __forceinline__ void next_block(const StateArgs &a, BlockPos &p) {
    if (++p.b < a.nb) return;
    p.b = 0;
    if (++p.h < a.H) return;
    p.h = 0;
    if (p.kv == 0) {
        p.kv = 1;
        return;
    }
    p.kv = 0;
    if (++p.t < a.n_tokens) return;
    p.t = 0;
    ++p.layer;
}

__device__ __forceinline__ int64_t code_off(const StateArgs &a, const BlockPos &p) {
    return p.layer * a.g.c_layer + (int64_t)p.t * a.g.c_tok + p.h * a.g.c_head + p.b * 32;
}
__device__ __forceinline__ int64_t scale_off(const StateArgs &a, const BlockPos &p) {
    return p.layer * a.g.s_layer + (int64_t)p.t * a.g.s_tok + p.h * a.g.s_head + p.b;
}

// the 68 words of a unit from its eight blocks' scales and code words (block pairs, see the file comment)
__device__ __forceinline__ void assemble(const uint32_t (&sc)[8], const uint4 (&c)[16], uint32_t (&w)[68]) {
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
        const uint32_t a[8] = {c[4 * pr].x, c[4 * pr].y, c[4 * pr].z, c[4 * pr].w,
                               c[4 * pr + 1].x, c[4 * pr + 1].y, c[4 * pr + 1].z, c[4 * pr + 1].w};
        const uint32_t b[8] = {c[4 * pr + 2].x, c[4 * pr + 2].y, c[4 * pr + 2].z, c[4 * pr + 2].w,
                               c[4 * pr + 3].x, c[4 * pr + 3].y, c[4 * pr + 3].z, c[4 * pr + 3].w};
        uint32_t *o = w + 17 * pr;
        o[0] = __byte_perm(sc[2 * pr], a[0], 0x5410);          // scale, codes 0-1
#pragma unroll
        for (int k = 1; k < 8; ++k) o[k] = __byte_perm(a[k - 1], a[k], 0x5432);   // codes 4k-2 .. 4k+1
        o[8] = __byte_perm(a[7], sc[2 * pr + 1], 0x5432);      // codes 30-31, second scale
#pragma unroll
        for (int k = 0; k < 8; ++k) o[9 + k] = b[k];
    }
}

// the inverse: eight scales and code words from the 68 words of a unit
__device__ __forceinline__ void disassemble(const uint32_t (&w)[68], uint32_t (&sc)[8], uint4 (&c)[16]) {
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
        const uint32_t *o = w + 17 * pr;
        uint32_t a[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) a[k] = __byte_perm(o[k], o[k + 1], 0x5432);
        sc[2 * pr] = o[0] & 0xFFFFu;
        sc[2 * pr + 1] = o[8] >> 16;
        c[4 * pr] = make_uint4(a[0], a[1], a[2], a[3]);
        c[4 * pr + 1] = make_uint4(a[4], a[5], a[6], a[7]);
        c[4 * pr + 2] = make_uint4(o[9], o[10], o[11], o[12]);
        c[4 * pr + 3] = make_uint4(o[13], o[14], o[15], o[16]);
    }
}

__global__ void __launch_bounds__(THREADS) pack_q8_kernel(const StateArgs a) {
    const int64_t u = (int64_t)blockIdx.x * THREADS + threadIdx.x;
    const int64_t beta0 = u * 8;
    if (beta0 >= a.n_blocks) return;
    const int nblk = (int)min((int64_t)8, a.n_blocks - beta0);
    uint32_t sc[8];
    uint4 c[16];
    BlockPos p = block_pos(a, beta0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < nblk) {
            const uint8_t *src = (p.kv ? a.vq : a.kq) + code_off(a, p);
            c[2 * i] = __ldg(reinterpret_cast<const uint4 *>(src));
            c[2 * i + 1] = __ldg(reinterpret_cast<const uint4 *>(src) + 1);
            sc[i] = __ldg((p.kv ? a.vs : a.ks) + scale_off(a, p));
            next_block(a, p);
        } else {
            c[2 * i] = c[2 * i + 1] = make_uint4(0u, 0u, 0u, 0u);
            sc[i] = 0u;
        }
    }
    uint32_t w[68];
    assemble(sc, c, w);
    uint8_t *dst = a.body + u * 272;
    if (nblk == 8) {
#pragma unroll
        for (int k = 0; k < 17; ++k)
            *reinterpret_cast<uint4 *>(dst + 16 * k) = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    } else {
        // the body ends inside this unit: 17 halfwords per block
        uint16_t *d16 = reinterpret_cast<uint16_t *>(dst);
#pragma unroll
        for (int x = 0; x < 136; ++x)
            if (x < 17 * nblk) d16[x] = (uint16_t)(w[x >> 1] >> (16 * (x & 1)));
    }
}

__global__ void __launch_bounds__(THREADS) unpack_q8_kernel(const StateArgs a) {
    const int64_t u = (int64_t)blockIdx.x * THREADS + threadIdx.x;
    const int64_t beta0 = u * 8;
    if (beta0 >= a.n_blocks) return;
    const int nblk = (int)min((int64_t)8, a.n_blocks - beta0);
    const uint8_t *src = a.body + u * 272;
    uint32_t w[68];
    if (nblk == 8) {
#pragma unroll
        for (int k = 0; k < 17; ++k) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src) + k);
            w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < 68; ++k) w[k] = 0u;
        const uint16_t *s16 = reinterpret_cast<const uint16_t *>(src);
#pragma unroll
        for (int x = 0; x < 136; ++x)
            if (x < 17 * nblk) w[x >> 1] |= (uint32_t)__ldg(s16 + x) << (16 * (x & 1));
    }
    uint32_t sc[8];
    uint4 c[16];
    disassemble(w, sc, c);
    BlockPos p = block_pos(a, beta0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < nblk) {
            uint8_t *dst = (p.kv ? a.vq : a.kq) + code_off(a, p);
            reinterpret_cast<uint4 *>(dst)[0] = c[2 * i];
            reinterpret_cast<uint4 *>(dst)[1] = c[2 * i + 1];
            (p.kv ? a.vs : a.ks)[scale_off(a, p)] = (uint16_t)sc[i];
            next_block(a, p);
        }
    }
}

// f16: chunk gamma of the body -> (record, head, chunk within the head row)
__device__ __forceinline__ uint8_t *f16_cache_ptr(const StateArgs &a, int64_t gamma) {
    const int cpr = a.D / 8;                    // 16-byte chunks per head row
    const int64_t row = gamma / cpr;            // (record, head) in stream order
    const int ch = (int)(gamma - row * cpr);
    const int64_t rec = row / a.H;
    const int h = (int)(row - rec * a.H);
    const int kv = (int)(rec & 1);
    const int64_t lt = rec >> 1;
    const int layer = (int)(lt / a.n_tokens);
    const int t = (int)(lt - (int64_t)layer * a.n_tokens);
    return (kv ? a.vq : a.kq) + 2 * (layer * a.g.c_layer + (int64_t)t * a.g.c_tok + h * a.g.c_head) + 16 * ch;
}

template <bool PACK>
__global__ void __launch_bounds__(THREADS) copy_f16_kernel(const StateArgs a) {
    const int64_t first = ((int64_t)blockIdx.x * THREADS + threadIdx.x) * F16_CHUNKS;
    uint4 v[F16_CHUNKS];
#pragma unroll
    for (int i = 0; i < F16_CHUNKS; ++i) {
        const int64_t gamma = first + i;
        if (gamma < a.n_chunks)
            v[i] = PACK ? __ldg(reinterpret_cast<const uint4 *>(f16_cache_ptr(a, gamma)))
                        : __ldg(reinterpret_cast<const uint4 *>(a.body) + gamma);
    }
#pragma unroll
    for (int i = 0; i < F16_CHUNKS; ++i) {
        const int64_t gamma = first + i;
        if (gamma < a.n_chunks) {
            if (PACK) reinterpret_cast<uint4 *>(a.body)[gamma] = v[i];
            else *reinterpret_cast<uint4 *>(f16_cache_ptr(a, gamma)) = v[i];
        }
    }
}

StateArgs make_args(const kvc_cache &c, int n_tokens, uint8_t *body) {
    StateArgs a = {};
    a.kq = static_cast<uint8_t *>(c.k_q);
    a.vq = static_cast<uint8_t *>(c.v_q);
    a.ks = static_cast<uint16_t *>(c.k_s);
    a.vs = static_cast<uint16_t *>(c.v_s);
    a.g = geom_of(c.d);
    a.n_tokens = n_tokens;
    a.H = c.d.n_head_kv;
    a.D = c.d.head_dim;
    a.nb = c.d.head_dim / 32;
    const int64_t n_records = (int64_t)c.d.n_layer * n_tokens * 2;
    a.n_blocks = n_records * a.H * a.nb;
    a.n_chunks = n_records * a.H * (a.D / 8);
    a.body = body;
    return a;
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

int grid_for(int64_t work, int per_thread) {
    return (int)((work + (int64_t)THREADS * per_thread - 1) / ((int64_t)THREADS * per_thread));
}

}  // namespace

int launch_state_pack(const kvc_cache &c, int n_tokens, uint8_t *dst, cudaStream_t s) {
    const bool q8 = c.d.type == KVC_Q8_0;
    write_header<<<1, 1, 0, s>>>(dst, c.d.n_layer, c.d.n_head_kv, c.d.head_dim, q8 ? 1u : 0u, n_tokens);
    const StateArgs a = make_args(c, n_tokens, dst + 32);
    if (n_tokens > 0) {
        if (q8) pack_q8_kernel<<<grid_for(a.n_blocks, 8), THREADS, 0, s>>>(a);
        else copy_f16_kernel<true><<<grid_for(a.n_chunks, F16_CHUNKS), THREADS, 0, s>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
}

int launch_state_unpack(const kvc_cache &c, int n_tokens, const uint8_t *src, cudaStream_t s) {
    const bool q8 = c.d.type == KVC_Q8_0;
    const StateArgs a = make_args(c, n_tokens, const_cast<uint8_t *>(src) + 32);
    if (n_tokens > 0) {
        if (q8) unpack_q8_kernel<<<grid_for(a.n_blocks, 8), THREADS, 0, s>>>(a);
        else copy_f16_kernel<false><<<grid_for(a.n_chunks, F16_CHUNKS), THREADS, 0, s>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
}

}  // namespace kvc
