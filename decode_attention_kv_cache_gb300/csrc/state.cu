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
// are a 272-byte unit that starts on a 16-byte boundary (32 + 272u); a lane
// assembles one unit from its eight blocks' 32-byte code runs and 2-byte
// scales with byte permutes (a block pair is 17 words: scale + codes shifted
// by two bytes, then the second scale, then the second block's codes
// word-aligned), and unpack splits it the same way back.  A warp takes 32
// consecutive units through shared memory, so that both sides move in long
// runs: the cache side as 16-byte code chunks with consecutive lanes on
// consecutive chunks (8 lanes per 128-byte row of a head) and 2-byte scales,
// the stream side as the warp's 8704 contiguous bytes, 16 per lane.  The
// stream's last bytes (a body that ends inside a 16-byte chunk) move halfword
// by halfword.  f16: records are runs of 16-byte chunks; a warp moves 128 consecutive chunks, lane by
// lane.
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
    uint32_t hdr[8];               // pack: the header words, written by the first block before the body
};

// pack: the first block's first two threads write the 32-byte header in front of the body
__device__ __forceinline__ void write_header_words(const StateArgs &a) {
    if (blockIdx.x == 0 && threadIdx.x < 2)
        reinterpret_cast<uint4 *>(a.body - 32)[threadIdx.x] =
            make_uint4(a.hdr[4 * threadIdx.x], a.hdr[4 * threadIdx.x + 1], a.hdr[4 * threadIdx.x + 2],
                       a.hdr[4 * threadIdx.x + 3]);
}

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

// p moved on by n blocks in stream order (n >= 0)
__device__ __forceinline__ void advance(const StateArgs &a, BlockPos &p, int n) {
    const int bpr = a.H * a.nb;
    int within = p.h * a.nb + p.b + n;
    while (within >= bpr) {
        within -= bpr;
        if (p.kv == 0) {
            p.kv = 1;
        } else {
            p.kv = 0;
            if (++p.t == a.n_tokens) {
                p.t = 0;
                ++p.layer;
            }
        }
    }
    p.h = within / a.nb;
    p.b = within - p.h * a.nb;
}

constexpr int QW = 4;                    // warps per CTA (q8_0 pack and unpack)
constexpr int WARP_UNITS = 32;
constexpr int WARP_BLOCKS = 8 * WARP_UNITS;
constexpr int WARP_BYTES = 272 * WARP_UNITS;

struct __align__(16) WarpStage {
    uint8_t buf[WARP_BYTES];             // the warp's block codes (swizzled chunks), then its 32 units
    uint16_t sc[WARP_BLOCKS];            // the warp's block scales
};

// Position of 16-byte code chunk c (block c / 2, half c % 2) in the staging: XOR-swizzled so that a
// lane reading its unit's 16 consecutive chunks and lanes writing consecutive chunks are both free
// of bank conflicts.
__device__ __forceinline__ int phys_chunk(int c) { return c ^ ((c >> 4) & 7); }

__global__ void __launch_bounds__(QW * 32) pack_q8_kernel(const StateArgs a) {
    write_header_words(a);
    __shared__ WarpStage stage[QW];
    const int lane = threadIdx.x & 31;
    WarpStage &S = stage[threadIdx.x >> 5];
    const int64_t wg = (int64_t)blockIdx.x * QW + (threadIdx.x >> 5);
    const int64_t beta0 = wg * WARP_BLOCKS;
    if (beta0 >= a.n_blocks) return;   // the whole warp
    {
        // code chunk 32 m + lane of the warp: block beta0 + 16 m + lane / 2, half lane % 2
        uint4 v[16];
        BlockPos p = block_pos(a, beta0 + (lane >> 1));
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            v[m] = make_uint4(0u, 0u, 0u, 0u);
            if (beta0 + 16 * m + (lane >> 1) < a.n_blocks)
                v[m] = __ldg(reinterpret_cast<const uint4 *>((p.kv ? a.vq : a.kq) + code_off(a, p)) + (lane & 1));
            if (m < 15) advance(a, p, 16);
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) *reinterpret_cast<uint4 *>(S.buf + 16 * phys_chunk(32 * m + lane)) = v[m];
        // scale of block beta0 + 32 m + lane
        uint16_t s8[8];
        BlockPos q = block_pos(a, beta0 + lane);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            s8[m] = 0;
            if (beta0 + 32 * m + lane < a.n_blocks) s8[m] = __ldg((q.kv ? a.vs : a.ks) + scale_off(a, q));
            if (m < 7) advance(a, q, 32);
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) S.sc[32 * m + lane] = s8[m];
    }
    __syncwarp();
    // my unit: blocks 8 lane .. 8 lane + 7, i.e. chunks 16 lane .. 16 lane + 15
    uint4 c[16];
    uint32_t sc[8];
#pragma unroll
    for (int k = 0; k < 16; ++k) c[k] = *reinterpret_cast<const uint4 *>(S.buf + 16 * phys_chunk(16 * lane + k));
    {
        const uint4 s4 = *reinterpret_cast<const uint4 *>(S.sc + 8 * lane);
        const uint32_t sw[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) sc[i] = (sw[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
    }
    __syncwarp();
    uint32_t w[68];
    assemble(sc, c, w);
#pragma unroll
    for (int k = 0; k < 17; ++k)
        *reinterpret_cast<uint4 *>(S.buf + 272 * lane + 16 * k) = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    __syncwarp();
    // the warp's stream bytes (the body may end inside them)
    const int64_t off0 = wg * WARP_BYTES;
    const int nbytes = (int)min((int64_t)WARP_BYTES, a.n_blocks * 34 - off0);
#pragma unroll
    for (int m = 0; m < 17; ++m) {
        const int o = 16 * (32 * m + lane);
        if (o + 16 <= nbytes) {
            *reinterpret_cast<uint4 *>(a.body + off0 + o) = *reinterpret_cast<const uint4 *>(S.buf + o);
        } else if (o < nbytes) {
            for (int x = o; x < nbytes; x += 2)
                *reinterpret_cast<uint16_t *>(a.body + off0 + x) = *reinterpret_cast<const uint16_t *>(S.buf + x);
        }
    }
}

__global__ void __launch_bounds__(QW * 32) unpack_q8_kernel(const StateArgs a) {
    __shared__ WarpStage stage[QW];
    const int lane = threadIdx.x & 31;
    WarpStage &S = stage[threadIdx.x >> 5];
    const int64_t wg = (int64_t)blockIdx.x * QW + (threadIdx.x >> 5);
    const int64_t beta0 = wg * WARP_BLOCKS;
    if (beta0 >= a.n_blocks) return;   // the whole warp
    // the warp's stream bytes into the staging (zero past the body's end)
    const int64_t off0 = wg * WARP_BYTES;
    const int nbytes = (int)min((int64_t)WARP_BYTES, a.n_blocks * 34 - off0);
    {
        uint4 v[17];
#pragma unroll
        for (int m = 0; m < 17; ++m) {
            const int o = 16 * (32 * m + lane);
            v[m] = make_uint4(0u, 0u, 0u, 0u);
            if (o + 16 <= nbytes) {
                v[m] = __ldg(reinterpret_cast<const uint4 *>(a.body + off0 + o));
            } else if (o < nbytes) {
                uint32_t t[4] = {0u, 0u, 0u, 0u};
                for (int x = o; x < nbytes; x += 2)
                    t[(x - o) >> 2] |= (uint32_t)__ldg(reinterpret_cast<const uint16_t *>(a.body + off0 + x))
                                       << (8 * ((x - o) & 3));
                v[m] = make_uint4(t[0], t[1], t[2], t[3]);
            }
        }
#pragma unroll
        for (int m = 0; m < 17; ++m) *reinterpret_cast<uint4 *>(S.buf + 16 * (32 * m + lane)) = v[m];
    }
    __syncwarp();
    uint32_t w[68];
#pragma unroll
    for (int k = 0; k < 17; ++k) {
        const uint4 v = *reinterpret_cast<const uint4 *>(S.buf + 272 * lane + 16 * k);
        w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
    }
    uint32_t sc[8];
    uint4 c[16];
    disassemble(w, sc, c);
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 16; ++k) *reinterpret_cast<uint4 *>(S.buf + 16 * phys_chunk(16 * lane + k)) = c[k];
    *reinterpret_cast<uint4 *>(S.sc + 8 * lane) = make_uint4(sc[0] | (sc[1] << 16), sc[2] | (sc[3] << 16),
                                                           sc[4] | (sc[5] << 16), sc[6] | (sc[7] << 16));
    __syncwarp();
    // code chunk 32 m + lane and scale 32 m + lane of the warp to the cache
    BlockPos p = block_pos(a, beta0 + (lane >> 1));
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        if (beta0 + 16 * m + (lane >> 1) < a.n_blocks)
            reinterpret_cast<uint4 *>((p.kv ? a.vq : a.kq) + code_off(a, p))[lane & 1] =
                *reinterpret_cast<const uint4 *>(S.buf + 16 * phys_chunk(32 * m + lane));
        if (m < 15) advance(a, p, 16);
    }
    BlockPos q = block_pos(a, beta0 + lane);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        if (beta0 + 32 * m + lane < a.n_blocks) (q.kv ? a.vs : a.ks)[scale_off(a, q)] = S.sc[32 * m + lane];
        if (m < 7) advance(a, q, 32);
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

// a warp moves 32 * F16_CHUNKS consecutive chunks, lane-interleaved: each access is 512 contiguous bytes
template <bool PACK>
__global__ void __launch_bounds__(THREADS) copy_f16_kernel(const StateArgs a) {
    if (PACK) write_header_words(a);
    const int lane = threadIdx.x & 31;
    const int64_t first = ((int64_t)blockIdx.x * THREADS + (threadIdx.x - lane)) * F16_CHUNKS + lane;
    uint4 v[F16_CHUNKS];
#pragma unroll
    for (int i = 0; i < F16_CHUNKS; ++i) {
        const int64_t gamma = first + 32 * i;
        if (gamma < a.n_chunks)
            v[i] = PACK ? __ldg(reinterpret_cast<const uint4 *>(f16_cache_ptr(a, gamma)))
                        : __ldg(reinterpret_cast<const uint4 *>(a.body) + gamma);
    }
#pragma unroll
    for (int i = 0; i < F16_CHUNKS; ++i) {
        const int64_t gamma = first + 32 * i;
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

// ---- a head range: the cache holds kv heads [head0, head0 + H) of a stream of H_total heads ----
// A cache split by head (its kv heads spread over several caches, as over several devices) packs each
// part into its place of one stream, and restores each part from it.
struct RangeArgs {
    uint8_t *body;
    uint8_t *kq, *vq;
    uint16_t *ks, *vs;
    Geom g;
    int64_t n_units;    // units this cache holds: n_layer * n_tokens * 2 * H * units per head
    int64_t rec;        // stream bytes of one record of all H_total heads
    int n_tokens, H, head0, upr;   // upr: units per head (head_dim / 32 blocks, or head_dim / 8 chunks)
    int bph;            // stream bytes per head
};

// f16 head range: one thread moves one 16-byte chunk of 8 values (a head's 2 * head_dim stream bytes
// start 16-byte aligned).
template <bool PACK>
__global__ void __launch_bounds__(256) range_f16_kernel(const RangeArgs a) {
    const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= a.n_units) return;
    const int64_t row = u / a.upr;                   // (layer, position, K/V, local head) in stream order
    const int b = (int)(u - row * a.upr);
    const int64_t rk = row / a.H;                    // (layer, position, K/V)
    const int hl = (int)(row - rk * a.H);
    const int kv = (int)(rk & 1);
    const int64_t lt = rk >> 1;
    const int layer = (int)(lt / a.n_tokens);
    const int t = (int)(lt - (int64_t)layer * a.n_tokens);
    const int64_t head_row = layer * a.g.c_layer + (int64_t)t * a.g.c_tok + hl * a.g.c_head;
    uint4 *vals = reinterpret_cast<uint4 *>((kv ? a.vq : a.kq) + 2 * head_row) + b;
    uint4 *chunk = reinterpret_cast<uint4 *>(a.body + rk * a.rec + (int64_t)(a.head0 + hl) * a.bph) + b;
    if (PACK) *chunk = *vals;
    else *vals = *chunk;
}

// q8_0 head range, pack: one warp per record run.  The part's H heads of one (layer, position, K/V)
// record are H * head_dim/32 consecutive 34-byte blocks of the stream, a run that starts on a 4-byte
// boundary (32-byte header; records and heads of 34 * head_dim/32 bytes, a multiple of 4).  The warp
// assembles the run in shared memory, one block per lane, then stores it in 4-byte words with
// consecutive lanes on consecutive words (halfword stores straight to the stream measured 4x slower).
constexpr int RUN_WARPS = 8;
__global__ void __launch_bounds__(RUN_WARPS * 32) range_q8_pack_kernel(const RangeArgs a, int run_bytes) {
    extern __shared__ __align__(16) uint8_t run_smem[];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t rk = (int64_t)blockIdx.x * RUN_WARPS + wid;         // (layer, position, K/V)
    const int64_t n_runs = a.n_units / ((int64_t)a.H * a.upr);
    if (rk >= n_runs) return;   // the whole warp
    uint16_t *run = reinterpret_cast<uint16_t *>(run_smem + wid * run_bytes);
    const int kv = (int)(rk & 1);
    const int64_t lt = rk >> 1;
    const int layer = (int)(lt / a.n_tokens);
    const int t = (int)(lt - (int64_t)layer * a.n_tokens);
    uint32_t *s = reinterpret_cast<uint32_t *>(a.body + rk * a.rec + (int64_t)a.head0 * a.bph);
    const int n_blocks = a.H * a.upr, n_words = run_bytes / 4;
    auto block_ptrs = [&](int j, uint4 *&codes, uint16_t *&scale) {
        const int hl = j / a.upr, b = j - hl * a.upr;
        codes = reinterpret_cast<uint4 *>((kv ? a.vq : a.kq) + layer * a.g.c_layer + (int64_t)t * a.g.c_tok +
                                          hl * a.g.c_head + 32 * b);
        scale = (kv ? a.vs : a.ks) + layer * a.g.s_layer + (int64_t)t * a.g.s_tok + hl * a.g.s_head + b;
    };
    for (int j = lane; j < n_blocks; j += 32) {
        uint4 *codes;
        uint16_t *scale;
        block_ptrs(j, codes, scale);
        const uint4 c0 = codes[0], c1 = codes[1];
        const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        uint16_t *blk = run + 17 * j;
        blk[0] = *scale;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            blk[1 + 2 * i] = (uint16_t)(w[i] & 0xFFFFu);
            blk[2 + 2 * i] = (uint16_t)(w[i] >> 16);
        }
    }
    __syncwarp();
    const uint32_t *src = reinterpret_cast<const uint32_t *>(run);
    for (int i = lane; i < n_words; i += 32) s[i] = src[i];
}

// q8_0 head range, unpack: one thread per block, 17 halfword loads from the stream (a block starts on
// an even offset), then the 32 codes and the scale to the cache (measured faster than staging runs).
__global__ void __launch_bounds__(256) range_q8_unpack_kernel(const RangeArgs a) {
    const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= a.n_units) return;
    const int64_t row = u / a.upr;                   // (layer, position, K/V, local head) in stream order
    const int b = (int)(u - row * a.upr);
    const int64_t rk = row / a.H;                    // (layer, position, K/V)
    const int hl = (int)(row - rk * a.H);
    const int kv = (int)(rk & 1);
    const int64_t lt = rk >> 1;
    const int layer = (int)(lt / a.n_tokens);
    const int t = (int)(lt - (int64_t)layer * a.n_tokens);
    const uint16_t *blk = reinterpret_cast<const uint16_t *>(a.body + rk * a.rec + (int64_t)(a.head0 + hl) * a.bph +
                                                             34 * b);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = (uint32_t)blk[1 + 2 * i] | ((uint32_t)blk[2 + 2 * i] << 16);
    uint4 *codes = reinterpret_cast<uint4 *>((kv ? a.vq : a.kq) + layer * a.g.c_layer + (int64_t)t * a.g.c_tok +
                                             hl * a.g.c_head + 32 * b);
    (kv ? a.vs : a.ks)[layer * a.g.s_layer + (int64_t)t * a.g.s_tok + hl * a.g.s_head + b] = blk[0];
    codes[0] = make_uint4(w[0], w[1], w[2], w[3]);
    codes[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

RangeArgs make_range_args(const kvc_cache &c, int head0, int H_total, int n_tokens, uint8_t *body) {
    RangeArgs a = {};
    const bool q8 = c.d.type == KVC_Q8_0;
    a.body = body;
    a.kq = static_cast<uint8_t *>(c.k_q);
    a.vq = static_cast<uint8_t *>(c.v_q);
    a.ks = static_cast<uint16_t *>(c.k_s);
    a.vs = static_cast<uint16_t *>(c.v_s);
    a.g = geom_of(c.d);
    a.n_tokens = n_tokens;
    a.H = c.d.n_head_kv;
    a.head0 = head0;
    a.upr = q8 ? c.d.head_dim / 32 : c.d.head_dim / 8;
    a.bph = q8 ? (c.d.head_dim / 32) * 34 : c.d.head_dim * 2;
    a.rec = (int64_t)H_total * a.bph;
    a.n_units = (int64_t)c.d.n_layer * n_tokens * 2 * a.H * a.upr;
    return a;
}

int grid_q8(int64_t n_blocks) {
    const int64_t per_cta = (int64_t)QW * WARP_BLOCKS;
    return (int)((n_blocks + per_cta - 1) / per_cta);
}

int grid_for(int64_t work, int per_thread) {
    return (int)((work + (int64_t)THREADS * per_thread - 1) / ((int64_t)THREADS * per_thread));
}

}  // namespace

int launch_state_pack(const kvc_cache &c, int n_tokens, uint8_t *dst, cudaStream_t s) {
    const bool q8 = c.d.type == KVC_Q8_0;
    StateArgs a = make_args(c, n_tokens, dst + 32);
    const uint32_t hdr[8] = {0x3143564Bu, 1u, (uint32_t)c.d.n_layer, (uint32_t)c.d.n_head_kv, (uint32_t)c.d.head_dim,
                             q8 ? 1u : 0u, (uint32_t)n_tokens, 0u};
    for (int i = 0; i < 8; ++i) a.hdr[i] = hdr[i];
    if (n_tokens == 0)   // the header alone
        write_header<<<1, 1, 0, s>>>(dst, c.d.n_layer, c.d.n_head_kv, c.d.head_dim, q8 ? 1u : 0u, 0u);
    else if (q8)         // the kernels write the header too: one launch
        pack_q8_kernel<<<grid_q8(a.n_blocks), QW * 32, 0, s>>>(a);
    else
        copy_f16_kernel<true><<<grid_for(a.n_chunks, F16_CHUNKS), THREADS, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
}

int launch_state_pack_heads(const kvc_cache &c, int head0, int H_total, int n_tokens, uint8_t *dst, cudaStream_t s) {
    const bool q8 = c.d.type == KVC_Q8_0;
    write_header<<<1, 1, 0, s>>>(dst, c.d.n_layer, H_total, c.d.head_dim, q8 ? 1u : 0u, n_tokens);
    const RangeArgs a = make_range_args(c, head0, H_total, n_tokens, dst + 32);
    if (a.n_units > 0) {
        if (q8) {
            const int run_bytes = a.H * a.bph;
            const int64_t n_runs = (int64_t)c.d.n_layer * n_tokens * 2;
            const size_t smem = (size_t)RUN_WARPS * run_bytes;
            if (smem > 48 * 1024 && allow_dynamic_smem((const void *)range_q8_pack_kernel, (int)smem) != KVC_OK)
                return KVC_ECUDA;
            range_q8_pack_kernel<<<(unsigned)((n_runs + RUN_WARPS - 1) / RUN_WARPS), RUN_WARPS * 32, smem, s>>>(
                a, run_bytes);
        } else {
            range_f16_kernel<true><<<(int)((a.n_units + 255) / 256), 256, 0, s>>>(a);
        }
    }
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
}

int launch_state_unpack_heads(const kvc_cache &c, int head0, int H_total, int n_tokens, const uint8_t *src,
                              cudaStream_t s) {
    const bool q8 = c.d.type == KVC_Q8_0;
    const RangeArgs a = make_range_args(c, head0, H_total, n_tokens, const_cast<uint8_t *>(src) + 32);
    if (a.n_units > 0) {
        if (q8) {
            range_q8_unpack_kernel<<<(int)((a.n_units + 255) / 256), 256, 0, s>>>(a);
        } else {
            range_f16_kernel<false><<<(int)((a.n_units + 255) / 256), 256, 0, s>>>(a);
        }
    }
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
}

int launch_state_unpack(const kvc_cache &c, int n_tokens, const uint8_t *src, cudaStream_t s) {
    const bool q8 = c.d.type == KVC_Q8_0;
    const StateArgs a = make_args(c, n_tokens, const_cast<uint8_t *>(src) + 32);
    if (n_tokens > 0) {
        if (q8) unpack_q8_kernel<<<grid_q8(a.n_blocks), QW * 32, 0, s>>>(a);
        else copy_f16_kernel<false><<<grid_for(a.n_chunks, F16_CHUNKS), THREADS, 0, s>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
}

}  // namespace kvc
