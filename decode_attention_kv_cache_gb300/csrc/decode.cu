// Single-token decode attention over the KV cache: split-K over the key range,
// then a combine pass.
//
// What it computes: for the query token at position pos and each query head h,
// softmax over keys j <= pos of q.khat_j / sqrt(D), applied to vhat_j, kv head
// h / G - the generation step the pages time as "generation t/s" (llama.cpp
// PR #58 "completion : allow the prompt to be processed under its own split
// mode", section "Why"; llama.cpp PR #59 "llama : switch the split mode of a
// live context", section "Why").
//
// Split pass, head_dim 128 (decode_tc_kernel, described where it is defined):
// one wave of CTAs, one per SM, over (split, kv head); 128-key tiles by TMA;
// tcgen05 MMAs over query-head rows replicated so that one thread owns one
// row's online softmax; two MMA issuers; q8_0 codes dequantised in place.  For
// decode_step the CTA whose split holds pos first quantises and stores the
// token (the append kernel's quantiser), then copies that tile.
//
// Split pass, head_dim 64 (decode_split_kernel): one wave of CTAs, grid (split,
// kv head), two CTAs per SM.  A CTA streams the key range [split*len,
// (split+1)*len) of one kv head: warp 0 issues TMA copies of 64-key K and V
// blocks into a ring of shared-memory stages (128-byte swizzle; 64-byte for the
// 64-byte q8_0 rows), so many stages are in flight at once; four consumer warps each take one 16-key group of a
// stage for all G query heads of the group.  A consumer warp computes the
// group's scores with mma.sync m16n8k16 (rows = query heads of the group,
// columns = keys), keeps an online softmax per head, and accumulates P*V with
// a second mma.sync (rows = heads, columns = head_dim), reading its fragments
// from the stage:
//   - q8_0 codes are converted to exact fp16 integers with two byte permutes
//     and one fp16 subtraction; the K scale is applied per 32-value block to
//     the fp32 partial scores, the V scale is folded into P per block, so the
//     only rounding besides fp32 accumulation is fp16(p*d);
//   - f16 values feed the MMAs as stored.
// Head-dim slots are permuted inside each MMA (the dot product does not care)
// so that every thread reads 8 or 16 (K) and 4 or 8 (V) contiguous bytes per
// row.  The four warps are merged in shared memory in a fixed order and the
// CTA writes (m, l, O) for its range to the scratch buffer.  For decode_step, warp 0 of the CTA whose
// split holds pos stores the token first, before any stage is copied.
//
// Combine pass: launched with programmatic dependent launch, so its CTAs are
// resident while the split pass runs and wait for it on the device
// (griddepcontrol.wait); one CTA per query head merges the splits in split
// order (deterministic) and divides by the softmax sum.
//
// Split boundaries are absolute key positions, so the result does not depend
// on the cache layout.  Every mbarrier wait is bounded (2 s); a wait that gives
// up sets the device status word and the CTA skips its remaining work.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <map>
#include <mutex>

#include "kvc_internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace kvc {
namespace {

// set by a split pass that gave up a bounded wait (read and cleared with the other kernels' status)
__device__ int g_decode_status;

// Diagnostic build (-DKVC_TRACE, see build.py): the tensor-core split pass records clock64 stamps of its
// pipeline events in CTA (0, 0) - event e of tile k in g_trace[e][k] (e = 1..13), overall events in
// g_trace[0][.] - for kvc_trace_read.  The stamps change no work; a normal build compiles them away.
#ifdef KVC_TRACE
__device__ unsigned long long g_trace[16][64];
#define KVC_TR(ev, k)                                                                   \
    do {                                                                              \
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (k) < 64)          \
            g_trace[ev][k] = clock64();                                               \
    } while (0)
#else
#define KVC_TR(ev, k) do { } while (0)
#endif

using namespace ptx;

constexpr int MAX_SPLIT = 256;
constexpr int CWARPS = 4;                          // consumer warps
constexpr int GROUP_KEYS = 16;                     // keys per consumer warp and stage
constexpr int STAGE_KEYS = CWARPS * GROUP_KEYS;    // keys per stage
constexpr int CTAS_PER_SM = 2;

template <int D, bool Q8>
struct DCfg {
    static constexpr int ROW = Q8 ? D : 2 * D;             // bytes of one key row
    static constexpr int BLK_ROW = Q8 ? D : 128;            // bytes per row of one swizzled column block
    static constexpr int NBLK = ROW / BLK_ROW;              // column blocks of a K or V tile
    static constexpr int HALF = STAGE_KEYS * ROW;           // K (or V) bytes of a stage
    static constexpr int STAGE = 2 * HALF;
    static constexpr int NST = (96 * 1024) / STAGE;          // ring stages (two CTAs per SM)
    static constexpr int OFF_BAR = NST * STAGE;
    static constexpr int USED = OFF_BAR + 2 * NST * 8 + 16;
    static constexpr int ALLOC = USED + 1024;                // room to align the ring to 1024 bytes
    // the warps' partial results, merged at the end, reuse the ring
    static constexpr int MERGE = CWARPS * 16 * (D + 2) * 4;
    static_assert(MERGE <= OFF_BAR, "merge buffers must fit in the ring");
    static_assert(NST >= 2, "ring too small");
};

// Byte offset, within one K or V tile of a stage, of byte c of key row r (TMA 128- or 64-byte swizzle).
template <int D, bool Q8>
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
    using L = DCfg<D, Q8>;
    const int blk = c / L::BLK_ROW, cb = c % L::BLK_ROW;
    if constexpr (L::BLK_ROW == 128)
        return (uint32_t)(blk * (STAGE_KEYS * 128) + r * 128 + ((((cb >> 4) ^ (r & 7))) << 4) + (cb & 15));
    else
        return (uint32_t)(blk * (STAGE_KEYS * 64) + r * 64 + ((((cb >> 4) ^ ((r >> 1) & 3))) << 4) + (cb & 15));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}


// Two int8 codes placed in bytes 0 and 2 of `t` (bytes 1 and 3 ignored) -> fp16x2 of the exact codes.
__device__ __forceinline__ uint32_t codes_to_half2(uint32_t t) {
    const uint32_t m = (t & 0x00FF00FFu) ^ 0x64806480u;  // fp16 1024 + (q + 128)
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&m), bias);
    return *reinterpret_cast<uint32_t *>(&r);
}

template <int DT>
__device__ __forceinline__ float load_q(const void *q, int64_t i) {
    if constexpr (DT == KVC_IN_F32) return __ldcg(static_cast<const float *>(q) + i);
    else {
        const uint16_t u = __ldcg(static_cast<const unsigned short *>(q) + i);
        if constexpr (DT == KVC_IN_BF16) return __uint_as_float((uint32_t)u << 16);
        else return __half2float(__ushort_as_half(u));
    }
}

struct DecodeArgs {
    const void *q;
    const uint16_t *ks;
    const uint16_t *vs;
    float *part;       // scratch
    Geom g;
    int layer, n_keys, group, split_len, n_split, n_head_kv;
    float scale_log2;
    uint64_t stall_ns;   // test hook (tensor-core pass): > 0 makes the MMA thread's first P wait one that runs out
    // Fused decode step (tensor-core pass only; all null for decode_attn).  k_new / v_new: the token's
    // K and V rows, [n_head_kv][128] in the query's dtype, stored at position n_keys - 1 of the cache
    // (codes kq / vq, scales ks_w / vs_w) by the CTA whose split holds that position.
    const void *k_new, *v_new;
    void *kq, *vq;
    uint16_t *ks_w, *vs_w;
};

// Several sequences decoded by one launch: each has its own cache (and so its own tensor maps),
// position, query, scratch and output.  Grid z (or y for the combine pass) is the sequence.
constexpr int MAX_BATCH = 8;
template <int NS>
struct TcBatch {
    CUtensorMap tk[NS];
    CUtensorMap tv[NS];
    DecodeArgs a[NS];
};
template <int NS>
struct CombineBatch {
    const float *part[NS];
    float *out[NS];
    int n_split[NS];
};

// One consumer warp's fragments of a 16-key group.
template <int D, bool Q8>
struct Tiles {
    static constexpr int NB = D / 32;
    // K: [n-tile t][block b] 8 code bytes (q8_0) or 8 halves (f16)
    uint2 k8[Q8 ? 2 : 1][Q8 ? NB : 1];
    uint4 k16[Q8 ? 1 : 2][Q8 ? 1 : NB];
    // V: [key r][block b] 4 code bytes (q8_0) or 4 halves (f16)
    uint32_t v8[Q8 ? 4 : 1][Q8 ? NB : 1];
    uint2 v16[Q8 ? 1 : 4][Q8 ? 1 : NB];
};

// scales of keys j0+4c+r: NB fp16 values packed two per word
template <int D>
struct Scales {
    static constexpr int NB = D / 32;
    uint32_t sk[4][NB / 2], sv[4][NB / 2];
    __device__ __forceinline__ float kscale(int r, int b) const {
        return __half2float(__ushort_as_half((unsigned short)(sk[r][b >> 1] >> (16 * (b & 1)))));
    }
    __device__ __forceinline__ float vscale(int r, int b) const {
        return __half2float(__ushort_as_half((unsigned short)(sv[r][b >> 1] >> (16 * (b & 1)))));
    }
};

template <int D>
__device__ __forceinline__ void load_scales(const DecodeArgs &a, int hkv, int j0, int cq, Scales<D> &S) {
    constexpr int NB = D / 32;
    const int last = a.n_keys - 1;
    const int64_t base_s = a.layer * a.g.s_layer + hkv * a.g.s_head;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        // a key's NB scales are contiguous and 2*NB-byte aligned; keys past the end reuse the last
        // key's (their codes are zero-filled and their scores masked)
        const int key = min(j0 + 4 * cq + r, last);
        const int64_t srow = base_s + (int64_t)key * a.g.s_tok;
        if constexpr (NB == 4) {
            const uint2 wk = __ldcg(reinterpret_cast<const uint2 *>(a.ks + srow));
            const uint2 wv = __ldcg(reinterpret_cast<const uint2 *>(a.vs + srow));
            S.sk[r][0] = wk.x; S.sk[r][1] = wk.y;
            S.sv[r][0] = wv.x; S.sv[r][1] = wv.y;
        } else {
            S.sk[r][0] = __ldcg(reinterpret_cast<const unsigned int *>(a.ks + srow));
            S.sv[r][0] = __ldcg(reinterpret_cast<const unsigned int *>(a.vs + srow));
        }
    }
}

// The group's K fragments from stage `sb`: rows 16*cw .. 16*cw + 15 of its K tile.
template <int D, bool Q8>
__device__ __forceinline__ void load_group_k(const uint8_t *sb, int cw, int gq, int cq, Tiles<D, Q8> &T) {
    constexpr int NB = D / 32;
    const uint8_t *kb = sb;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int row = GROUP_KEYS * cw + 4 * (gq >> 1) + 2 * t + (gq & 1);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if constexpr (Q8)
                T.k8[t][b] = *reinterpret_cast<const uint2 *>(kb + tile_off<D, Q8>(row, 32 * b + 8 * cq));
            else
                T.k16[t][b] = *reinterpret_cast<const uint4 *>(kb + tile_off<D, Q8>(row, 2 * (32 * b + 8 * cq)));
        }
    }
}

// The group's V fragments from stage `sb`: rows 16*cw .. 16*cw + 15 of its V tile.
template <int D, bool Q8>
__device__ __forceinline__ void load_group_v(const uint8_t *sb, int cw, int gq, int cq, Tiles<D, Q8> &T) {
    constexpr int NB = D / 32;
    const uint8_t *vb = sb + DCfg<D, Q8>::HALF;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int row = GROUP_KEYS * cw + 4 * cq + r;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if constexpr (Q8)
                T.v8[r][b] = *reinterpret_cast<const uint32_t *>(vb + tile_off<D, Q8>(row, 32 * b + 4 * gq));
            else
                T.v16[r][b] = *reinterpret_cast<const uint2 *>(vb + tile_off<D, Q8>(row, 2 * (32 * b + 4 * gq)));
        }
    }
}

// 8 query values (chunk i of the loaded 16-byte words) as fp32
template <int DT, int N>
__device__ __forceinline__ void to_f32x8(const uint4 (&raw)[N], int i, float (&x)[8]) {
    if constexpr (DT == KVC_IN_F32) {
        const uint4 a = raw[2 * i], b = raw[2 * i + 1];
        x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y); x[2] = __uint_as_float(a.z);
        x[3] = __uint_as_float(a.w); x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
        x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
    } else {
        const uint4 u = raw[i];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if constexpr (DT == KVC_IN_BF16) {
                x[2 * e] = __uint_as_float(w[e] << 16);
                x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
            } else {
                x[2 * e] = __half2float(__ushort_as_half((unsigned short)(w[e] & 0xFFFFu)));
                x[2 * e + 1] = __half2float(__ushort_as_half((unsigned short)(w[e] >> 16)));
            }
        }
    }
}

// Fused decode step: one warp stores the token's K and V rows of kv head hkv at position n_keys - 1,
// exactly as the append kernel does (q8_0 blocks by the shared quantiser, f16 values rounded to
// nearest even).  q8_0: one lane per 32-value block (K's blocks, then V's); f16: one lane per 8 values
// (K's, then V's).  The rows are read through L2: a kernel just before
// this one may have written them.
template <bool Q8, int DT, int D = 128>
__device__ __forceinline__ void store_new_token(const DecodeArgs &a, int hkv, int lane) {
    constexpr int ESZ = DT == KVC_IN_F32 ? 4 : 2;
    constexpr int NB = D / 32;                     // q8_0 blocks per row
    const int64_t pos = a.n_keys - 1;
    const Geom &g = a.g;
    if constexpr (Q8) {
        if (lane < 2 * NB) {
            const int is_v = lane / NB, b = lane % NB;
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(is_v ? a.v_new : a.k_new) +
                                                               ((int64_t)hkv * D + b * 32) * ESZ);
            constexpr int NW = 32 * ESZ / 16;   // 16-byte words of one block's input
            uint4 raw[NW];
#pragma unroll
            for (int i = 0; i < NW; ++i) raw[i] = __ldcg(src + i);
            float x[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float x8[8];
                to_f32x8<DT>(raw, c, x8);
#pragma unroll
                for (int e = 0; e < 8; ++e) x[8 * c + e] = x8[e];
            }
            uint32_t packed[8];
            const uint16_t scale = q8_0_quantize32(x, packed);
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<int8_t *>(is_v ? a.vq : a.kq) + a.layer * g.c_layer +
                                                   pos * g.c_tok + hkv * g.c_head + b * 32);
            dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
            (is_v ? a.vs_w : a.ks_w)[a.layer * g.s_layer + pos * g.s_tok + hkv * g.s_head + b] = scale;
        }
    } else {
        constexpr int UPR = D / 8;                 // 8-value units per row
        if (lane >= 2 * UPR) return;
        const int is_v = lane / UPR, c = lane % UPR;
        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(is_v ? a.v_new : a.k_new) +
                                                           ((int64_t)hkv * D + c * 8) * ESZ);
        uint4 raw[ESZ / 2];
#pragma unroll
        for (int i = 0; i < ESZ / 2; ++i) raw[i] = __ldcg(src + i);
        float x[8];
        to_f32x8<DT>(raw, 0, x);
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(is_v ? a.vq : a.kq) + a.layer * g.c_layer + pos * g.c_tok +
                                   hkv * g.c_head + c * 8) =
            make_uint4(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]), pack_half2(x[4], x[5]), pack_half2(x[6], x[7]));
    }
}

template <int D, bool Q8, int DT>
__global__ void __maxnreg__(200)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const DecodeArgs a) {
    using L = DCfg<D, Q8>;
    constexpr int NB = D / 32;
    constexpr int KS = D / 16;       // k-steps of the score MMA
    constexpr int NT = D / 8;        // n-tiles of the output MMA
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint64_t *empty = full + L::NST;
    volatile int *s_abort = reinterpret_cast<volatile int *>(empty + L::NST);
    const int split = blockIdx.x, hkv = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.group;
    const int j_begin = split * a.split_len;
    const int j_end = min(a.n_keys, j_begin + a.split_len);
    const int n_stages = (j_end - j_begin + STAGE_KEYS - 1) / STAGE_KEYS;

    if (threadIdx.x == 0) {
        *s_abort = 0;
        for (int i = 0; i < L::NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], CWARPS);
        }
        fence_mbar_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    __syncthreads();
    // inputs written by the kernels before this one are read only past this point; the combine
    // pass may be scheduled from here on (it waits for this grid to finish)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    if (a.k_new != nullptr) {
        // fused decode step: the CTA whose split holds the new position stores the token first; the
        // barrier orders those stores before the stage copies (with the async-proxy fence) and the
        // consumers' scale loads
        if (warp == 0 && split == a.n_split - 1) {
            store_new_token<Q8, DT, D>(a, hkv, lane);
            fence_proxy_async_global();
        }
        __syncthreads();
    }

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            int i = 0;
            for (; i < n_stages; ++i) {
                const int st = i % L::NST;
                if (i >= L::NST && !mbar_wait(&empty[st], ((i / L::NST) - 1) & 1, s_abort)) break;
                mbar_arrive_expect_tx(&full[st], L::STAGE);
                const int j = j_begin + i * STAGE_KEYS;
                uint8_t *dst = sm + st * L::STAGE;
                constexpr int ELEMS = Q8 ? L::BLK_ROW : L::BLK_ROW / 2;  // elements per block row
#pragma unroll
                for (int blk = 0; blk < L::NBLK; ++blk) {
                    tma_load_3d(dst + blk * (STAGE_KEYS * L::BLK_ROW), &tm_k, &full[st], blk * ELEMS, j, hkv);
                    tma_load_3d(dst + L::HALF + blk * (STAGE_KEYS * L::BLK_ROW), &tm_v, &full[st], blk * ELEMS, j,
                                hkv);
                }
            }
            if (*s_abort) {
                // after a wait gave up: let the copies still in flight land before the CTA exits
                volatile int never = 0;
                for (int st = 0; st < L::NST && st < i; ++st) {
                    const int last = st + ((i - 1 - st) / L::NST) * L::NST;
                    mbar_wait(&full[st], (last / L::NST) & 1, &never, 200000000ull);
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ consumers
        const int cw = warp - 1;
        const int gq = lane >> 2, cq = lane & 3;
        // Q as the A operand of the score MMA: rows = heads of the group; in k-step
        // s = 2b + e this thread's four head-dim slots are d0..d0+3, d0 = 32b + 8c + 4e.
        uint32_t qa[KS][4];
#pragma unroll
        for (int s = 0; s < KS; ++s) {
            const int d0 = 32 * (s >> 1) + 8 * cq + 4 * (s & 1);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int row = gq + 8 * half;
                float x[4] = {0.f, 0.f, 0.f, 0.f};
                if (row < G) {
                    const int64_t base = ((int64_t)hkv * G + row) * D + d0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) x[i] = load_q<DT>(a.q, base + i);
                }
                qa[s][half] = pack_half2(x[0], x[1]);       // a0a1 / a2a3: slots 2c, 2c+1
                qa[s][2 + half] = pack_half2(x[2], x[3]);   // a4a5 / a6a7: slots 2c+8, 2c+9
            }
        }
        Scales<D> sc_cur, sc_nxt;
        if (Q8 && n_stages > 0) load_scales<D>(a, hkv, j_begin + cw * GROUP_KEYS, cq, sc_cur);
#pragma unroll 1
        for (int i = 0; i < n_stages; ++i) {
            const int st = i % L::NST;
            const int j0 = j_begin + i * STAGE_KEYS + cw * GROUP_KEYS;
            if (Q8 && i + 1 < n_stages) load_scales<D>(a, hkv, j0 + STAGE_KEYS, cq, sc_nxt);
            if (!mbar_wait(&full[st], (i / L::NST) & 1, s_abort)) break;
            Tiles<D, Q8> cur;
            const uint8_t *sb = sm + st * L::STAGE;
            // K fragments now, V fragments after the softmax (fewer live registers); the stage is
            // released once both are read
            load_group_k<D, Q8>(sb, cw, gq, cq, cur);
            if (j0 < j_end) {
                // ---- scores: sc[t][i] for keys j0 + 4c + 2t + (i & 1), heads gq (i < 2) and gq + 8
                float sc[2][4];
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
                    if constexpr (Q8) {
#pragma unroll
                        for (int b = 0; b < NB; ++b) {
                            float acc[4] = {0.f, 0.f, 0.f, 0.f};
                            const uint32_t w0 = cur.k8[t][b].x, w1 = cur.k8[t][b].y;
                            mma16816(acc, qa[2 * b], codes_to_half2(__byte_perm(w0, 0, 0x0100)),
                                     codes_to_half2(__byte_perm(w0, 0, 0x0302)));
                            mma16816(acc, qa[2 * b + 1], codes_to_half2(__byte_perm(w1, 0, 0x0100)),
                                     codes_to_half2(__byte_perm(w1, 0, 0x0302)));
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                sc[t][e] += sc_cur.kscale(2 * t + (e & 1), b) * acc[e];
                        }
                    } else {
#pragma unroll
                        for (int b = 0; b < NB; ++b) {
                            mma16816(sc[t], qa[2 * b], cur.k16[t][b].x, cur.k16[t][b].y);
                            mma16816(sc[t], qa[2 * b + 1], cur.k16[t][b].z, cur.k16[t][b].w);
                        }
                    }
                }
                // ---- online softmax (log2 domain), rows gq and gq + 8
                float p[2][4];
                float alpha[2];
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    float x[4];
#pragma unroll
                    for (int t = 0; t < 2; ++t)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int key = j0 + 4 * cq + 2 * t + e;
                            x[2 * t + e] = key < j_end ? sc[t][2 * hr + e] * a.scale_log2 : -INFINITY;
                        }
                    float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    const float m_new = fmaxf(m_run[hr], mx);  // finite: key j0 < j_end is visible
                    alpha[hr] = ex2(m_run[hr] - m_new);
                    float rs = 0.f;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        p[hr][e] = ex2(x[e] - m_new);
                        rs += p[hr][e];
                    }
                    l_run[hr] = l_run[hr] * alpha[hr] + rs;
                    m_run[hr] = m_new;
                }
                if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        o[n][0] *= alpha[0]; o[n][1] *= alpha[0];
                        o[n][2] *= alpha[1]; o[n][3] *= alpha[1];
                    }
                }
                load_group_v<D, Q8>(sb, cw, gq, cq, cur);
                // order the stage reads before the TMA (async proxy) that refills it
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
                // ---- O += P V.  A = P (rows heads, k-slots 2c, 2c+1 <- keys 4c, 4c+1; 2c+8, 2c+9 <- 4c+2, 4c+3)
                //      B = V (k-slots as above, column n of n-tile 4b + s <- head-dim 32b + 4n + s)
                if constexpr (Q8) {
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        float dv[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) dv[r] = sc_cur.vscale(r, b);
                        uint32_t pa[4];
                        pa[0] = pack_half2(p[0][0] * dv[0], p[0][1] * dv[1]);
                        pa[1] = pack_half2(p[1][0] * dv[0], p[1][1] * dv[1]);
                        pa[2] = pack_half2(p[0][2] * dv[2], p[0][3] * dv[3]);
                        pa[3] = pack_half2(p[1][2] * dv[2], p[1][3] * dv[3]);
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const uint32_t sel = (uint32_t)s | ((uint32_t)(4 + s) << 8);
                            const uint32_t b0 = codes_to_half2(__byte_perm(cur.v8[0][b], cur.v8[1][b], sel));
                            const uint32_t b1 = codes_to_half2(__byte_perm(cur.v8[2][b], cur.v8[3][b], sel));
                            mma16816(o[4 * b + s], pa, b0, b1);
                        }
                    }
                } else {
                    uint32_t pa[4];
                    pa[0] = pack_half2(p[0][0], p[0][1]);
                    pa[1] = pack_half2(p[1][0], p[1][1]);
                    pa[2] = pack_half2(p[0][2], p[0][3]);
                    pa[3] = pack_half2(p[1][2], p[1][3]);
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const uint32_t sel = (s & 1) ? 0x7632u : 0x5410u;
                            const uint32_t w0 = (s < 2) ? cur.v16[0][b].x : cur.v16[0][b].y;
                            const uint32_t w1 = (s < 2) ? cur.v16[1][b].x : cur.v16[1][b].y;
                            const uint32_t w2 = (s < 2) ? cur.v16[2][b].x : cur.v16[2][b].y;
                            const uint32_t w3 = (s < 2) ? cur.v16[3][b].x : cur.v16[3][b].y;
                            mma16816(o[4 * b + s], pa, __byte_perm(w0, w1, sel), __byte_perm(w2, w3, sel));
                        }
                    }
                }
            } else {
                // a group past the end of the range: release the stage without computing
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }
            if (Q8) sc_cur = sc_nxt;
        }
    }

    // ---- merge the consumer warps in shared memory (fixed order) and write the CTA's partial;
    // the buffers reuse the ring, whose copies have all been consumed
    __syncthreads();
    float *s_m = reinterpret_cast<float *>(sm);
    float *s_l = s_m + CWARPS * 16;
    float *s_o = s_l + CWARPS * 16;   // [warp][row][D]
    if (warp > 0) {
        const int cw = warp - 1, gq = lane >> 2, cq = lane & 3;
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            float l = l_run[hr];
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            const int row = gq + 8 * hr;
            if (cq == 0) {
                s_m[cw * 16 + row] = m_run[hr];
                s_l[cw * 16 + row] = l;
            }
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int b = n >> 2, s = n & 3;
                s_o[(cw * 16 + row) * D + 32 * b + 8 * cq + s] = o[n][2 * hr];
                s_o[(cw * 16 + row) * D + 32 * b + 8 * cq + 4 + s] = o[n][2 * hr + 1];
            }
        }
    }
    __syncthreads();
    const int64_t pbase = ((int64_t)hkv * MAX_SPLIT + split) * G;
    float *part_o = a.part;
    float *part_ml = a.part + (int64_t)a.n_head_kv * MAX_SPLIT * G * D;
    for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
        const int row = e / D, d = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < CWARPS; ++w) M = fmaxf(M, s_m[w * 16 + row]);
        float acc = 0.f, lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < CWARPS; ++w) {
                const float f = ex2(s_m[w * 16 + row] - M);
                acc += f * s_o[(w * 16 + row) * D + d];
                lsum += f * s_l[w * 16 + row];
            }
        }
        part_o[(pbase + row) * D + d] = acc;
        if (d == 0) {
            part_ml[(pbase + row) * 2] = M;
            part_ml[(pbase + row) * 2 + 1] = lsum;
        }
    }
    if (threadIdx.x == 0 && *s_abort) atomicExch(&g_decode_status, 1);
}

// One output value merged over the splits: split i's (m, l) at ml_src[i * ml_step] and unnormalised
// value at o_src[i * o_step].  With up to MC splits (one wave of split CTAs gives at most 19 per kv
// head at 8 kv heads) every load is issued at once, so the merge costs one round trip to L2; more
// splits take the same steps in rounds of 8.  The weights are ex2(m_i - M) (M the largest split
// maximum); the denominator and the value are summed in split order, so the result is deterministic.
__device__ __forceinline__ float merge_splits(const float2 *ml_src, int64_t ml_step, const float *o_src, int64_t o_step,
                                              int n_split) {
    constexpr int MC = 24;
    float M = -INFINITY, L = 0.f, acc = 0.f;
    if (n_split <= MC) {
        float2 ml[MC];
        float v[MC];
#pragma unroll
        for (int i = 0; i < MC; ++i) {
            if (i < n_split) {
                ml[i] = __ldcg(ml_src + (int64_t)i * ml_step);
                v[i] = __ldcg(o_src + (int64_t)i * o_step);
            } else {
                ml[i] = make_float2(-INFINITY, 0.f);
                v[i] = 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < MC; ++i) M = fmaxf(M, ml[i].x);
#pragma unroll
        for (int i = 0; i < MC; ++i) {
            if (i < n_split) {
                const float w = (ml[i].x == -INFINITY) ? 0.f : ex2(ml[i].x - M);
                L = __fadd_rn(L, __fmul_rn(w, ml[i].y));
                acc = fmaf(w, v[i], acc);
            }
        }
    } else {
        for (int i = 0; i < n_split; ++i) M = fmaxf(M, __ldcg(ml_src + (int64_t)i * ml_step).x);
        for (int i0 = 0; i0 < n_split; i0 += 8) {
            float2 ml[8];
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (i0 + u < n_split) {
                    ml[u] = __ldcg(ml_src + (int64_t)(i0 + u) * ml_step);
                    v[u] = __ldcg(o_src + (int64_t)(i0 + u) * o_step);
                } else {
                    ml[u] = make_float2(-INFINITY, 0.f);
                    v[u] = 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (i0 + u < n_split) {
                    const float w = (ml[u].x == -INFINITY) ? 0.f : ex2(ml[u].x - M);
                    L = __fadd_rn(L, __fmul_rn(w, ml[u].y));
                    acc = fmaf(w, v[u], acc);
                }
            }
        }
    }
    return acc / L;
}

// One CTA per query head, one thread per output value (merge_splits).
template <int D, int NS>
__global__ void __launch_bounds__(D) decode_combine_kernel(const CombineBatch<NS> cb, int group, int n_head_kv) {
    const int seq = NS == 1 ? 0 : (int)blockIdx.y;
    const float *__restrict__ part = cb.part[seq];
    float *__restrict__ out = cb.out[seq];
    const int n_split = cb.n_split[seq];
    const int h = blockIdx.x, d = threadIdx.x;
    const int hkv = h / group, row = h % group;
    // the next kernel (the next step's append) may be scheduled now; it waits for this grid
    asm volatile("griddepcontrol.launch_dependents;");
    // launched as a programmatic dependent of the split pass: wait until its partials are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float *part_ml = part + (int64_t)n_head_kv * MAX_SPLIT * group * D;
    const int64_t p0 = ((int64_t)hkv * MAX_SPLIT) * group + row;   // partial index of split 0
    out[(int64_t)h * D + d] = merge_splits(reinterpret_cast<const float2 *>(part_ml) + p0, group,
                                           part + p0 * D + d, (int64_t)group * D, n_split);
}

// ---- tensor-core split pass for head_dim 128 ---------------------------------------------
// Measured on this part: one thread issues a tcgen05.mma about every 90 cycles whatever its N (16 to
// 128), MMAs that accumulate into the same tensor-memory columns advance only about one per 200
// cycles, and two issuing threads run side by side.  So the pass has two MMA issuers and keeps its
// dependent chains short.  Per key tile (128 keys):
//   S  = Q' K^T      M = 128 rows, N = 128 keys, two chains of 4 MMAs (head dims [0, 64) and
//                    [64, 128)), A = Q' and B = K in shared memory (both K-major); the softmax adds them
//   O' += P' V       M = 128 rows, N = 256, K = 64: 4 MMAs, A = P' and B = V in shared memory (V
//                    MN-major) with the tile's two 64-key halves side by side along N
// Q' holds the G query heads of the group (head slots 0..15, slots >= G zero) eight times over:
// row r = 16 rep + h.  Replica rep owns the 16 keys 16 rep .. 16 rep + 15 of every tile; the thread
// on TMEM lane r keeps the online softmax of row r over those keys alone (its own running max m and
// sum l), so no exchange between threads is needed per tile.  P' row r holds that thread's
// probabilities at its keys' positions within their half and zeros elsewhere (cleared once at the
// start, never written there again), so O' row r accumulates exactly its keys: the columns of the
// row's own half (0..127 for keys 0..63, 128..255 for keys 64..127) hold sum_j p_j V_j, the other
// half is unused.  At the end the replicas of each head are merged (inside each warp by shuffles, then
// across the four warps) into the split's (m, l, O) partial.  A thread rescales its own O' row when its running max grows by more
// than 2^8.
//   warp 0      one lane copies the group's query rows (one bulk copy, first in the queue), then loads
//               K tiles (f16) or their int8 codes (q8_0) by TMA
//   warp 1      allocates TMEM; one lane issues S(k + 1) once the softmax has read S(k)
//   warp 2      one lane issues PV(k) once P'(k) and V(k) are ready
//   warp 3      one lane loads V tiles or codes by TMA (K and V run ahead independently)
//   warps 4-7   softmax, thread = TMEM lane = row of Q' / P' / O'; they also build Q' and merge
//   warps 8-11  (q8_0) dequantise K rows in place into fp16 d*q, one thread per key row
//   warps 12-15 (q8_0) the same for V rows
constexpr int TK = 128;                 // keys per tile
constexpr int TKH = TK / 2;             // keys per half tile (the PV contraction)
// TMEM columns: S chain 0 (head dims [0, 64)) [0, 128), chain 1 [128, 256), O' [256, 512)
constexpr uint32_t TC_COLS = 512;
constexpr uint32_t COL_S = 0, COL_O = 256;
constexpr float TC_RESCALE_LOG2 = 8.0f;

// HS: head slots per replica (8 when the group has at most 8 query heads, else 16).  With 8 slots a
// replica is exactly one 8-row group of the 128-byte-swizzled Q' operand, so Q' is stored once (8 rows)
// and the S MMA reads it for every replica with a zero stride between row groups; the 30 KB saved buy a
// third V slot (V's refill waits for the PV of two tiles before, the longest wait of the pipeline).
template <bool Q8, int HS>
struct TCfg {
    static constexpr int D = 128;
    static constexpr int NREP = 128 / HS;                   // row replicas of the query heads
    static constexpr int RKEYS = TK / NREP;                 // keys of a tile each row owns (= HS)
    static constexpr int QROWS = HS == 8 ? 8 : 128;         // Q' rows stored
    static constexpr int QB = QROWS * D * 2;                // Q' operand: [64-dim block][QROWS][128 B]
    static constexpr int QBLK = QROWS * 128;                // bytes of one 64-dim block of Q'
    static constexpr int OPT = TK * D * 2;                  // fp16 K tile [64-dim block][128 keys][128 B], or
                                                            // V tile [half][64-dim block][64 keys][128 B]
    static constexpr int PB = 128 * TKH * 2;                // P' operand: [128 rows][64 keys], 16 KB
    static constexpr int NP = HS == 8 ? 1 : 2;              // P' buffers
    static constexpr int RAWB = TK * D;                     // int8 codes of a K or V tile: 16 KB
    static constexpr int NK = 3, NV = HS == 8 ? 3 : 2;      // ring slots; q8_0 codes land in place
    static constexpr int QSB = HS == 8 ? 8 * D * 4 : 0;     // staging of the query rows (else P' buffer 1)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + QB;
    static constexpr int OFF_V = OFF_K + NK * OPT;
    static constexpr int OFF_P = OFF_V + NV * OPT;
    static constexpr int OFF_QS = HS == 8 ? OFF_P + NP * PB : OFF_P + PB;
    static constexpr int OFF_BAR = OFF_P + NP * PB + QSB;
    static constexpr int USED = OFF_BAR + 512;
    static constexpr int ALLOC = USED + 1024;
    static_assert(ALLOC <= 232448, "shared memory plan too large");
    // the merge at the end reuses the K ring (a row of D + 4 floats per warp and head slot) and P' buffer 0
    // (their maxima and sums)
    static constexpr int OFF_MRG = OFF_K;
    static constexpr int OFF_ML = OFF_P;
    static constexpr int NDQ = 128;                         // dequantising threads per K or V (q8_0)
    static constexpr int THREADS = Q8 ? 512 : 256;
    static constexpr int CTAS = 1;                          // CTAs per SM (all 512 TMEM columns)
};

// q8_0 codes land inside the fp16 slot they are dequantised into, at the bytes of the fp16 row's first
// 64-dim block: K codes as one 128-key box at the slot's start (code row t at t * 128), V codes as two
// 64-key boxes at the starts of the blocks (half 0, dims 0-63) and (half 1, dims 0-63).  A thread reads
// its whole code row before it writes its fp16 row, whose first block covers exactly those bytes and
// whose second block lies where no codes are, so no thread overwrites another thread's codes.
enum TcBar {
    T_QREADY, T_QRAW, T_SFULL, T_SFREE, T_PFULL0, T_PFULL1, T_ODONE0, T_ODONE1, T_XCHG, T_DRAIN, T_DRAIN2, T_STALL,
    T_APPEND, T_KFULL, T_KEMPTY = T_KFULL + 4, T_VFULL = T_KEMPTY + 4, T_VEMPTY = T_VFULL + 4, T_KRAW = T_VEMPTY + 4,
    T_VRAW = T_KRAW + 4, T_NBAR = T_VRAW + 4
};
static_assert(T_NBAR * 8 + 8 <= 512, "barrier area too small");   // + TMEM address and abort flag

// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled block of 128-byte rows
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}
// the fp16 K tile: head dims [64 cb, 64 cb + 64) of key row r, chunk c (8 dims) of that block
__device__ __forceinline__ uint32_t k_off(int r, int cb, int c) { return (uint32_t)(cb * (TK * 128)) + sw128(r, c); }
// the fp16 V tile: key row r lies in half r / 64 at row r % 64
__device__ __forceinline__ uint32_t v_off(int r, int cb, int c) {
    return (uint32_t)((2 * (r / TKH) + cb) * (TKH * 128)) + sw128(r % TKH, c);
}
// 4 int8 codes times the fp16 scale, as two fp16x2 words (one rounding each): the sign bit flipped
// makes each code q + 128 as an unsigned byte, which under the high byte 0x64 is the fp16 value
// 1024 + q + 128 (exact); subtracting 1152 leaves q
__device__ __forceinline__ void dequant4(uint32_t w, __half2 d2, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    __half2 ra = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&a), bias), d2);
    __half2 rb = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&b), bias), d2);
    lo = *reinterpret_cast<uint32_t *>(&ra);
    hi = *reinterpret_cast<uint32_t *>(&rb);
}


// NS: sequences of a batch the parameters hold (1, or MAX_BATCH for a batched call; grid z = sequence)
template <bool Q8, int DT, int NS, int HS>
__global__ void __launch_bounds__(TCfg<Q8, HS>::THREADS, 1)
    decode_tc_kernel(const __grid_constant__ TcBatch<NS> b) {
    using L = TCfg<Q8, HS>;
    constexpr int NREP = L::NREP, RKEYS = L::RKEYS;
    constexpr int D = 128;
    const int seq = NS == 1 ? 0 : (int)blockIdx.z;
    const DecodeArgs &a = b.a[seq];
    const CUtensorMap *tm_k = &b.tk[seq], *tm_v = &b.tv[seq];
    if ((int)blockIdx.x >= a.n_split) return;   // a batch's shorter sequences use fewer splits
    if (threadIdx.x == 0) KVC_TR(0, 0);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + T_NBAR);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    const int split = blockIdx.x, hkv = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.group;
    const int j_begin = split * a.split_len;
    const int j_end = min(a.n_keys, j_begin + a.split_len);
    const int T = (j_end - j_begin + TK - 1) / TK;   // tiles of this split
    // fused decode step: this CTA stores the new token (at n_keys - 1, inside its last tile)
    const bool owns_new = a.k_new != nullptr && split == a.n_split - 1;

    if (threadIdx.x == 0) {
        *s_abort = 0;
        mbar_init(&bars[T_QREADY], 128);
        mbar_init(&bars[T_QRAW], 1);
        mbar_init(&bars[T_SFULL], 1);
        mbar_init(&bars[T_SFREE], 128);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[T_PFULL0 + i], 128);
            mbar_init(&bars[T_ODONE0 + i], 1);
        }
        mbar_init(&bars[T_XCHG], 128);
        mbar_init(&bars[T_DRAIN], 1);
        mbar_init(&bars[T_DRAIN2], 1);
        mbar_init(&bars[T_STALL], 1);   // nothing arrives here: only the test hook waits on it
        mbar_init(&bars[T_APPEND], 1);  // the new token is in the cache (fused step)
        for (int s = 0; s < L::NK; ++s) {
            mbar_init(&bars[T_KFULL + s], Q8 ? L::NDQ : 1);
            mbar_init(&bars[T_KEMPTY + s], 1);
        }
        for (int s = 0; s < L::NV; ++s) {
            mbar_init(&bars[T_VFULL + s], Q8 ? L::NDQ : 1);
            mbar_init(&bars[T_VEMPTY + s], 1);
        }
        for (int s = 0; s < (Q8 ? L::NK : 0); ++s) mbar_init(&bars[T_KRAW + s], 1);
        for (int s = 0; s < (Q8 ? L::NV : 0); ++s) mbar_init(&bars[T_VRAW + s], 1);
        fence_mbar_init();
        tma_prefetch_desc(tm_k);
        tma_prefetch_desc(tm_v);
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, TC_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    if ((warp == 0 || warp == 3) && lane == 0) {
        // the ring's first tiles into L2 while the kernel before this one finishes (a hint, safe before the
        // wait; prefetching further ahead inside the loop measured slower)
        const int kv = warp == 3, n = kv ? L::NV : L::NK;
        for (int k = 0; k < T && k < n; ++k) {
            const int j = j_begin + k * TK;
            for (int cb = 0; cb < (Q8 ? 1 : 2); ++cb) {
                if (!kv) tma_prefetch_l2_3d(tm_k, cb * 64, j, hkv);
                else for (int hf = 0; hf < 2; ++hf) tma_prefetch_l2_3d(tm_v, cb * 64, j + hf * TKH, hkv);
            }
        }
    }
    // inputs written by the kernels before this one are read only past this point
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    if (threadIdx.x == 0) KVC_TR(0, 1);

    if (warp == 0 || warp == 3) {
        // ------------------------------------------------------------------ producers (K: warp 0, V: warp 3)
        // Each loads its tiles into ring slots as soon as the MMAs that read a slot's previous tile have
        // completed; q8_0 codes complete on the slot's raw barrier (the dequantisers then fill the slot),
        // fp16 values on its full barrier.  Warp 0 first copies the group's query rows (G x 128 values in
        // the input type, contiguous) into a staging area, where the softmax threads build Q' from them.
        if (lane == 0) {
            const bool is_v = warp == 3;
            const int n = is_v ? L::NV : L::NK;
            const int bar_fill = is_v ? (Q8 ? T_VRAW : T_VFULL) : (Q8 ? T_KRAW : T_KFULL);
            const int bar_empty = is_v ? T_VEMPTY : T_KEMPTY;
            uint8_t *ring = sm + (is_v ? L::OFF_V : L::OFF_K);
            bool q_issued = false;
            if (!is_v) {
                constexpr uint32_t QE = DT == KVC_IN_F32 ? 4 : 2;
                const uint32_t qbytes = (uint32_t)G * D * QE;
                mbar_arrive_expect_tx(&bars[T_QRAW], qbytes);
                bulk_load(sm + L::OFF_QS, static_cast<const uint8_t *>(a.q) + (size_t)hkv * qbytes, qbytes,
                          &bars[T_QRAW]);
                q_issued = true;
            }
            int issued = 0;
            for (int k = 0; k < T; ++k) {
                const int j = j_begin + k * TK;
                const int s = k % n;
                if (k >= n && !mbar_wait(&bars[bar_empty + s], ((k / n) - 1) & 1, s_abort)) break;
                // the last tile holds the new token: copy it once the token is stored
                if (owns_new && k == T - 1 && !mbar_wait(&bars[T_APPEND], 0, s_abort)) break;
                KVC_TR(1 + (int)is_v, k);
                uint8_t *dst = ring + s * L::OPT;
                if constexpr (Q8) {
                    mbar_arrive_expect_tx(&bars[bar_fill + s], L::RAWB);
                    if (!is_v) {
                        tma_load_3d(dst, tm_k, &bars[bar_fill + s], 0, j, hkv);
                    } else {
                        for (int hf = 0; hf < 2; ++hf)
                            tma_load_3d(dst + v_off(hf * TKH, 0, 0), tm_v, &bars[bar_fill + s], 0, j + hf * TKH, hkv);
                    }
                } else {
                    mbar_arrive_expect_tx(&bars[bar_fill + s], L::OPT);
                    if (!is_v) {
                        for (int cb = 0; cb < 2; ++cb)
                            tma_load_3d(dst + k_off(0, cb, 0), tm_k, &bars[bar_fill + s], cb * 64, j, hkv);
                    } else {
                        for (int hf = 0; hf < 2; ++hf)
                            for (int cb = 0; cb < 2; ++cb)
                                tma_load_3d(dst + v_off(hf * TKH, cb, 0), tm_v, &bars[bar_fill + s], cb * 64,
                                            j + hf * TKH, hkv);
                    }
                }
                ++issued;
            }
            if (*s_abort) {
                // after a wait gave up: let the copies still in flight land before the CTA exits
                volatile int never = 0;
                for (int st = 0; st < n && st < issued; ++st) {
                    const int last = st + ((issued - 1 - st) / n) * n;
                    mbar_wait(&bars[bar_fill + st], (last / n) & 1, &never, 200000000ull);
                }
                if (q_issued) mbar_wait(&bars[T_QRAW], 0, &never, 200000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ S issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_f16(128, TK, 0, 0);      // A = Q' (K-major), B = K (K-major)
            const uint32_t sQ = smem_u32(sm + L::OFF_Q), sK = smem_u32(sm + L::OFF_K);
            bool ok = mbar_wait(&bars[T_QREADY], 0, s_abort);
            tc_fence_after();
            KVC_TR(0, 2);
            for (int k = 0; ok && k < T; ++k) {
                // S(k) into the S columns once every softmax thread has read S(k - 1)
                if (k > 0 && !mbar_wait(&bars[T_SFREE], (k - 1) & 1, s_abort)) { ok = false; break; }
                const int st = k % L::NK;
                if (!mbar_wait(&bars[T_KFULL + st], (k / L::NK) & 1, s_abort)) { ok = false; break; }
                tc_fence_after();
                KVC_TR(3, k);
                const uint32_t kb = sK + st * L::OPT;
                // two independent chains, interleaved: head dims [0, 64) into columns [0, 128), [64, 128)
                // into [128, 256); k-step i of chain c covers head dims 64 c + 16 i .. + 15
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint32_t qo = (uint32_t)(c * L::QBLK + i * 32), ko = (uint32_t)(c * (TK * 128) + i * 32);
                        umma_f16_ss(tmem + COL_S + 128 * c, sdesc_sw128(sQ + qo, 16, HS == 8 ? 0 : 1024),
                                    sdesc_sw128(kb + ko, 16, 1024), IDESC_S, i > 0);
                    }
                umma_commit(&bars[T_SFULL]);
                umma_commit(&bars[T_KEMPTY + st]);
                KVC_TR(4, k);
            }
            if (*s_abort) {
                // after a wait gave up: let the MMAs in flight finish before TMEM is freed
                volatile int never = 0;
                umma_commit(&bars[T_DRAIN]);
                mbar_wait(&bars[T_DRAIN], 0, &never, 200000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------------ PV issuer
        if (owns_new) {
            // fused step: store the new token first (the first P comes much later); its bytes reach the
            // TMA copies of the last tile through the async-proxy fence and the barrier's release
            store_new_token<Q8, DT>(a, hkv, lane);
            fence_proxy_async_global();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[T_APPEND]);
        }
        if (lane == 0) {
            constexpr uint32_t IDESC_O = idesc_f16(128, 2 * D, 0, 1);   // A = P' (K-major), B = V (MN-major)
            const uint32_t sP = smem_u32(sm + L::OFF_P), sV = smem_u32(sm + L::OFF_V);
            bool ok = true;
            for (int k = 0; ok && k < T; ++k) {
                // test hook: a bounded wait on a barrier nothing arrives at, in place of the first P
                // wait; it gives up after stall_ns (raising the abort flag) with S MMAs in flight
                if (a.stall_ns != 0 && k == 0) {
                    mbar_wait(&bars[T_STALL], 0, s_abort, a.stall_ns);
                    ok = false;
                    break;
                }
                // O' += P'(k) V(k): k-step ks covers keys [16 ks, 16 ks + 16) of both halves
                if (!mbar_wait(&bars[T_PFULL0 + k % L::NP], (k / L::NP) & 1, s_abort)) { ok = false; break; }
                const int vs = k % L::NV;
                if (!mbar_wait(&bars[T_VFULL + vs], (k / L::NV) & 1, s_abort)) { ok = false; break; }
                tc_fence_after();
                KVC_TR(5, k);
                const uint32_t pb = sP + (k % L::NP) * L::PB, vb = sV + vs * L::OPT;
#pragma unroll
                for (int ks = 0; ks < TKH / 16; ++ks)
                    umma_f16_ss(tmem + COL_O, sdesc_sw128(pb + ks * 32, 16, 1024),
                                sdesc_sw128(vb + ks * 16 * 128, TKH * 128, 1024), IDESC_O, (k > 0 || ks > 0) ? 1u : 0u);
                umma_commit(&bars[T_ODONE0 + (k & 1)]);
                umma_commit(&bars[T_VEMPTY + vs]);
                KVC_TR(6, k);
            }
            if (*s_abort) {
                volatile int never = 0;
                umma_commit(&bars[T_DRAIN2]);
                mbar_wait(&bars[T_DRAIN2], 0, &never, 200000000ull);
            }
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------------ softmax (row per thread)
        const int quarter = warp & 3;                   // this warp's TMEM lanes: 32 quarter .. + 31
        const int r = quarter * 32 + lane;              // row of Q', P' and O'
        const int rep = r / HS, h = r % HS;             // replica, head slot
        const int hf = quarter >> 1;                    // the half of the tile its keys lie in
        const int sub = lane / HS;                      // which of the warp's replicas (its 32 keys)
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        bool ok = true;
        {
            // Q' row r (head slot h of the group, zero for h >= G; with 8 slots only rows 0-7 are stored)
            // from the staged query rows; row r of P' buffer 0 cleared (with two buffers, buffer 1 held
            // the staged rows and is cleared before its first use, once every thread has read them)
            ok = mbar_wait(&bars[T_QRAW], 0, s_abort);
            uint8_t *qt = sm + L::OFF_Q;
            constexpr int QW = DT == KVC_IN_F32 ? 2 : 1;        // 16-byte words per 8 values
            // 8 stored rows: thread r converts chunk r / 8 of row r % 8; 128 rows: thread r its own row
            const int qrow = HS == 8 ? (r & 7) : r, qslot = qrow % HS;
            const uint8_t *qs = sm + L::OFF_QS + qslot * D * (DT == KVC_IN_F32 ? 4 : 2);
#pragma unroll 4
            for (int cc = HS == 8 ? (r >> 3) : 0; cc < (HS == 8 ? (r >> 3) + 1 : D / 8); ++cc) {
                uint4 raw[QW];
#pragma unroll
                for (int i = 0; i < QW; ++i)
                    raw[i] = (ok && qslot < G) ? *reinterpret_cast<const uint4 *>(qs + (cc * QW + i) * 16)
                                               : make_uint4(0u, 0u, 0u, 0u);
                float x[8];
                to_f32x8<DT>(raw, 0, x);
                *reinterpret_cast<uint4 *>(qt + (cc >> 3) * L::QBLK + sw128(qrow, cc & 7)) =
                    make_uint4(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]), pack_half2(x[4], x[5]),
                               pack_half2(x[6], x[7]));
            }
            uint4 *prow = reinterpret_cast<uint4 *>(sm + L::OFF_P + r * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) prow[c] = make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
            mbar_arrive(&bars[T_QREADY]);
            if (threadIdx.x == 128) KVC_TR(0, 6);
        }
        float m_run = -INFINITY, l_run = 0.f;
        int pv_seen[2] = {0, 0};
        auto wait_pv = [&](int j) -> bool {  // PV(j) and every MMA before it have completed
            const int bb = j & 1, n = j >> 1;
            if (pv_seen[bb] > n) return true;
            if (!mbar_wait(&bars[T_ODONE0 + bb], n & 1, s_abort)) return false;
            pv_seen[bb] = n + 1;
            tc_fence_after();
            return true;
        };
        const float sl2 = a.scale_log2;
        for (int k = 0; ok && k < T; ++k) {
            if (!mbar_wait(&bars[T_SFULL], k & 1, s_abort)) { ok = false; break; }
            tc_fence_after();
            if (threadIdx.x == 128) KVC_TR(7, k);
            // the warp's 32 key columns (its two replicas' keys) of both chains, then S may be overwritten
            uint32_t s0[32], s1[32];
            tmem_ld32(tmem + COL_S + 32 * quarter + lane_base, s0);
            tmem_ld32(tmem + COL_S + 128 + 32 * quarter + lane_base, s1);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&bars[T_SFREE]);
            if (threadIdx.x == 128) KVC_TR(8, k);
            const int key0 = j_begin + k * TK + RKEYS * rep;   // absolute position of my first key
            float x[RKEYS];
#pragma unroll
            for (int i = 0; i < RKEYS; ++i) {
                // the warp's 32 columns hold its replicas' keys in order: mine are sub * RKEYS + i
                float s = __uint_as_float(s0[i]) + __uint_as_float(s1[i]);
#pragma unroll
                for (int q = 1; q < 32 / RKEYS; ++q)
                    if (sub == q) s = __uint_as_float(s0[q * RKEYS + i]) + __uint_as_float(s1[q * RKEYS + i]);
                x[i] = key0 + i < j_end ? s * sl2 : -INFINITY;
            }
            float mx = fmax3(x[0], x[1], x[2]);
#pragma unroll
            for (int i = 3; i < RKEYS; i += 2) mx = fmax3(mx, x[i], i + 1 < RKEYS ? x[i + 1] : x[i]);
            // lazy rescale: the running max moves only when it grows by more than 2^8 (a row that has
            // seen no visible key yet takes the first maximum; its O' row is still zero)
            float alpha = 1.f;
            bool grow = false;
            if (m_run == -INFINITY) {
                m_run = mx;
            } else if (mx > m_run + TC_RESCALE_LOG2) {
                alpha = ex2(m_run - mx);
                m_run = mx;
                grow = true;
            }
            const float m_sub = m_run == -INFINITY ? 0.f : m_run;   // all keys masked so far: p = 0
            uint32_t pk[RKEYS / 2];
            float rs = 0.f;
#pragma unroll
            for (int i = 0; i < RKEYS; i += 2) {
                const float p0 = ex2(x[i] - m_sub), p1 = ex2(x[i + 1] - m_sub);
                rs += p0 + p1;
                pk[i / 2] = pack_half2(p0, p1);
            }
            l_run = l_run * alpha + rs;
            // P' buffer k % NP was last read by PV(k - NP); O' must hold PV(k - 1) before a rescale
            if (k >= L::NP && !wait_pv(k - L::NP)) { ok = false; break; }
            if (__any_sync(0xffffffffu, grow)) {
                if (k >= 1 && !wait_pv(k - 1)) { ok = false; break; }
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    const uint32_t ta = tmem + COL_O + 128 * hf + 32 * c + lane_base;
                    tmem_ld32(ta, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(ta, o);
                }
                tmem_st_wait();
            }
            // my RKEYS probabilities at my keys' positions in row r of P' buffer k % NP: my keys are
            // RKEYS (rep % (NREP / 2)) .. + RKEYS - 1 of my half, 16-byte chunks c0 .. c0 + RKEYS / 8 - 1
            {
                uint8_t *prow = sm + L::OFF_P + (k % L::NP) * L::PB + r * 128;
                if (L::NP == 2 && k == 1) {
                    // buffer 1 held the staged query rows: clear my row once every thread has read them
                    if (!mbar_wait(&bars[T_QREADY], 0, s_abort)) { ok = false; break; }
#pragma unroll
                    for (int c = 0; c < 8; ++c) reinterpret_cast<uint4 *>(prow)[c] = make_uint4(0u, 0u, 0u, 0u);
                }
                const int c0 = (RKEYS / 8) * (rep % (NREP / 2));
#pragma unroll
                for (int c = 0; c < RKEYS / 8; ++c)
                    *reinterpret_cast<uint4 *>(prow + (((c0 + c) ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars[T_PFULL0 + k % L::NP]);
            if (threadIdx.x == 128) KVC_TR(9, k);
        }
        // ---- epilogue (the operand rings are free once the last PV has completed).  The replicas of each
        // head slot are merged first inside the warp - lanes h, h + HS, ... hold slot h's replicas - by a
        // reduce-scatter over shuffles that leaves each lane a quarter (8 slots) or half (16 slots) of the
        // slot's columns, written to shared memory; then across the four warps, one warp per head and a
        // lane per four head dims.  The orders are fixed, so the result is deterministic.
        if (threadIdx.x == 128) KVC_TR(0, 3);
        constexpr int RW = 32 / HS;                  // replicas of a head slot in one warp (4 or 2)
        constexpr int WROW = D + 4;                  // floats per (warp, slot) row in shared memory
        float *wm = reinterpret_cast<float *>(sm + L::OFF_MRG);   // [quarter][slot][WROW]
        float *wml = reinterpret_cast<float *>(sm + L::OFF_ML);   // [quarter][slot][2]: (max, sum)
        static_assert(4 * HS * WROW * 4 <= L::NK * L::OPT && 4 * HS * 8 <= L::PB, "merge areas too small");
        bool have = ok && T > 0 && wait_pv(T - 1);
        have = __all_sync(0xffffffffu, have);        // the shuffles below need the whole warp
        if (have) {
            float mw = m_run;
#pragma unroll
            for (int off = HS; off < 32; off <<= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, off));
            const float w = m_run == -INFINITY ? 0.f : ex2(m_run - mw);
            float lw = w * l_run;
#pragma unroll
            for (int off = HS; off < 32; off <<= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
            float *dst = wm + (quarter * HS + h) * WROW;
            const bool up16 = (lane & 16) != 0, up8 = (lane & 8) != 0;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + COL_O + 128 * hf + 32 * c + lane_base, o);
                tmem_ld_wait();
                // lanes 16 apart: the lower keeps columns 0-15 of the chunk, the upper 16-31
                float k1[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float lo = __uint_as_float(o[e]) * w, hi = __uint_as_float(o[e + 16]) * w;
                    k1[e] = (up16 ? hi : lo) + __shfl_xor_sync(0xffffffffu, up16 ? lo : hi, 16);
                }
                if constexpr (RW == 4) {
                    // lanes 8 apart: the lower keeps 8 of those 16 columns, the upper the other 8
                    float k2[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        k2[e] = (up8 ? k1[e + 8] : k1[e]) + __shfl_xor_sync(0xffffffffu, up8 ? k1[e] : k1[e + 8], 8);
                    float *d8 = dst + 32 * c + 16 * up16 + 8 * up8;
                    *reinterpret_cast<float4 *>(d8) = make_float4(k2[0], k2[1], k2[2], k2[3]);
                    *reinterpret_cast<float4 *>(d8 + 4) = make_float4(k2[4], k2[5], k2[6], k2[7]);
                } else {
                    float *d16 = dst + 32 * c + 16 * up16;
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *reinterpret_cast<float4 *>(d16 + e) = make_float4(k1[e], k1[e + 1], k1[e + 2], k1[e + 3]);
                }
            }
            if (lane < HS) *reinterpret_cast<float2 *>(wml + 2 * (quarter * HS + h)) = make_float2(mw, lw);
        } else {
            ok = false;
        }
        if (threadIdx.x == 128) KVC_TR(0, 7);
        mbar_arrive(&bars[T_XCHG]);
        bool wrote = false;
        if (ok && mbar_wait(&bars[T_XCHG], 0, s_abort) && !*s_abort) {
            const int64_t pbase = ((int64_t)hkv * MAX_SPLIT + split) * G;
            float *part_o = a.part;
            float *part_ml = a.part + (int64_t)a.n_head_kv * MAX_SPLIT * G * D;
            for (int hh = quarter; hh < G; hh += 4) {
                float2 ml[4];
                float M = -INFINITY;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    ml[q] = *reinterpret_cast<const float2 *>(wml + 2 * (q * HS + hh));
                    M = fmaxf(M, ml[q].x);
                }
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                float lsum = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float wq = ml[q].x == -INFINITY ? 0.f : ex2(ml[q].x - M);
                    lsum += wq * ml[q].y;
                    const float4 v = *reinterpret_cast<const float4 *>(wm + (q * HS + hh) * WROW + 4 * lane);
                    acc.x += wq * v.x;
                    acc.y += wq * v.y;
                    acc.z += wq * v.z;
                    acc.w += wq * v.w;
                }
                *reinterpret_cast<float4 *>(part_o + (pbase + hh) * D + 4 * lane) = acc;
                if (lane == 0) *reinterpret_cast<float2 *>(part_ml + (pbase + hh) * 2) = make_float2(M, lsum);
            }
            wrote = true;
        }
        if (threadIdx.x == 128) KVC_TR(0, 4);
        if (!wrote && r < G) {
            // a split that gave up leaves an empty partial (m = -inf, l = 0), which the combine
            // weighs 0, rather than another call's leftovers
            float *part_ml = a.part + (int64_t)a.n_head_kv * MAX_SPLIT * G * D;
            const int64_t pi = ((int64_t)hkv * MAX_SPLIT + split) * G + r;
            part_ml[pi * 2] = -INFINITY;
            part_ml[pi * 2 + 1] = 0.f;
        }
    } else if constexpr (Q8) {
        // ------------------------------------------------------------------ dequantise (q8_0)
        if (warp >= 8) {
            const int kv = warp >= 12;              // warps 8-11: K rows, warps 12-15: V rows
            const int t = (threadIdx.x - 256) & 127;   // key row of the tile
            const uint16_t *scl = kv ? a.vs : a.ks;
            const int n = kv ? L::NV : L::NK;
            const int bar_full = kv ? T_VFULL : T_KFULL;
            uint8_t *ring = sm + (kv ? L::OFF_V : L::OFF_K);
            // the four fp16 scales of my key's row (keys past the end: any finite scale, their codes are
            // zero-filled), loaded through L2: the append before this kernel may have written them
            auto scales = [&](int k) -> uint2 {
                // the last tile's scales include the new token's (fused step): read them once it is stored
                if (owns_new && k == T - 1) mbar_wait(&bars[T_APPEND], 0, s_abort);
                const int key = min(j_begin + k * TK + t, a.n_keys - 1);
                return __ldcg(reinterpret_cast<const uint2 *>(scl + a.layer * a.g.s_layer + hkv * a.g.s_head +
                                                               (int64_t)key * a.g.s_tok));
            };
            const int bar_raw = kv ? T_VRAW : T_KRAW;
            uint2 sw_n = T > 0 ? scales(0) : make_uint2(0u, 0u);
            for (int k = 0; k < T; ++k) {
                const uint2 sw = sw_n;
                if (k + 1 < T) sw_n = scales(k + 1);
                const int s = k % n;
                if (!mbar_wait(&bars[bar_raw + s], (k / n) & 1, s_abort)) break;
                if (t == 0) KVC_TR(10 + 2 * kv, k);
                uint8_t *slot = ring + s * L::OPT;
                // my row's 128 codes (in the bytes of my fp16 row's first block): 16-byte chunk i holds head
                // dims 16 i .. 16 i + 15 (block i / 2); all read before any write
                uint4 q[D / 16];
#pragma unroll
                for (int i = 0; i < D / 16; ++i)
                    q[i] = *reinterpret_cast<const uint4 *>(slot + (kv ? v_off(t, 0, i) : k_off(t, 0, i)));
#pragma unroll
                for (int i = 0; i < D / 16; ++i) {
                    const int blk = i >> 1;
                    const uint32_t w2 = blk < 2 ? sw.x : sw.y;
                    const unsigned short sb = (unsigned short)(w2 >> (16 * (blk & 1)));
                    const __half2 d2 = __halves2half2(__ushort_as_half(sb), __ushort_as_half(sb));
                    uint32_t o[8];
                    dequant4(q[i].x, d2, o[0], o[1]);
                    dequant4(q[i].y, d2, o[2], o[3]);
                    dequant4(q[i].z, d2, o[4], o[5]);
                    dequant4(q[i].w, d2, o[6], o[7]);
                    // fp16 chunks 2 i and 2 i + 1 of the row: 64-dim block i / 4, chunk (2 i) % 8 in it
                    const int cb = i >> 2, c0 = (2 * i) & 7;
                    const uint32_t o0 = kv ? v_off(t, cb, c0) : k_off(t, cb, c0);
                    const uint32_t o1 = kv ? v_off(t, cb, c0 + 1) : k_off(t, cb, c0 + 1);
                    *reinterpret_cast<uint4 *>(slot + o0) = make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4 *>(slot + o1) = make_uint4(o[4], o[5], o[6], o[7]);
                }
                // order the operand writes before the MMA (async proxy) reads them, and before the next
                // TMA into this slot (which comes after those MMAs)
                fence_proxy_async_smem();
                mbar_arrive(&bars[bar_full + s]);
                if (t == 0) KVC_TR(11 + 2 * kv, k);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) KVC_TR(0, 5);
    if (threadIdx.x == 0 && *s_abort) atomicExch(&g_decode_status, 1);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TC_COLS);
    }
}

// The tensor-core split pass and the combine, one launch each, over n_seq sequences (NS = 1, or
// MAX_BATCH for a batched call).  Sequence i: cache caches[i], arguments a0[i] (its q and its scratch
// as part), output outs[i].  A fused step (a0[i].k_new set) stores the token in the split pass.  The sequences share the SMs evenly: one wave over (split, kv head,
// sequence), whole tiles per split.
template <bool Q8, int DT, int NS>
int launch_tc(const kvc_cache *caches, const DecodeArgs *a0, int n_seq, int n_head_q, float *const *outs,
              cudaStream_t s) {
    using L = TCfg<Q8, 16>;   // the larger shared-memory plan; both variants take the same launch shape
    constexpr int D = 128;
    TcBatch<NS> b;
    CombineBatch<NS> cb;
    memset(&b, 0, sizeof(b));
    memset(&cb, 0, sizeof(cb));
    int target = (L::CTAS * sm_count()) / (a0[0].n_head_kv * n_seq);
    if (target < 1) target = 1;
    int max_split = 1;
    for (int i = 0; i < n_seq; ++i) {
        DecodeArgs a = a0[i];
        int n_split = (a.n_keys + TK - 1) / TK;
        if (n_split > target) n_split = target;
        if (n_split > MAX_SPLIT) n_split = MAX_SPLIT;
        if (n_split < 1) n_split = 1;
        int len = (a.n_keys + n_split - 1) / n_split;
        len = (len + TK - 1) / TK * TK;
        n_split = (a.n_keys + len - 1) / len;
        a.split_len = len;
        a.n_split = n_split;
        const kvc_cache &c = caches[i];
        const Geom &g = a.g;
        const int eb = Q8 ? 1 : 2;
        const uint8_t *kb = static_cast<const uint8_t *>(c.k_q), *vb = static_cast<const uint8_t *>(c.v_q);
        const CUtensorMapDataType dt = Q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        const uint32_t box0 = 128 / eb;   // 128-byte rows: all 128 codes (q8_0) or 64 halves (f16)
        // K by 128-key tiles, V by 64-key halves (the halves sit side by side along the PV MMA's N)
        if (!make_map_3d(&b.tk[i], dt, kb + (int64_t)eb * a.layer * g.c_layer, D, a.n_keys, a.n_head_kv,
                         eb * g.c_tok, eb * g.c_head, box0, TK, 1, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map_3d(&b.tv[i], dt, vb + (int64_t)eb * a.layer * g.c_layer, D, a.n_keys, a.n_head_kv,
                         eb * g.c_tok, eb * g.c_head, box0, TKH, 1, CU_TENSOR_MAP_SWIZZLE_128B))
            return KVC_ECUDA;
        b.a[i] = a;
        cb.part[i] = a.part;
        cb.out[i] = outs[i];
        cb.n_split[i] = n_split;
        if (n_split > max_split) max_split = n_split;
    }
    const uint64_t stall_ns = take_test_stall(KVC_TEST_DECODE);
    for (int i = 0; i < n_seq; ++i) b.a[i].stall_ns = stall_ns;
    const int group = a0[0].group, n_head_kv = a0[0].n_head_kv;
    auto kern = group <= 8 ? decode_tc_kernel<Q8, DT, NS, 8> : decode_tc_kernel<Q8, DT, NS, 16>;
    const int smem = group <= 8 ? TCfg<Q8, 8>::ALLOC : TCfg<Q8, 16>::ALLOC;
    if (allow_dynamic_smem((const void *)kern, smem) != KVC_OK) return KVC_ECUDA;
    // both passes may start while the previous kernel of the stream finishes; each waits for it on
    // the device before reading what it wrote
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(max_split, n_head_kv, n_seq);
    cfg.blockDim = dim3(L::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, b) != cudaSuccess) return KVC_ECUDA;
    cudaLaunchConfig_t cfg2 = {};
    cfg2.gridDim = dim3(n_head_q, n_seq);
    cfg2.blockDim = dim3(D);
    cfg2.dynamicSmemBytes = 0;
    cfg2.stream = s;
    cfg2.attrs = attr;
    cfg2.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg2, decode_combine_kernel<D, NS>, cb, group, n_head_kv) != cudaSuccess)
        return KVC_ECUDA;
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
}

// The fused-step fields of a: the token's rows k and v and the cache's buffers it is stored in.
void set_fused(DecodeArgs &a, const kvc_cache &c, const void *k, const void *v) {
    a.k_new = k;
    a.v_new = v;
    a.kq = c.k_q;
    a.vq = c.v_q;
    a.ks_w = static_cast<uint16_t *>(c.k_s);
    a.vs_w = static_cast<uint16_t *>(c.v_s);
}

template <int D, bool Q8, int DT>
int launch_t(const kvc_cache &c, int layer, int pos, const void *q, int n_head_q, float *out,
             float *scratch, cudaStream_t s, const void *k_new = nullptr, const void *v_new = nullptr) {
    using L = DCfg<D, Q8>;
    DecodeArgs a;
    memset(&a, 0, sizeof(a));
    a.q = q;
    a.ks = static_cast<const uint16_t *>(c.k_s);
    a.vs = static_cast<const uint16_t *>(c.v_s);
    a.part = scratch;
    a.g = geom_of(c.d);
    a.layer = layer;
    a.n_keys = pos + 1;
    a.n_head_kv = c.d.n_head_kv;
    a.group = n_head_q / c.d.n_head_kv;
    a.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)D));
    a.stall_ns = 0;
    if (k_new != nullptr) set_fused(a, c, k_new, v_new);
    if constexpr (D == 128) {
        return launch_tc<Q8, DT, 1>(&c, &a, 1, n_head_q, &out, s);
    } else {
    // one wave: CTAS_PER_SM CTAs per SM over (split, kv head), whole stages per split
    const int target = (CTAS_PER_SM * sm_count()) / a.n_head_kv;
    int n_split = (a.n_keys + STAGE_KEYS - 1) / STAGE_KEYS;
    if (n_split > target) n_split = target;
    if (n_split > MAX_SPLIT) n_split = MAX_SPLIT;
    if (n_split < 1) n_split = 1;
    int len = (a.n_keys + n_split - 1) / n_split;
    len = (len + STAGE_KEYS - 1) / STAGE_KEYS * STAGE_KEYS;
    n_split = (a.n_keys + len - 1) / len;
    a.split_len = len;
    a.n_split = n_split;
    // K and V of this layer as (element in row, key, kv head); keys past pos read as zeros
    CUtensorMap tk, tv;
    const Geom &g = a.g;
    const uint8_t *kb = static_cast<const uint8_t *>(c.k_q), *vb = static_cast<const uint8_t *>(c.v_q);
    const int eb = Q8 ? 1 : 2;
    const CUtensorMapDataType dt = Q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUtensorMapSwizzle sw = L::BLK_ROW == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const uint32_t box0 = L::BLK_ROW / eb;
    if (!make_map_3d(&tk, dt, kb + (int64_t)eb * layer * g.c_layer, D, a.n_keys, a.n_head_kv, eb * g.c_tok,
                     eb * g.c_head, box0, STAGE_KEYS, 1, sw) ||
        !make_map_3d(&tv, dt, vb + (int64_t)eb * layer * g.c_layer, D, a.n_keys, a.n_head_kv, eb * g.c_tok,
                     eb * g.c_head, box0, STAGE_KEYS, 1, sw))
        return KVC_ECUDA;
    auto split_kern = decode_split_kernel<D, Q8, DT>;
    if (allow_dynamic_smem((const void *)split_kern, L::ALLOC) != KVC_OK) return KVC_ECUDA;
    // both passes may start while the previous kernel of the stream finishes; each waits for it on
    // the device before reading what it wrote
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_split, a.n_head_kv);
    cfg.blockDim = dim3((CWARPS + 1) * 32);
    cfg.dynamicSmemBytes = L::ALLOC;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, split_kern, tk, tv, a) != cudaSuccess) return KVC_ECUDA;
    cudaLaunchConfig_t cfg2 = {};
    cfg2.gridDim = dim3(n_head_q);
    cfg2.blockDim = dim3(D);
    cfg2.dynamicSmemBytes = 0;
    cfg2.stream = s;
    cfg2.attrs = attr;
    cfg2.numAttrs = 1;
    CombineBatch<1> cb;
    cb.part[0] = scratch;
    cb.out[0] = out;
    cb.n_split[0] = n_split;
    if (cudaLaunchKernelEx(&cfg2, decode_combine_kernel<D, 1>, cb, a.group, a.n_head_kv) != cudaSuccess)
        return KVC_ECUDA;
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
    }
}

template <int D, bool Q8>
int launch_d(const kvc_cache &c, int layer, int pos, const void *q, int dtype, int n_head_q, float *out,
             float *scratch, cudaStream_t s, const void *k_new = nullptr, const void *v_new = nullptr) {
    switch (dtype) {
        case KVC_IN_F32: return launch_t<D, Q8, KVC_IN_F32>(c, layer, pos, q, n_head_q, out, scratch, s, k_new, v_new);
        case KVC_IN_BF16: return launch_t<D, Q8, KVC_IN_BF16>(c, layer, pos, q, n_head_q, out, scratch, s, k_new, v_new);
        default: return launch_t<D, Q8, KVC_IN_F16>(c, layer, pos, q, n_head_q, out, scratch, s, k_new, v_new);
    }
}

// ---- fixed scratch for decode_attn_noalloc ---------------------------------------------
// Some callers cannot allocate device memory: code hosted inside an engine that
// owns every device allocation, or code on a path where cudaMalloc's implicit
// device synchronisation is not allowed.  For them the split-K partials live in
// this file-scope device array instead of a caller buffer.  Every device that
// loads the library holds it until the process exits; all calls share it.
constexpr size_t NOALLOC_SCRATCH_BYTES = (size_t)8 << 20;  // 8 MiB
static __device__ __align__(256) float g_noalloc_scratch[NOALLOC_SCRATCH_BYTES / sizeof(float)];

// The context the calling thread has current, by its process-unique id (cuCtxGetId, fetched through the
// runtime like the tensor-map encoder, so the library links no libcuda); 0 when there is none yet.
unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext *);
    using GetId = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// The array's device address in the calling thread's current context.  In host code the symbol
// name is only a host-side stand-in, so the address is looked up through cudaGetSymbolAddress
// with the device current, once per context, and cached under the context's id: a context
// created again after a reset of the device (which may place the array elsewhere) has a new id
// and gets a fresh lookup.
int noalloc_scratch_address(float **out) {
    static std::mutex mu;
    static std::map<unsigned long long, float *> addr;   // context id -> address
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = current_context_id();
    if (id != 0) {
        auto it = addr.find(id);
        if (it != addr.end()) {
            *out = it->second;
            return KVC_OK;
        }
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return KVC_ECUDA;
    const unsigned long long id2 = current_context_id();   // the lookup may have made the context current
    if (id2 != 0) addr[id2] = static_cast<float *>(p);
    *out = static_cast<float *>(p);
    return KVC_OK;
}

}  // namespace

int read_and_clear_decode_status(int32_t *status) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_decode_status, sizeof(int)) != cudaSuccess) return KVC_ECUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_decode_status, &zero, sizeof(int)) != cudaSuccess) return KVC_ECUDA;
    *status = v;
    return KVC_OK;
}

size_t decode_noalloc_capacity() { return NOALLOC_SCRATCH_BYTES; }

int launch_decode_noalloc(const kvc_cache &c, int layer, int pos, const void *q, int dtype, int n_head_q,
                          float *out, cudaStream_t s) {
    float *scratch = nullptr;
    const int rc = noalloc_scratch_address(&scratch);
    if (rc != KVC_OK) return rc;
    // every partial the combine pass reads is written by the split pass first: nothing needs clearing
    return launch_decode(c, layer, pos, q, dtype, n_head_q, out, scratch, s);
}

int decode_max_split() { return MAX_SPLIT; }

int decode_max_batch() { return MAX_BATCH; }

namespace {

template <bool Q8, int DT>
int launch_batch_t(const kvc_cache *caches, int n_seq, int layer, const int *pos, const void *q, int n_head_q,
                   float *out, float *scratch, size_t seq_scratch_floats, cudaStream_t s, const void *k = nullptr,
                   const void *v = nullptr) {
    constexpr int D = 128;
    DecodeArgs a[MAX_BATCH];
    memset(a, 0, sizeof(a));
    float *outs[MAX_BATCH];
    const size_t kv_bytes = (size_t)caches[0].d.n_head_kv * D * dtype_bytes(DT);
    const size_t q_bytes = (size_t)n_head_q * D * dtype_bytes(DT);
    for (int i = 0; i < n_seq; ++i) {
        const kvc_cache &c = caches[i];
        a[i].q = static_cast<const uint8_t *>(q) + i * q_bytes;
        a[i].ks = static_cast<const uint16_t *>(c.k_s);
        a[i].vs = static_cast<const uint16_t *>(c.v_s);
        a[i].part = scratch + i * seq_scratch_floats;
        a[i].g = geom_of(c.d);
        a[i].layer = layer;
        a[i].n_keys = pos[i] + 1;
        a[i].n_head_kv = c.d.n_head_kv;
        a[i].group = n_head_q / c.d.n_head_kv;
        a[i].split_len = a[i].n_split = 0;
        a[i].scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)D));
        a[i].stall_ns = 0;
        outs[i] = out + (size_t)i * n_head_q * D;
        if (k != nullptr)
            set_fused(a[i], c, static_cast<const uint8_t *>(k) + i * kv_bytes, static_cast<const uint8_t *>(v) + i * kv_bytes);
    }
    return launch_tc<Q8, DT, MAX_BATCH>(caches, a, n_seq, n_head_q, outs, s);
}

}  // namespace

int launch_decode_batch(const kvc_cache *caches, int n_seq, int layer, const int *pos, const void *q, int dtype,
                        int n_head_q, float *out, float *scratch, size_t seq_scratch_bytes, cudaStream_t s) {
    const kvc_desc &d = caches[0].d;
    const size_t seq_floats = seq_scratch_bytes / sizeof(float);
    if (n_seq == 1 || d.head_dim != 128) {
        // one sequence, or head_dim 64 (its split pass takes one cache per launch): a launch pair per sequence
        const size_t q_bytes = (size_t)n_head_q * d.head_dim * dtype_bytes(dtype);
        for (int i = 0; i < n_seq; ++i) {
            const int rc = launch_decode(caches[i], layer, pos[i], static_cast<const uint8_t *>(q) + i * q_bytes, dtype,
                                         n_head_q, out + (size_t)i * n_head_q * d.head_dim, scratch + i * seq_floats, s);
            if (rc != KVC_OK) return rc;
        }
        return KVC_OK;
    }
    const bool q8 = d.type == KVC_Q8_0;
    switch (dtype) {
        case KVC_IN_F32:
            return q8 ? launch_batch_t<true, KVC_IN_F32>(caches, n_seq, layer, pos, q, n_head_q, out, scratch, seq_floats, s)
                      : launch_batch_t<false, KVC_IN_F32>(caches, n_seq, layer, pos, q, n_head_q, out, scratch, seq_floats, s);
        case KVC_IN_BF16:
            return q8 ? launch_batch_t<true, KVC_IN_BF16>(caches, n_seq, layer, pos, q, n_head_q, out, scratch, seq_floats, s)
                      : launch_batch_t<false, KVC_IN_BF16>(caches, n_seq, layer, pos, q, n_head_q, out, scratch, seq_floats, s);
        default:
            return q8 ? launch_batch_t<true, KVC_IN_F16>(caches, n_seq, layer, pos, q, n_head_q, out, scratch, seq_floats, s)
                      : launch_batch_t<false, KVC_IN_F16>(caches, n_seq, layer, pos, q, n_head_q, out, scratch, seq_floats, s);
    }
}

int launch_decode(const kvc_cache &c, int layer, int pos, const void *q, int dtype, int n_head_q,
                  float *out, float *scratch, cudaStream_t s) {
    const bool q8 = c.d.type == KVC_Q8_0;
    if (c.d.head_dim == 128)
        return q8 ? launch_d<128, true>(c, layer, pos, q, dtype, n_head_q, out, scratch, s)
                  : launch_d<128, false>(c, layer, pos, q, dtype, n_head_q, out, scratch, s);
    return q8 ? launch_d<64, true>(c, layer, pos, q, dtype, n_head_q, out, scratch, s)
              : launch_d<64, false>(c, layer, pos, q, dtype, n_head_q, out, scratch, s);
}

int launch_decode_step(const kvc_cache &c, int layer, int pos, const void *q, const void *k, const void *v, int dtype,
                       int n_head_q, float *out, float *scratch, cudaStream_t s) {
    const bool q8 = c.d.type == KVC_Q8_0;
    if (c.d.head_dim == 128)
        return q8 ? launch_d<128, true>(c, layer, pos, q, dtype, n_head_q, out, scratch, s, k, v)
                  : launch_d<128, false>(c, layer, pos, q, dtype, n_head_q, out, scratch, s, k, v);
    return q8 ? launch_d<64, true>(c, layer, pos, q, dtype, n_head_q, out, scratch, s, k, v)
              : launch_d<64, false>(c, layer, pos, q, dtype, n_head_q, out, scratch, s, k, v);
}

int launch_decode_step_batch(const kvc_cache *caches, int n_seq, int layer, const int *pos, const void *q, const void *k,
                             const void *v, int dtype, int n_head_q, float *out, float *scratch,
                             size_t seq_scratch_bytes, cudaStream_t s) {
    const kvc_desc &d = caches[0].d;
    const size_t seq_floats = seq_scratch_bytes / sizeof(float);
    if (n_seq == 1 || d.head_dim != 128) {
        const size_t q_bytes = (size_t)n_head_q * d.head_dim * dtype_bytes(dtype);
        const size_t kv_bytes = (size_t)d.n_head_kv * d.head_dim * dtype_bytes(dtype);
        for (int i = 0; i < n_seq; ++i) {
            const int rc = launch_decode_step(caches[i], layer, pos[i], static_cast<const uint8_t *>(q) + i * q_bytes,
                                              static_cast<const uint8_t *>(k) + i * kv_bytes,
                                              static_cast<const uint8_t *>(v) + i * kv_bytes, dtype, n_head_q,
                                              out + (size_t)i * n_head_q * d.head_dim, scratch + i * seq_floats, s);
            if (rc != KVC_OK) return rc;
        }
        return KVC_OK;
    }
    const bool q8 = d.type == KVC_Q8_0;
    switch (dtype) {
        case KVC_IN_F32:
            return q8 ? launch_batch_t<true, KVC_IN_F32>(caches, n_seq, layer, pos, q, n_head_q, out, scratch, seq_floats, s, k, v)
                      : launch_batch_t<false, KVC_IN_F32>(caches, n_seq, layer, pos, q, n_head_q, out, scratch, seq_floats, s, k, v);
        case KVC_IN_BF16:
            return q8 ? launch_batch_t<true, KVC_IN_BF16>(caches, n_seq, layer, pos, q, n_head_q, out, scratch, seq_floats, s, k, v)
                      : launch_batch_t<false, KVC_IN_BF16>(caches, n_seq, layer, pos, q, n_head_q, out, scratch, seq_floats, s, k, v);
        default:
            return q8 ? launch_batch_t<true, KVC_IN_F16>(caches, n_seq, layer, pos, q, n_head_q, out, scratch, seq_floats, s, k, v)
                      : launch_batch_t<false, KVC_IN_F16>(caches, n_seq, layer, pos, q, n_head_q, out, scratch, seq_floats, s, k, v);
    }
}

}  // namespace kvc

#ifdef KVC_TRACE
// Diagnostic build only: clear, or copy out (16 x 64 uint64), the split pass's clock stamps.
extern "C" int kvc_trace_clear() {
    static unsigned long long z[16 * 64] = {};
    return cudaMemcpyToSymbol(kvc::g_trace, z, sizeof(z)) == cudaSuccess ? 0 : -1;
}
extern "C" int kvc_trace_read(unsigned long long *host) {
    return cudaMemcpyFromSymbol(host, kvc::g_trace, sizeof(kvc::g_trace)) == cudaSuccess ? 0 : -1;
}
#endif
