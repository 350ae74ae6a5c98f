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
// Split pass: one wave of CTAs, grid (split, kv head), two CTAs per SM.  A CTA
// streams the key range [split*len, (split+1)*len) of one kv head: warp 0
// issues TMA copies of 64-key K and V blocks into a ring of shared-memory
// stages (128-byte swizzle; 64-byte for 64-byte rows), so many stages are in
// flight at once; four consumer warps each take one 16-key group of a stage
// for all G query heads of the group.  A consumer warp computes the group's
// scores with mma.sync m16n8k16 (rows = query heads of the group, columns =
// keys), keeps an online softmax per head, and accumulates P*V with a second
// mma.sync (rows = heads, columns = head_dim), reading its fragments from the
// stage:
//   - q8_0 codes are converted to exact fp16 integers with two byte permutes
//     and one fp16 subtraction; the K scale is applied per 32-value block to
//     the fp32 partial scores, the V scale is folded into P per block, so the
//     only rounding besides fp32 accumulation is fp16(p*d);
//   - f16 values feed the MMAs as stored.
// Head-dim slots are permuted inside each MMA (the dot product does not care)
// so that every thread reads 8 or 16 (K) and 4 or 8 (V) contiguous bytes per
// row.  The four warps are merged in shared memory in a fixed order and the
// CTA writes (m, l, O) for its range to the scratch buffer.
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

namespace kvc {
namespace {

// set by a split pass that gave up a bounded wait (read and cleared with the other kernels' status)
__device__ int g_decode_status;

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
    if constexpr (DT == KVC_IN_F32) return __ldg(static_cast<const float *>(q) + i);
    else {
        const uint16_t u = __ldg(static_cast<const uint16_t *>(q) + i);
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
            const uint2 wk = __ldg(reinterpret_cast<const uint2 *>(a.ks + srow));
            const uint2 wv = __ldg(reinterpret_cast<const uint2 *>(a.vs + srow));
            S.sk[r][0] = wk.x; S.sk[r][1] = wk.y;
            S.sv[r][0] = wv.x; S.sv[r][1] = wv.y;
        } else {
            S.sk[r][0] = __ldg(reinterpret_cast<const uint32_t *>(a.ks + srow));
            S.sv[r][0] = __ldg(reinterpret_cast<const uint32_t *>(a.vs + srow));
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

// One CTA per query head, one thread per output value.  With up to MC splits (one wave of split
// CTAs gives at most 19 per kv head at 8 kv heads) a thread issues every split's (m, l) pair and
// partial value at once, so the pass costs one round trip to L2 and no block barrier; more splits
// take the same steps in rounds of 8.  The weights are ex2(m_i - M) (M the largest split maximum),
// the denominator and the value are summed in split order, so the result is deterministic.
template <int D, int NS>
__global__ void __launch_bounds__(D) decode_combine_kernel(const CombineBatch<NS> cb, int group, int n_head_kv) {
    constexpr int MC = 24;
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
    const float *part_o = part;
    const float *part_ml = part + (int64_t)n_head_kv * MAX_SPLIT * group * D;
    const int64_t p0 = ((int64_t)hkv * MAX_SPLIT) * group + row;   // partial index of split 0
    const float2 *ml_src = reinterpret_cast<const float2 *>(part_ml) + p0;   // split i at + i * group
    const float *o_src = part_o + p0 * D + d;                                 // split i at + i * group * D
    const int64_t o_step = (int64_t)group * D;
    float M = -INFINITY, L = 0.f, acc = 0.f;
    if (n_split <= MC) {
        float2 ml[MC];
        float v[MC];
#pragma unroll
        for (int i = 0; i < MC; ++i) {
            if (i < n_split) {
                ml[i] = __ldcg(ml_src + (int64_t)i * group);
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
        for (int i = 0; i < n_split; ++i) M = fmaxf(M, __ldcg(ml_src + (int64_t)i * group).x);
        for (int i0 = 0; i0 < n_split; i0 += 8) {
            float2 ml[8];
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (i0 + u < n_split) {
                    ml[u] = __ldcg(ml_src + (int64_t)(i0 + u) * group);
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
    out[(int64_t)h * D + d] = acc / L;
}

// ---- tensor-core split pass for head_dim 128 ---------------------------------------------
// Tiles of 128 keys.  S^T = K Q^T with M = 128 keys, N = 16 (the G query heads of the group,
// zero-padded), both operands in shared memory; O^T += V^T P^T with M = 128 head-dim rows, N = 16,
// V as an MN-major operand and P^T written to shared memory by the softmax threads.  Accumulators
// live in tensor memory (S double-buffered), so the warps hold no MMA state.  A chain of dependent
// N = 16 MMAs advances about one step per 220 cycles, while independent chains issued interleaved
// overlap (MMAs of one kind: interleaving S and PV steps costs more than it saves); so S is
// accumulated as two partial sums (head-dim halves) and O^T as two (key halves of each tile), and the
// MMA issuer interleaves the two chains of each.
//   warp 0      TMA producer: K and V tiles (f16) or their int8 codes (q8_0)
//   warp 1      allocates TMEM; one lane issues the MMAs: S(0), S(1), then per tile PV(k), S(k+2)
//   warps 2-5   softmax: thread = key of the tile (TMEM lane); per-head tile maxima are combined
//               across the four warps through shared memory; P^T to shared memory; O^T rescaled
//               (thread = head-dim row) when a running max grows by more than 2^8
//   warps 6-9   (q8_0) dequantise K and V rows into fp16 d*q, separate K and V rings (one thread
//               per key row; NDQ = 256 gives two per row, one per head-dim half)
constexpr int TK = 128;                 // keys per tile
constexpr int NH = 16;                  // MMA N: query heads of a group, padded
// TMEM: S buffer b, half hh at column 32 b + 16 hh; O^T part hh at COL_O + 16 hh
constexpr uint32_t TC_COLS = 128;
constexpr uint32_t COL_O = 64;
constexpr float TC_RESCALE_LOG2 = 8.0f;

template <bool Q8>
struct TCfg {
    static constexpr int D = 128;
    static constexpr int OPT = TK * D * 2;                 // one fp16 K or V tile: 32 KB
    static constexpr int RAWT = 2 * TK * D;                // int8 K and V codes of a tile: 32 KB
    static constexpr int NK = Q8 ? 2 : 3, NV = Q8 ? 2 : 3, NR = Q8 ? 2 : 0;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + NK * OPT;
    static constexpr int OFF_RAW = OFF_V + NV * OPT;
    static constexpr int OFF_QT = OFF_RAW + NR * RAWT;      // Q^T operand: 16 rows x 128, 4 KB
    static constexpr int OFF_PT = OFF_QT + NH * D * 2;      // two P^T operands: 16 rows x 128 keys
    static constexpr int OFF_RED = OFF_PT + 2 * NH * TK * 2;  // [parity][warp][head] floats
    static constexpr int OFF_BAR = OFF_RED + 2 * 4 * NH * 4;
    static constexpr int USED = OFF_BAR + 512;
    static constexpr int ALLOC = USED + 1024;
    static_assert(ALLOC <= 232448, "shared memory plan too large");
    static constexpr int NDQ = 128;                         // dequantising threads (q8_0): 1 or 2 per key
    static constexpr int THREADS = Q8 ? 192 + NDQ : 192;
    static constexpr int CTAS = 1;                          // CTAs per SM
};

enum TcBar {
    T_QREADY, T_SFULL0, T_SFULL1, T_PFULL0, T_PFULL1, T_ODONE0, T_ODONE1, T_XCHG, T_DRAIN, T_STALL,
    T_KFULL, T_KEMPTY = T_KFULL + 4, T_VFULL = T_KEMPTY + 4, T_VEMPTY = T_VFULL + 4, T_RFULL = T_VEMPTY + 4,
    T_REMPTY = T_RFULL + 4, T_NBAR = T_REMPTY + 4
};
static_assert(T_NBAR * 8 + 8 <= 512, "barrier area too small");

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&r)[16]) {
    uint32_t u[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
          "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
        : "r"(taddr));
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __uint_as_float(u[i]);
}
__device__ __forceinline__ void tmem_st16f(uint32_t taddr, const float (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(r[0])), "r"(__float_as_uint(r[1])), "r"(__float_as_uint(r[2])), "r"(__float_as_uint(r[3])),
        "r"(__float_as_uint(r[4])), "r"(__float_as_uint(r[5])), "r"(__float_as_uint(r[6])), "r"(__float_as_uint(r[7])),
        "r"(__float_as_uint(r[8])), "r"(__float_as_uint(r[9])), "r"(__float_as_uint(r[10])), "r"(__float_as_uint(r[11])),
        "r"(__float_as_uint(r[12])), "r"(__float_as_uint(r[13])), "r"(__float_as_uint(r[14])), "r"(__float_as_uint(r[15]))
        : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    umma_f16_ss(d_tmem, a_desc, b_desc, idesc, accumulate);
}
// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled block of 128-byte rows
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
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

// GM: heads the softmax loops cover (8 when the group has at most 8 query heads, else 16)
// NS: sequences of a batch the parameters hold (1, or MAX_BATCH for a batched call; grid z = sequence)
template <bool Q8, int DT, int GM, int NS>
__global__ void __launch_bounds__(TCfg<Q8>::THREADS, TCfg<Q8>::CTAS)
    decode_tc_kernel(const __grid_constant__ TcBatch<NS> b) {
    using L = TCfg<Q8>;
    constexpr int D = 128;
    const int seq = NS == 1 ? 0 : (int)blockIdx.z;
    const DecodeArgs &a = b.a[seq];
    const CUtensorMap *tm_k = &b.tk[seq], *tm_v = &b.tv[seq];
    if ((int)blockIdx.x >= a.n_split) return;   // a batch's shorter sequences use fewer splits
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + T_NBAR);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    float *s_red = reinterpret_cast<float *>(sm + L::OFF_RED);
    const int split = blockIdx.x, hkv = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.group;
    const int j_begin = split * a.split_len;
    const int j_end = min(a.n_keys, j_begin + a.split_len);
    const int T = (j_end - j_begin + TK - 1) / TK;   // tiles of this split

    if (threadIdx.x == 0) {
        *s_abort = 0;
        mbar_init(&bars[T_QREADY], 128);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars[T_SFULL0 + b], 1);
            mbar_init(&bars[T_PFULL0 + b], 128);
            mbar_init(&bars[T_ODONE0 + b], 1);
        }
        mbar_init(&bars[T_XCHG], 128);
        mbar_init(&bars[T_DRAIN], 1);
        mbar_init(&bars[T_STALL], 1);   // nothing arrives here: only the test hook waits on it
        for (int s = 0; s < L::NK; ++s) {
            mbar_init(&bars[T_KFULL + s], Q8 ? L::NDQ : 1);
            mbar_init(&bars[T_KEMPTY + s], 1);
        }
        for (int s = 0; s < L::NV; ++s) {
            mbar_init(&bars[T_VFULL + s], Q8 ? L::NDQ : 1);
            mbar_init(&bars[T_VEMPTY + s], 1);
        }
        if constexpr (Q8) {
            for (int s = 0; s < L::NR; ++s) {
                mbar_init(&bars[T_RFULL + s], 1);
                mbar_init(&bars[T_REMPTY + s], L::NDQ);
            }
        }
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
    // inputs written by the kernels before this one are read only past this point
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            int kn = 0, vn = 0;   // tiles whose K (or raw) and V copies have been issued
            for (int k = 0; k < T; ++k) {
                const int j = j_begin + k * TK;
                if constexpr (Q8) {
                    const int rs = k % L::NR;
                    if (k >= L::NR && !mbar_wait(&bars[T_REMPTY + rs], ((k / L::NR) - 1) & 1, s_abort)) break;
                    uint8_t *dst = sm + L::OFF_RAW + rs * L::RAWT;
                    mbar_arrive_expect_tx(&bars[T_RFULL + rs], L::RAWT);
                    tma_load_3d(dst, tm_k, &bars[T_RFULL + rs], 0, j, hkv);
                    tma_load_3d(dst + TK * D, tm_v, &bars[T_RFULL + rs], 0, j, hkv);
                    ++kn;
                } else {
                    const int ks = k % L::NK, vs = k % L::NV;
                    if (k >= L::NK && !mbar_wait(&bars[T_KEMPTY + ks], ((k / L::NK) - 1) & 1, s_abort)) break;
                    mbar_arrive_expect_tx(&bars[T_KFULL + ks], L::OPT);
                    for (int dh = 0; dh < 2; ++dh)
                        tma_load_3d(sm + L::OFF_K + ks * L::OPT + dh * TK * 128, tm_k, &bars[T_KFULL + ks], dh * 64, j,
                                    hkv);
                    ++kn;
                    if (k >= L::NV && !mbar_wait(&bars[T_VEMPTY + vs], ((k / L::NV) - 1) & 1, s_abort)) break;
                    mbar_arrive_expect_tx(&bars[T_VFULL + vs], L::OPT);
                    for (int dh = 0; dh < 2; ++dh)
                        tma_load_3d(sm + L::OFF_V + vs * L::OPT + dh * TK * 128, tm_v, &bars[T_VFULL + vs], dh * 64, j,
                                    hkv);
                    ++vn;
                }
            }
            if (*s_abort) {
                // after a wait gave up: let the copies still in flight land before the CTA exits
                volatile int never = 0;
                auto drain = [&](int first_bar, int stages, int n) {
                    for (int st = 0; st < stages && st < n; ++st) {
                        const int last = st + ((n - 1 - st) / stages) * stages;
                        mbar_wait(&bars[first_bar + st], (last / stages) & 1, &never, 200000000ull);
                    }
                };
                if constexpr (Q8) {
                    drain(T_RFULL, L::NR, kn);
                } else {
                    drain(T_KFULL, L::NK, kn);
                    drain(T_VFULL, L::NV, vn);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_f16(128, NH, 0, 0);   // A = K (K-major), B = Q (K-major)
            constexpr uint32_t IDESC_O = idesc_f16(128, NH, 1, 0);   // A = V^T (MN-major), B = P^T (K-major)
            const uint32_t sK = smem_u32(sm + L::OFF_K), sV = smem_u32(sm + L::OFF_V);
            const uint32_t sQ = smem_u32(sm + L::OFF_QT), sP = smem_u32(sm + L::OFF_PT);
            bool ok = mbar_wait(&bars[T_QREADY], 0, s_abort);
            tc_fence_after();
            auto wait_k = [&](int j) -> bool {
                if (!mbar_wait(&bars[T_KFULL + j % L::NK], (j / L::NK) & 1, s_abort)) return false;
                tc_fence_after();
                return true;
            };
            // step s (0..3) of both halves of S(j): head-dim k-steps s and 4 + s
            auto s_mma = [&](int j, int s) {
                const uint32_t kb = sK + (j % L::NK) * L::OPT;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int ks = 4 * hh + s;
                    const uint32_t kk = (ks & 3) * 32;
                    umma_ss(tmem + 32 * (j & 1) + 16 * hh, sdesc_sw128(kb + (ks >> 2) * (TK * 128) + kk, 16, 1024),
                            sdesc_sw128(sQ + (ks >> 2) * (NH * 128) + kk, 16, 1024), IDESC_S, s > 0);
                }
            };
            // step s of both key halves of PV(k): key k-steps s and 4 + s
            auto pv_mma = [&](int k, int s) {
                const uint32_t vb = sV + (k % L::NV) * L::OPT, pb = sP + (k & 1) * (NH * TK * 2);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int ks = 4 * hh + s;
                    umma_ss(tmem + COL_O + 16 * hh, sdesc_sw128(vb + ks * 16 * 128, TK * 128, 1024),
                            sdesc_sw128(pb + (ks >> 2) * (NH * 128) + (ks & 3) * 32, 16, 1024), IDESC_O,
                            (k > 0 || s > 0) ? 1u : 0u);
                }
            };
            auto commit_s = [&](int j) {
                umma_commit(&bars[T_SFULL0 + (j & 1)]);
                umma_commit(&bars[T_KEMPTY + j % L::NK]);
            };
            // S(0) and S(1) (S(1) into the other buffer), then per tile PV(k) with S(k + 2)
            for (int j = 0; ok && j < 2 && j < T; ++j) {
                if (!wait_k(j)) { ok = false; break; }
#pragma unroll
                for (int s = 0; s < 4; ++s) s_mma(j, s);
                commit_s(j);
            }
            for (int k = 0; ok && k < T; ++k) {
                // test hook: a bounded wait on a barrier nothing arrives at, in place of the first P
                // wait; it gives up after stall_ns (raising the abort flag) with S MMAs in flight
                if (a.stall_ns != 0 && k == 0) {
                    mbar_wait(&bars[T_STALL], 0, s_abort, a.stall_ns);
                    ok = false;
                    break;
                }
                if (!mbar_wait(&bars[T_PFULL0 + (k & 1)], (k >> 1) & 1, s_abort)) { ok = false; break; }
                const int vs = k % L::NV;
                if (!mbar_wait(&bars[T_VFULL + vs], (k / L::NV) & 1, s_abort)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < 4; ++s) pv_mma(k, s);
                umma_commit(&bars[T_ODONE0 + (k & 1)]);
                umma_commit(&bars[T_VEMPTY + vs]);
                // S(k + 2) reuses S(k)'s buffer, which the softmax read before publishing P(k)
                if (k + 2 < T) {
                    if (!wait_k(k + 2)) { ok = false; break; }
#pragma unroll
                    for (int s = 0; s < 4; ++s) s_mma(k + 2, s);
                    commit_s(k + 2);
                }
            }
            if (*s_abort) {
                // after a wait gave up: let the MMAs in flight finish before TMEM is freed
                volatile int never = 0;
                umma_commit(&bars[T_DRAIN]);
                mbar_wait(&bars[T_DRAIN], 0, &never, 200000000ull);
            }
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------------------ softmax
        const int quarter = warp & 3;
        const int L0 = quarter * 32 + lane;      // TMEM lane: key of the tile / head-dim row of O^T
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        // Q^T operand (rows >= G zero) and both P^T operands cleared (their rows >= G stay zero)
        {
            uint8_t *qt = sm + L::OFF_QT;
            const int h = L0 >> 3, c = L0 & 7;
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    x[e] = h < G ? load_q<DT>(a.q, ((int64_t)hkv * G + h) * D + blk * 64 + c * 8 + e) : 0.f;
                *reinterpret_cast<uint4 *>(qt + blk * (NH * 128) + sw128(h, c)) =
                    make_uint4(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]), pack_half2(x[4], x[5]),
                               pack_half2(x[6], x[7]));
            }
            uint4 *pt = reinterpret_cast<uint4 *>(sm + L::OFF_PT);
#pragma unroll
            for (int i = 0; i < 4; ++i) pt[L0 + 128 * i] = make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
            mbar_arrive(&bars[T_QREADY]);
        }
        float m_run[GM], l_part[GM];
#pragma unroll
        for (int h = 0; h < GM; ++h) {
            m_run[h] = -INFINITY;
            l_part[h] = 0.f;
        }
        uint32_t x_seq = 0;
        int pv_seen[2] = {0, 0};
        bool ok = true;
        auto wait_pv = [&](int j) -> bool {  // PV(j) and every MMA before it have completed
            const int b = j & 1, n = j >> 1;
            if (pv_seen[b] > n) return true;
            if (!mbar_wait(&bars[T_ODONE0 + b], n & 1, s_abort)) return false;
            pv_seen[b] = n + 1;
            tc_fence_after();
            return true;
        };
        const float sl2 = a.scale_log2;
        for (int k = 0; k < T; ++k) {
            if (!mbar_wait(&bars[T_SFULL0 + (k & 1)], (k >> 1) & 1, s_abort)) { ok = false; break; }
            tc_fence_after();
            float sc[NH], sc_hi[NH];
            tmem_ld16(tmem + 32 * (k & 1) + lane_base, sc);
            tmem_ld16(tmem + 32 * (k & 1) + 16 + lane_base, sc_hi);
#pragma unroll
            for (int h = 0; h < NH; ++h) sc[h] += sc_hi[h];
            const bool valid = j_begin + k * TK + L0 < j_end;
            // branch-free over the 16 padded heads: heads >= G score -inf, offset 0, so p = 0 exactly
            float x[GM];
#pragma unroll
            for (int h = 0; h < GM; ++h) x[h] = (valid && h < G) ? sc[h] * sl2 : -INFINITY;
            // per-head maximum over the warp (one warp reduction per head), then over the four warps;
            // the four values of a head are adjacent ([head][warp]) and read as one 16-byte load
            float *slot = s_red + (x_seq & 1) * 4 * NH;
            {
                float v = -INFINITY;
#pragma unroll
                for (int h = 0; h < GM; ++h) {
                    float mx;
                    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(mx) : "f"(x[h]));
                    v = lane == h ? mx : v;
                }
                if (lane < GM) slot[lane * 4 + quarter] = v;
            }
            mbar_arrive(&bars[T_XCHG]);
            if (!mbar_wait(&bars[T_XCHG], x_seq & 1, s_abort)) { ok = false; break; }
            ++x_seq;
            bool rescale = false;
            float alpha[GM];
#pragma unroll
            for (int h = 0; h < GM; ++h) {
                const float4 w4 = *reinterpret_cast<const float4 *>(slot + 4 * h);
                const float M = fmaxf(fmaxf(w4.x, w4.y), fmaxf(w4.z, w4.w));
                // the split's first key is visible, so M is finite on the first tile for heads < G
                const bool grow = k > 0 && M > m_run[h] + TC_RESCALE_LOG2;
                alpha[h] = grow ? ex2(m_run[h] - M) : 1.f;
                m_run[h] = (k == 0 || grow) ? M : m_run[h];
                rescale |= grow;
            }
            float p[GM];
#pragma unroll
            for (int h = 0; h < GM; ++h) {
                const float m_sub = m_run[h] == -INFINITY ? 0.f : m_run[h];
                p[h] = ex2(x[h] - m_sub);
                l_part[h] = l_part[h] * alpha[h] + p[h];
            }
            // P^T buffer k & 1 was last read by PV(k - 2); O^T must hold PV(k - 1) before a rescale
            if (k >= 2 && !wait_pv(k - 2)) { ok = false; break; }
            if (rescale && k >= 1) {
                if (!wait_pv(k - 1)) { ok = false; break; }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float o[NH];
                    tmem_ld16(tmem + COL_O + 16 * hh + lane_base, o);
#pragma unroll
                    for (int h = 0; h < GM; ++h) o[h] *= alpha[h];
                    tmem_st16f(tmem + COL_O + 16 * hh + lane_base, o);
                }
                tmem_st_wait();
            }
            uint8_t *pt = sm + L::OFF_PT + (k & 1) * (NH * TK * 2) + (L0 >> 6) * (NH * 128);
            const int kc = (L0 & 63) >> 3, kb = (L0 & 7) * 2;
#pragma unroll
            for (int h = 0; h < GM; ++h)
                if (h < G) *reinterpret_cast<__half *>(pt + sw128(h, kc) + kb) = __float2half_rn(p[h]);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars[T_PFULL0 + (k & 1)]);
        }
        // ---- epilogue: this split's (m, l, O) per head of the group
        bool wrote = false;
        if (ok && T > 0 && wait_pv(T - 1)) {
            float o[NH], o_hi[NH];
            tmem_ld16(tmem + COL_O + lane_base, o);
            tmem_ld16(tmem + COL_O + 16 + lane_base, o_hi);
#pragma unroll
            for (int h = 0; h < NH; ++h) o[h] += o_hi[h];
            // row sums: over the warp (fixed tree), then the four warps in order
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int h = 0; h < GM; ++h) l_part[h] += __shfl_xor_sync(0xffffffffu, l_part[h], off);
            float *slot = s_red + (x_seq & 1) * 4 * NH;
            if (lane < GM) {
                float v = l_part[0];
#pragma unroll
                for (int h = 1; h < GM; ++h) v = lane == h ? l_part[h] : v;
                slot[lane * 4 + quarter] = v;
            }
            mbar_arrive(&bars[T_XCHG]);
            if (mbar_wait(&bars[T_XCHG], x_seq & 1, s_abort)) {
                ++x_seq;
                const int64_t pbase = ((int64_t)hkv * MAX_SPLIT + split) * G;
                float *part_o = a.part;
                float *part_ml = a.part + (int64_t)a.n_head_kv * MAX_SPLIT * G * D;
#pragma unroll
                for (int h = 0; h < GM; ++h)
                    if (h < G) part_o[(pbase + h) * D + L0] = o[h];
                if (L0 < G) {
                    float mv = m_run[0];
#pragma unroll
                    for (int h = 1; h < GM; ++h) mv = L0 == h ? m_run[h] : mv;
                    const float4 w4 = *reinterpret_cast<const float4 *>(slot + 4 * L0);
                    part_ml[(pbase + L0) * 2] = mv;
                    part_ml[(pbase + L0) * 2 + 1] = ((w4.x + w4.y) + w4.z) + w4.w;
                }
                wrote = true;
            }
        }
        if (!wrote && L0 < G) {
            // a split that gave up leaves an empty partial (m = -inf, l = 0), which the combine
            // weighs 0, rather than another call's leftovers
            float *part_ml = a.part + (int64_t)a.n_head_kv * MAX_SPLIT * G * D;
            const int64_t pi = ((int64_t)hkv * MAX_SPLIT + split) * G + L0;
            part_ml[pi * 2] = -INFINITY;
            part_ml[pi * 2 + 1] = 0.f;
        }
    } else if constexpr (Q8) {
        // ------------------------------------------------------------------ dequantise (q8_0)
        constexpr int HPT = 256 / L::NDQ;               // head-dim halves per thread
        const int dt = threadIdx.x - 192;
        const int r = dt & (TK - 1), hd0 = dt / TK;   // key row of the tile, first head-dim half
        constexpr int NB = D / 32;
        bool ok = true;
        uint32_t sk_n[HPT], sv_n[HPT];
        // the fp16 scales of blocks 2 hd and 2 hd + 1 of my key's K and V rows, for my halves hd
        auto scales = [&](int k, uint32_t (&sk)[HPT], uint32_t (&sv)[HPT]) {
            const int key = min(j_begin + k * TK + r, a.n_keys - 1);  // keys past the end: any finite scale
            const int64_t srow = a.layer * a.g.s_layer + hkv * a.g.s_head + (int64_t)key * a.g.s_tok;
#pragma unroll
            for (int hh = 0; hh < HPT; ++hh) {
                sk[hh] = __ldg(reinterpret_cast<const uint32_t *>(a.ks + srow) + hd0 + hh);
                sv[hh] = __ldg(reinterpret_cast<const uint32_t *>(a.vs + srow) + hd0 + hh);
            }
        };
        if (T > 0) scales(0, sk_n, sv_n);
        for (int k = 0; ok && k < T; ++k) {
            uint32_t sk[HPT], sv[HPT];
#pragma unroll
            for (int hh = 0; hh < HPT; ++hh) {
                sk[hh] = sk_n[hh];
                sv[hh] = sv_n[hh];
            }
            if (k + 1 < T) scales(k + 1, sk_n, sv_n);
            const int rs = k % L::NR;
            if (!mbar_wait(&bars[T_RFULL + rs], (k / L::NR) & 1, s_abort)) { ok = false; break; }
            const uint8_t *raw = sm + L::OFF_RAW + rs * L::RAWT;
#pragma unroll 1
            for (int kv = 0; kv < 2; ++kv) {
                const int s = k % (kv ? L::NV : L::NK);
                const int n = kv ? L::NV : L::NK;
                if (k >= n && !mbar_wait(&bars[(kv ? T_VEMPTY : T_KEMPTY) + s], ((k / n) - 1) & 1, s_abort)) {
                    ok = false;
                    break;
                }
                const uint8_t *src = raw + kv * (TK * D);
                uint8_t *dst = sm + (kv ? L::OFF_V : L::OFF_K) + s * L::OPT;
#pragma unroll
                for (int hh = 0; hh < HPT; ++hh) {
                const int hd = hd0 + hh;
                const uint32_t sw = kv ? sv[hh] : sk[hh];
                // my half row: 16-byte code chunks 4 hd .. 4 hd + 3 (two 32-value blocks)
                uint4 q[D / 32];
#pragma unroll
                for (int i = 0; i < D / 32; ++i) q[i] = *reinterpret_cast<const uint4 *>(src + sw128(r, 4 * hd + i));
#pragma unroll
                for (int i = 0; i < D / 32; ++i) {
                    const int c = 4 * hd + i;
                    const unsigned short sb = (unsigned short)(sw >> (16 * (i >> 1)));
                    const __half2 d2 = __halves2half2(__ushort_as_half(sb), __ushort_as_half(sb));
                    uint32_t o[8];
                    dequant4(q[i].x, d2, o[0], o[1]);
                    dequant4(q[i].y, d2, o[2], o[3]);
                    dequant4(q[i].z, d2, o[4], o[5]);
                    dequant4(q[i].w, d2, o[6], o[7]);
                    // fp16 chunk 2c and 2c + 1 of the row: column block (2c) / 8, chunk (2c) % 8 inside it
                    *reinterpret_cast<uint4 *>(dst + (c >> 2) * (TK * 128) + sw128(r, (2 * c) & 7)) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4 *>(dst + (c >> 2) * (TK * 128) + sw128(r, (2 * c + 1) & 7)) =
                        make_uint4(o[4], o[5], o[6], o[7]);
                }
                }
                // order the operand writes before the MMA (async proxy) reads them
                fence_proxy_async_smem();
                mbar_arrive(&bars[(kv ? T_VFULL : T_KFULL) + s]);
            }
            if (!ok) break;
            // the raw stage's generic reads are ordered by the fence above before its TMA refill
            mbar_arrive(&bars[T_REMPTY + rs]);
        }
        (void)NB;
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *s_abort) atomicExch(&g_decode_status, 1);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TC_COLS);
    }
}

// The tensor-core split pass and the combine, one launch each, over n_seq sequences (NS = 1, or
// MAX_BATCH for a batched call).  Sequence i: cache caches[i], arguments a0[i] (its q and its scratch
// as part), output outs[i].  The sequences share the SMs evenly: one wave over (split, kv head,
// sequence), whole tiles per split.
template <bool Q8, int DT, int NS>
int launch_tc(const kvc_cache *caches, const DecodeArgs *a0, int n_seq, int n_head_q, float *const *outs,
              cudaStream_t s) {
    using L = TCfg<Q8>;
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
        if (!make_map_3d(&b.tk[i], dt, kb + (int64_t)eb * a.layer * g.c_layer, D, a.n_keys, a.n_head_kv,
                         eb * g.c_tok, eb * g.c_head, box0, TK, 1, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map_3d(&b.tv[i], dt, vb + (int64_t)eb * a.layer * g.c_layer, D, a.n_keys, a.n_head_kv,
                         eb * g.c_tok, eb * g.c_head, box0, TK, 1, CU_TENSOR_MAP_SWIZZLE_128B))
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
    auto kern = group <= 8 ? decode_tc_kernel<Q8, DT, 8, NS> : decode_tc_kernel<Q8, DT, 16, NS>;
    if (allow_dynamic_smem((const void *)kern, L::ALLOC) != KVC_OK) return KVC_ECUDA;
    // both passes may start while the previous kernel of the stream finishes; each waits for it on
    // the device before reading what it wrote
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(max_split, n_head_kv, n_seq);
    cfg.blockDim = dim3(L::THREADS);
    cfg.dynamicSmemBytes = L::ALLOC;
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

template <int D, bool Q8, int DT>
int launch_t(const kvc_cache &c, int layer, int pos, const void *q, int n_head_q, float *out,
             float *scratch, cudaStream_t s) {
    using L = DCfg<D, Q8>;
    DecodeArgs a;
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
             float *scratch, cudaStream_t s) {
    switch (dtype) {
        case KVC_IN_F32: return launch_t<D, Q8, KVC_IN_F32>(c, layer, pos, q, n_head_q, out, scratch, s);
        case KVC_IN_BF16: return launch_t<D, Q8, KVC_IN_BF16>(c, layer, pos, q, n_head_q, out, scratch, s);
        default: return launch_t<D, Q8, KVC_IN_F16>(c, layer, pos, q, n_head_q, out, scratch, s);
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
                   float *out, float *scratch, size_t seq_scratch_floats, cudaStream_t s) {
    constexpr int D = 128;
    DecodeArgs a[MAX_BATCH];
    float *outs[MAX_BATCH];
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

}  // namespace kvc
