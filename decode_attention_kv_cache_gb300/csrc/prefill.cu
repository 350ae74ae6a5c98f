// Prefill attention for one chunk of query rows over the KV cache, on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// What it computes: for each query row t of the chunk [pos0, pos0 + C) and
// query head h, softmax over keys j <= t of q.khat_j / sqrt(D), applied to
// vhat_j, with kv head h / G (grouped-query attention) - the flash attention
// the pages run over the cache while a prompt is processed in ubatches
// (llama.cpp PR #17 "--split-overlap", section "Results": "native FA";
// llama.cpp PR #58 "completion : allow the prompt to be processed under its
// own split mode", section "Why").
//
// Design (one CTA = 128 query rows of one query head; key tiles of 128 at
// absolute positions 0, 128, 256, ...):
//   warp 0      TMA producer: the Q tile once, then the K/V tiles (int8 codes
//               for q8_0, fp16 values for f16) into shared memory.
//   warp 1      allocates 512 TMEM columns; one lane issues the MMAs:
//               S = Q K^T (M=128, N=128, fp16 x fp16 -> fp32 in TMEM), and
//               O += P V (M=128, N=D, V as an MN-major operand).
//   warps 4-7   softmax: thread r owns query row r (TMEM lane r); reads its S
//               row from TMEM, applies the causal mask, keeps a running max
//               and sum, writes P (fp16) to shared memory for the PV MMA, and
//               in the end divides O by the sum and stores it (fp32).
//   warps 8-11  (q8_0 only) dequantise the int8 K/V tile: thread r converts key
//               row r to fp16 d*q in the 128-byte-swizzled operand layout.
// The running max is re-based only when it grows by more than 2^8, so most
// tiles need no O rescale; the decision is per row, so results stay exact
// per row and independent of the chunking.
//
// Operand type: fp16 for Q, K, V and P (the same tensor rate as bf16): int8
// codes are exact in fp16, d*q rounds once to 11 bits, and the f16 cache
// feeds the MMA as stored.
//
// Every mbarrier wait is bounded (2 s wall clock); a wait that gives up sets a
// device status word and the CTA skips the rest of its work, frees its TMEM
// and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {

__device__ int g_device_status;

namespace {

using namespace ptx;

constexpr int BM = 128;           // query rows per CTA
constexpr int BN = 128;           // keys per tile
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.0f;

enum Bar {
    B_QFULL, B_QREADY, B_RAWFULL, B_RAWEMPTY, B_KVFULL0, B_KVFULL1, B_KVEMPTY0, B_KVEMPTY1,
    B_SFULL0, B_SFULL1, B_PFULL, B_ODONE, NBAR
};

template <int D, bool Q8>
struct Layout {
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2;    // one fp16 K or V stage
    static constexpr int P_BYTES = BM * BN * 2;
    static constexpr int RAW_BYTES = Q8 ? BN * D : 0;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;
    static constexpr int OFF_P = OFF_V + 2 * KV_BYTES;
    static constexpr int OFF_RAWK = OFF_P + P_BYTES;
    static constexpr int OFF_RAWV = OFF_RAWK + RAW_BYTES;
    static constexpr int OFF_BAR = OFF_RAWV + RAW_BYTES;
    static constexpr int USED = OFF_BAR + 256;
    // at least ~120 KB so that one CTA runs per SM (it allocates all 512 TMEM columns)
    static constexpr int ALLOC = (USED + 1024 > 122880) ? USED + 1024 : 122880;
    static constexpr int THREADS = Q8 ? 384 : 256;
};

struct Args {
    const float *q_f32;
    const uint16_t *ks;
    const uint16_t *vs;
    float *out;
    Geom g;
    int layer, pos0, n_rows, kv_len, n_head_q, group, n_qtiles;
    float scale_log2;
};

// Byte offset of 16-byte chunk `c` (0..7) of row `row` in a 128-byte-swizzled
// tile whose 8-row atoms are 1024 bytes.
__device__ __forceinline__ uint32_t sw128(int row, int c) {
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4));
}
// Same for a 64-byte-swizzled tile of 64-byte rows.
__device__ __forceinline__ uint32_t sw64(int row, int c) {
    return (uint32_t)(row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
}
// Chunk `cc` (8 halves) of row `row` in an fp16 operand tile of `rows` rows:
// 64-half column blocks of rows*128 bytes each, 128-byte swizzle inside.
__device__ __forceinline__ uint32_t op_off(int rows, int row, int cc) {
    return (uint32_t)((cc >> 3) * rows * 128) + sw128(row, cc & 7);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    return (uint32_t)__half_as_ushort(__float2half_rn(lo)) |
           ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}

// 4 int8 codes (one 32-bit word) times the fp16 scale, as two fp16x2 words.
__device__ __forceinline__ void dequant4(uint32_t w, __half2 d2, uint32_t &lo, uint32_t &hi) {
    // (byte ^ 0x80) in the low 8 bits of an fp16 with exponent bits 0x64 is 1024 + q + 128 exactly
    const uint32_t a = (__byte_perm(w, 0, 0x0100) & 0x00FF00FFu) ^ 0x64806480u;
    const uint32_t b = (__byte_perm(w, 0, 0x0302) & 0x00FF00FFu) ^ 0x64806480u;
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    __half2 qa = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);  // exact integers
    __half2 qb = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
    __half2 ra = __hmul2(qa, d2);  // one rounding: fp16(d * q)
    __half2 rb = __hmul2(qb, d2);
    lo = *reinterpret_cast<uint32_t *>(&ra);
    hi = *reinterpret_cast<uint32_t *>(&rb);
}

template <int D, bool Q8, int QDT>
__global__ void __launch_bounds__(Layout<D, Q8>::THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const Args a) {
    using L = Layout<D, Q8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + NBAR);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qtile = a.n_qtiles - 1 - (int)blockIdx.x;  // the longest key ranges start first
    const int h = blockIdx.y, hkv = h / a.group;
    const int r0 = qtile * BM;
    const int rows = min(BM, a.n_rows - r0);
    const int t_first = a.pos0 + r0;
    const int t_last = t_first + rows - 1;
    const int n_tiles = t_last / BN + 1;

    if (threadIdx.x == 0) {
        *s_abort = 0;
        mbar_init(&bars[B_QFULL], 1);
        mbar_init(&bars[B_QREADY], 128);
        mbar_init(&bars[B_RAWFULL], 1);
        mbar_init(&bars[B_RAWEMPTY], 128);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[B_KVFULL0 + s], Q8 ? 128 : 1);
            mbar_init(&bars[B_KVEMPTY0 + s], 1);
            mbar_init(&bars[B_SFULL0 + s], 1);
        }
        mbar_init(&bars[B_PFULL], 128);
        mbar_init(&bars[B_ODONE], 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t TM_S0 = tmem, TM_O = tmem + 256;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            if (QDT != KVC_IN_F32) {
                mbar_arrive_expect_tx(&bars[B_QFULL], BM * D * 2);
                for (int dh = 0; dh < D / 64; ++dh)
                    tma_load_3d(sm + L::OFF_Q + dh * BM * 128, &tm_q, &bars[B_QFULL], dh * 64, h, r0);
            }
            for (int j = 0; j < n_tiles; ++j) {
                if (Q8) {
                    if (j > 0 && !mbar_wait(&bars[B_RAWEMPTY], (j - 1) & 1, s_abort)) break;
                    mbar_arrive_expect_tx(&bars[B_RAWFULL], 2 * BN * D);
                    tma_load_3d(sm + L::OFF_RAWK, &tm_k, &bars[B_RAWFULL], 0, j * BN, hkv);
                    tma_load_3d(sm + L::OFF_RAWV, &tm_v, &bars[B_RAWFULL], 0, j * BN, hkv);
                } else {
                    const int st = j & 1;
                    if (j >= 2 && !mbar_wait(&bars[B_KVEMPTY0 + st], ((j >> 1) - 1) & 1, s_abort)) break;
                    mbar_arrive_expect_tx(&bars[B_KVFULL0 + st], 2 * BN * D * 2);
                    for (int dh = 0; dh < D / 64; ++dh) {
                        tma_load_3d(sm + L::OFF_K + st * L::KV_BYTES + dh * BN * 128, &tm_k,
                                    &bars[B_KVFULL0 + st], dh * 64, j * BN, hkv);
                        tma_load_3d(sm + L::OFF_V + st * L::KV_BYTES + dh * BN * 128, &tm_v,
                                    &bars[B_KVFULL0 + st], dh * 64, j * BN, hkv);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_f16(BM, BN, 0, 0);
            constexpr uint32_t IDESC_O = idesc_f16(BM, D, 0, 1);
            const uint32_t sQ = smem_u32(sm + L::OFF_Q), sK = smem_u32(sm + L::OFF_K);
            const uint32_t sV = smem_u32(sm + L::OFF_V), sP = smem_u32(sm + L::OFF_P);
            auto issue_s = [&](int st) {
                const uint32_t kb = sK + st * L::KV_BYTES;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * (BM * 128) + (ks & 3) * 32;
                    umma_f16_ss(TM_S0 + st * BN, sdesc_sw128(sQ + off, 16, 1024),
                                sdesc_sw128(kb + off, 16, 1024), IDESC_S, ks > 0);
                }
            };
            auto issue_o = [&](int st, bool acc) {
                const uint32_t vb = sV + st * L::KV_BYTES;
#pragma unroll
                for (int ks = 0; ks < BN / 16; ++ks) {
                    const uint64_t ad = sdesc_sw128(sP + (ks >> 2) * (BM * 128) + (ks & 3) * 32, 16, 1024);
                    // V tile [key][d]: MN-major; next 64 d's at +BN*128 bytes, next 8 keys at +1024
                    const uint64_t bd = sdesc_sw128(vb + ks * 16 * 128, BN * 128, 1024);
                    umma_f16_ss(TM_O, ad, bd, IDESC_O, (acc || ks > 0) ? 1u : 0u);
                }
            };
            bool ok = mbar_wait(&bars[B_QREADY], 0, s_abort) && mbar_wait(&bars[B_KVFULL0], 0, s_abort);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                umma_commit(&bars[B_SFULL0]);
                for (int j = 0; j < n_tiles; ++j) {
                    if (j + 1 < n_tiles) {
                        const int st = (j + 1) & 1;
                        if (!mbar_wait(&bars[B_KVFULL0 + st], ((j + 1) >> 1) & 1, s_abort)) break;
                        tc_fence_after();
                        issue_s(st);
                        umma_commit(&bars[B_SFULL0 + st]);
                    }
                    if (!mbar_wait(&bars[B_PFULL], j & 1, s_abort)) break;
                    tc_fence_after();
                    issue_o(j & 1, j > 0);
                    umma_commit(&bars[B_KVEMPTY0 + (j & 1)]);
                    umma_commit(&bars[B_ODONE]);
                }
            }
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        // ---------------------------------------------------------------- softmax
        const int r = threadIdx.x - 128;                 // query row in the tile = TMEM lane
        const int t = t_first + r;                       // its absolute position
        const bool valid = r < rows;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        uint8_t *sQp = sm + L::OFF_Q;
        bool ok = true;
        if (QDT == KVC_IN_F32) {
            const float *src = a.q_f32 + ((int64_t)(r0 + r) * a.n_head_q + h) * D;
#pragma unroll 1
            for (int cc = 0; cc < D / 8; ++cc) {
                float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
                if (valid) {
                    x0 = __ldg(reinterpret_cast<const float4 *>(src + cc * 8));
                    x1 = __ldg(reinterpret_cast<const float4 *>(src + cc * 8 + 4));
                }
                uint4 o = make_uint4(pack_half2(x0.x, x0.y), pack_half2(x0.z, x0.w),
                                     pack_half2(x1.x, x1.y), pack_half2(x1.z, x1.w));
                *reinterpret_cast<uint4 *>(sQp + op_off(BM, r, cc)) = o;
            }
        } else {
            ok = mbar_wait(&bars[B_QFULL], 0, s_abort);
            if (ok && QDT == KVC_IN_BF16) {
#pragma unroll 1
                for (int cc = 0; cc < D / 8; ++cc) {
                    uint4 *p = reinterpret_cast<uint4 *>(sQp + op_off(BM, r, cc));
                    uint4 v = *p;
                    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        w[i] = pack_half2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
                    *p = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars[B_QREADY]);

        float m_ref = -INFINITY, l = 0.f;
        const float sl2 = a.scale_log2;
        uint8_t *sPp = sm + L::OFF_P;
#pragma unroll 1
        for (int j = 0; ok && j < n_tiles; ++j) {
            const int st = j & 1;
            if (!mbar_wait(&bars[B_SFULL0 + st], (j >> 1) & 1, s_abort)) { ok = false; break; }
            tc_fence_after();
            const uint32_t s_addr = TM_S0 + st * BN + lane_base;
            const int key0 = j * BN;
            const bool need_mask = key0 + BN - 1 > t_first;
            // pass 1: row max of the scaled, masked scores
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t s[32];
                tmem_ld32(s_addr + c * 32, s);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float x = __uint_as_float(s[i]) * sl2;
                    if (need_mask && key0 + c * 32 + i > t) x = -INFINITY;
                    mx = fmaxf(mx, x);
                }
            }
            const float m_new = fmaxf(m_ref, mx);
            float m_use = m_ref, alpha = 1.f;
            if (j == 0) {
                m_use = m_new;  // key 0 is visible to every row, so m_new is finite
            } else if (m_new > m_ref + RESCALE_LOG2) {
                m_use = m_new;
                alpha = ex2(m_ref - m_new);
            }
            // pass 2: probabilities (fp16) and their sum
            uint32_t pk[BN / 2];
            float rs = 0.f;
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t s[32];
                tmem_ld32(s_addr + c * 32, s);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float x0 = __uint_as_float(s[i]) * sl2, x1 = __uint_as_float(s[i + 1]) * sl2;
                    if (need_mask && key0 + c * 32 + i > t) x0 = -INFINITY;
                    if (need_mask && key0 + c * 32 + i + 1 > t) x1 = -INFINITY;
                    const float p0 = ex2(x0 - m_use), p1 = ex2(x1 - m_use);
                    rs += p0 + p1;
                    pk[c * 16 + i / 2] = pack_half2(p0, p1);
                }
            }
            l = l * alpha + rs;
            if (j > 0) {
                // the PV MMA of the previous tile must be done: O is rescaled and P rewritten
                if (!mbar_wait(&bars[B_ODONE], (j - 1) & 1, s_abort)) { ok = false; break; }
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(TM_O + lane_base + c * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(TM_O + lane_base + c * 32, o);
                    }
                    tmem_st_wait();
                }
            }
#pragma unroll
            for (int cc = 0; cc < BN / 8; ++cc)
                *reinterpret_cast<uint4 *>(sPp + op_off(BM, r, cc)) =
                    make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bars[B_PFULL]);
            m_ref = m_use;
        }
        if (ok && mbar_wait(&bars[B_ODONE], (n_tiles - 1) & 1, s_abort)) {
            tc_fence_after();
            const float inv = 1.f / l;
            float *dst = a.out + ((int64_t)(r0 + r) * a.n_head_q + h) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(TM_O + lane_base + c * 32, o);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4 *>(dst + c * 32 + i) =
                            make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv,
                                        __uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
                }
            }
        }
    } else if (Q8 && warp >= 8) {
        // ---------------------------------------------------------------- dequantise
        const int r = threadIdx.x - 256;  // key row in the tile
        constexpr int NB = D / 32;
        const uint8_t *rawk = sm + L::OFF_RAWK, *rawv = sm + L::OFF_RAWV;
#pragma unroll 1
        for (int j = 0; j < n_tiles; ++j) {
            const int key = j * BN + r;
            uint16_t sk[NB], sv[NB];
            const int64_t soff = a.layer * a.g.s_layer + (int64_t)key * a.g.s_tok + hkv * a.g.s_head;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                sk[b] = key < a.kv_len ? __ldg(a.ks + soff + b) : (uint16_t)0;
                sv[b] = key < a.kv_len ? __ldg(a.vs + soff + b) : (uint16_t)0;
            }
            if (!mbar_wait(&bars[B_RAWFULL], j & 1, s_abort)) break;
            uint4 rk[D / 16], rv[D / 16];
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
                const uint32_t off = (D == 128) ? sw128(r, c) : sw64(r, c);
                rk[c] = *reinterpret_cast<const uint4 *>(rawk + off);
                rv[c] = *reinterpret_cast<const uint4 *>(rawv + off);
            }
            mbar_arrive(&bars[B_RAWEMPTY]);
            const int st = j & 1;
            if (j >= 2 && !mbar_wait(&bars[B_KVEMPTY0 + st], ((j >> 1) - 1) & 1, s_abort)) break;
            uint8_t *dk = sm + L::OFF_K + st * L::KV_BYTES;
            uint8_t *dv = sm + L::OFF_V + st * L::KV_BYTES;
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
                const __half2 k2 = __halves2half2(__ushort_as_half(sk[c >> 1]), __ushort_as_half(sk[c >> 1]));
                const __half2 v2 = __halves2half2(__ushort_as_half(sv[c >> 1]), __ushort_as_half(sv[c >> 1]));
                uint32_t ko[8], vo[8];
                dequant4(rk[c].x, k2, ko[0], ko[1]);
                dequant4(rk[c].y, k2, ko[2], ko[3]);
                dequant4(rk[c].z, k2, ko[4], ko[5]);
                dequant4(rk[c].w, k2, ko[6], ko[7]);
                dequant4(rv[c].x, v2, vo[0], vo[1]);
                dequant4(rv[c].y, v2, vo[2], vo[3]);
                dequant4(rv[c].z, v2, vo[4], vo[5]);
                dequant4(rv[c].w, v2, vo[6], vo[7]);
                *reinterpret_cast<uint4 *>(dk + op_off(BN, r, 2 * c)) = make_uint4(ko[0], ko[1], ko[2], ko[3]);
                *reinterpret_cast<uint4 *>(dk + op_off(BN, r, 2 * c + 1)) = make_uint4(ko[4], ko[5], ko[6], ko[7]);
                *reinterpret_cast<uint4 *>(dv + op_off(BN, r, 2 * c)) = make_uint4(vo[0], vo[1], vo[2], vo[3]);
                *reinterpret_cast<uint4 *>(dv + op_off(BN, r, 2 * c + 1)) = make_uint4(vo[4], vo[5], vo[6], vo[7]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars[B_KVFULL0 + st]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *s_abort) atomicExch(&g_device_status, 1);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---- host side ----------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool make_map_3d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t d0, uint64_t d1,
                 uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1,
                 uint32_t b2, CUtensorMapSwizzle sw) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool Q8, int QDT>
int launch_t(const kvc_cache &c, int layer, int pos0, int n, const void *q, int n_head_q, float *out,
             cudaStream_t s) {
    using L = Layout<D, Q8>;
    const Geom g = geom_of(c.d);
    const int H = c.d.n_head_kv, kv_len = pos0 + n;
    CUtensorMap tq, tk, tv;
    const uint8_t *kb = static_cast<const uint8_t *>(c.k_q), *vb = static_cast<const uint8_t *>(c.v_q);
    bool ok;
    if (Q8) {
        const CUtensorMapSwizzle sw = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
        ok = make_map_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, kb + layer * g.c_layer, D, kv_len, H, g.c_tok,
                         g.c_head, D, BN, 1, sw) &&
             make_map_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, vb + layer * g.c_layer, D, kv_len, H, g.c_tok,
                         g.c_head, D, BN, 1, sw);
    } else {
        ok = make_map_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, kb + 2 * layer * g.c_layer, D, kv_len, H,
                         2 * g.c_tok, 2 * g.c_head, 64, BN, 1, CU_TENSOR_MAP_SWIZZLE_128B) &&
             make_map_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, vb + 2 * layer * g.c_layer, D, kv_len, H,
                         2 * g.c_tok, 2 * g.c_head, 64, BN, 1, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (!ok) return KVC_ECUDA;
    if (QDT != KVC_IN_F32) {
        const CUtensorMapDataType dt =
            QDT == KVC_IN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        if (!make_map_3d(&tq, dt, q, D, n_head_q, n, (uint64_t)D * 2, (uint64_t)n_head_q * D * 2, 64, 1, BM,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return KVC_ECUDA;
    } else {
        tq = tk;  // unused by the f32 variant
    }
    Args a;
    a.q_f32 = QDT == KVC_IN_F32 ? static_cast<const float *>(q) : nullptr;
    a.ks = static_cast<const uint16_t *>(c.k_s);
    a.vs = static_cast<const uint16_t *>(c.v_s);
    a.out = out;
    a.g = g;
    a.layer = layer;
    a.pos0 = pos0;
    a.n_rows = n;
    a.kv_len = kv_len;
    a.n_head_q = n_head_q;
    a.group = n_head_q / H;
    a.n_qtiles = (n + BM - 1) / BM;
    a.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)D));
    auto kern = prefill_kernel<D, Q8, QDT>;
    static bool attr_set = false;  // per instantiation
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC) != cudaSuccess)
            return KVC_ECUDA;
        attr_set = true;
    }
    dim3 grid(a.n_qtiles, n_head_q);
    kern<<<grid, L::THREADS, L::ALLOC, s>>>(tq, tk, tv, a);
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
}

template <int D, bool Q8>
int launch_d(const kvc_cache &c, int layer, int pos0, int n, const void *q, int dtype, int n_head_q,
             float *out, cudaStream_t s) {
    switch (dtype) {
        case KVC_IN_F32: return launch_t<D, Q8, KVC_IN_F32>(c, layer, pos0, n, q, n_head_q, out, s);
        case KVC_IN_BF16: return launch_t<D, Q8, KVC_IN_BF16>(c, layer, pos0, n, q, n_head_q, out, s);
        default: return launch_t<D, Q8, KVC_IN_F16>(c, layer, pos0, n, q, n_head_q, out, s);
    }
}

}  // namespace

int launch_prefill(const kvc_cache &c, int layer, int pos0, int n_tokens, const void *q, int dtype,
                   int n_head_q, float *out, cudaStream_t s) {
    if (n_tokens == 0) return KVC_OK;
    const bool q8 = c.d.type == KVC_Q8_0;
    if (c.d.head_dim == 128)
        return q8 ? launch_d<128, true>(c, layer, pos0, n_tokens, q, dtype, n_head_q, out, s)
                  : launch_d<128, false>(c, layer, pos0, n_tokens, q, dtype, n_head_q, out, s);
    return q8 ? launch_d<64, true>(c, layer, pos0, n_tokens, q, dtype, n_head_q, out, s)
              : launch_d<64, false>(c, layer, pos0, n_tokens, q, dtype, n_head_q, out, s);
}

int read_and_clear_device_status(int32_t *status) {
    if (cudaDeviceSynchronize() != cudaSuccess) return KVC_ECUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return KVC_ECUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return KVC_ECUDA;
    *status = v;
    return KVC_OK;
}

}  // namespace kvc
