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
// Split pass: grid (split, kv head), 4 warps per CTA.  A CTA streams its key
// range [split*len, (split+1)*len) of one kv head for all G query heads of the
// group; each warp takes 16-key groups in turn.  The warp computes the group's
// scores with mma.sync m16n8k16 (rows = query heads of the group, columns =
// keys), keeps an online softmax per head, and accumulates P*V with a second
// mma.sync (rows = heads, columns = head_dim).  K and V come straight from
// global memory into registers in the fragment layouts:
//   - q8_0 codes are converted to exact fp16 integers with two byte permutes
//     and one fp16 subtraction; the K scale is applied per 32-value block to
//     the fp32 partial scores, the V scale is folded into P per block, so the
//     only rounding besides fp32 accumulation is fp16(p*d);
//   - f16 values feed the MMAs as stored.
// Head-dim slots are permuted inside each MMA (the dot product does not care)
// so that every thread reads 8 (K) or 4 (V) contiguous code bytes per row.
// The four warps are merged in shared memory in a fixed order and the CTA
// writes (m, l, O) for its range to the scratch buffer.
//
// Combine pass: one CTA per query head, one thread per output value; merges
// the splits in split order (deterministic) and divides by the softmax sum.
//
// Split boundaries are absolute key positions, so the result does not depend
// on the cache layout.  No inter-CTA waits.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {
namespace {

constexpr int MAX_SPLIT = 256;
constexpr int WARPS = 4;
constexpr int GROUP_KEYS = 16;

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    return (uint32_t)__half_as_ushort(__float2half_rn(lo)) |
           ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
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
    const void *kq;
    const uint16_t *ks;
    const void *vq;
    const uint16_t *vs;
    float *part;       // scratch
    Geom g;
    int layer, n_keys, group, split_len, n_split, n_head_kv;
    float scale_log2;
};

// Per-group register tiles loaded ahead of use.
template <int D, bool Q8>
struct Tiles {
    static constexpr int NB = D / 32;
    // K: [n-tile t][block b] 8 code bytes (q8_0) or 8 halves (f16)
    uint2 k8[2][NB];
    uint4 k16[Q8 ? 1 : 2][Q8 ? 1 : NB];
    // V: [key r][block b] 4 code bytes (q8_0) or 4 halves (f16)
    uint32_t v8[4][NB];
    uint2 v16[Q8 ? 1 : 4][Q8 ? 1 : NB];
    // scales of keys j0+4c+r: NB fp16 values packed two per word
    uint32_t sk[4][NB / 2], sv[4][NB / 2];
    __device__ __forceinline__ float kscale(int r, int b) const {
        return __half2float(__ushort_as_half((unsigned short)(sk[r][b >> 1] >> (16 * (b & 1)))));
    }
    __device__ __forceinline__ float vscale(int r, int b) const {
        return __half2float(__ushort_as_half((unsigned short)(sv[r][b >> 1] >> (16 * (b & 1)))));
    }
};

template <int D, bool Q8>
__device__ __forceinline__ void load_group(const DecodeArgs &a, int hkv, int j0, int gq, int cq,
                                           Tiles<D, Q8> &T) {
    constexpr int NB = D / 32;
    const int last = a.n_keys - 1;
    const int64_t base_c = a.layer * a.g.c_layer + hkv * a.g.c_head;
    const int64_t base_s = a.layer * a.g.s_layer + hkv * a.g.s_head;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int key = min(j0 + 4 * (gq >> 1) + 2 * t + (gq & 1), last);
        const int64_t row = base_c + (int64_t)key * a.g.c_tok;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if constexpr (Q8)
                T.k8[t][b] = __ldg(reinterpret_cast<const uint2 *>(static_cast<const int8_t *>(a.kq) + row + 32 * b + 8 * cq));
            else
                T.k16[t][b] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.kq) + row + 32 * b + 8 * cq));
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int key = min(j0 + 4 * cq + r, last);
        const int64_t row = base_c + (int64_t)key * a.g.c_tok;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if constexpr (Q8)
                T.v8[r][b] = __ldg(reinterpret_cast<const uint32_t *>(static_cast<const int8_t *>(a.vq) + row + 32 * b + 4 * gq));
            else
                T.v16[r][b] = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.vq) + row + 32 * b + 4 * gq));
        }
        if constexpr (Q8) {
            // a key's NB scales are contiguous and 2*NB-byte aligned
            const int64_t srow = base_s + (int64_t)key * a.g.s_tok;
            if constexpr (NB == 4) {
                const uint2 wk = __ldg(reinterpret_cast<const uint2 *>(a.ks + srow));
                const uint2 wv = __ldg(reinterpret_cast<const uint2 *>(a.vs + srow));
                T.sk[r][0] = wk.x; T.sk[r][1] = wk.y;
                T.sv[r][0] = wv.x; T.sv[r][1] = wv.y;
            } else {
                T.sk[r][0] = __ldg(reinterpret_cast<const uint32_t *>(a.ks + srow));
                T.sv[r][0] = __ldg(reinterpret_cast<const uint32_t *>(a.vs + srow));
            }
        }
    }
}

template <int D, bool Q8, int DT>
__global__ void __launch_bounds__(WARPS * 32) decode_split_kernel(const DecodeArgs a) {
    constexpr int NB = D / 32;
    constexpr int KS = D / 16;       // k-steps of the score MMA
    constexpr int NT = D / 8;        // n-tiles of the output MMA
    const int split = blockIdx.x, hkv = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const int G = a.group;
    const int j_begin = split * a.split_len;
    const int j_end = min(a.n_keys, j_begin + a.split_len);

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

    float o[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    Tiles<D, Q8> cur, nxt;
    int j0 = j_begin + warp * GROUP_KEYS;
    if (j0 < j_end) load_group<D, Q8>(a, hkv, j0, gq, cq, cur);
#pragma unroll 1
    for (; j0 < j_end; j0 += WARPS * GROUP_KEYS) {
        const int jn = j0 + WARPS * GROUP_KEYS;
        if (jn < j_end) load_group<D, Q8>(a, hkv, jn, gq, cq, nxt);

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
                    for (int i = 0; i < 4; ++i)
                        sc[t][i] += cur.kscale(2 * t + (i & 1), b) * acc[i];
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
            alpha[hr] = ptx::ex2(m_run[hr] - m_new);
            float rs = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                p[hr][i] = ptx::ex2(x[i] - m_new);
                rs += p[hr][i];
            }
            l_run[hr] = l_run[hr] * alpha[hr] + rs;
            m_run[hr] = m_new;
        }
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                o[i][0] *= alpha[0]; o[i][1] *= alpha[0];
                o[i][2] *= alpha[1]; o[i][3] *= alpha[1];
            }
        }
        // ---- O += P V.  A = P (rows heads, k-slots 2c, 2c+1 <- keys 4c, 4c+1; 2c+8, 2c+9 <- 4c+2, 4c+3)
        //      B = V (k-slots as above, column n of n-tile 4b + s <- head-dim 32b + 4n + s)
        if constexpr (Q8) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float dv[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) dv[r] = cur.vscale(r, b);
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
        cur = nxt;
    }

    // ---- merge the four warps in shared memory (fixed order) and write the CTA's partial
    __shared__ float s_m[WARPS][16], s_l[WARPS][16];
    __shared__ float s_o[WARPS][16][D];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        float l = l_run[hr];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        const int row = gq + 8 * hr;
        if (cq == 0) {
            s_m[warp][row] = m_run[hr];
            s_l[warp][row] = l;
        }
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const int b = i >> 2, s = i & 3;
            s_o[warp][row][32 * b + 8 * cq + s] = o[i][2 * hr];
            s_o[warp][row][32 * b + 8 * cq + 4 + s] = o[i][2 * hr + 1];
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
        for (int w = 0; w < WARPS; ++w) M = fmaxf(M, s_m[w][row]);
        float acc = 0.f, lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < WARPS; ++w) {
                const float f = ptx::ex2(s_m[w][row] - M);
                acc += f * s_o[w][row][d];
                lsum += f * s_l[w][row];
            }
        }
        part_o[(pbase + row) * D + d] = acc;
        if (d == 0) {
            part_ml[(pbase + row) * 2] = M;
            part_ml[(pbase + row) * 2 + 1] = lsum;
        }
    }
}

// One CTA per query head, one thread per output value.  The split maxima and
// weights are computed once per CTA in shared memory; each thread then sums its
// value over the splits in split order (independent loads, unrolled).
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const float *__restrict__ part, int n_split,
                                                           int group, int n_head_kv, float *__restrict__ out) {
    __shared__ float s_w[MAX_SPLIT];
    __shared__ float s_red[D / 32];
    __shared__ float s_M, s_L;
    const int h = blockIdx.x, d = threadIdx.x;
    const int hkv = h / group, row = h % group;
    const float *part_o = part;
    const float *part_ml = part + (int64_t)n_head_kv * MAX_SPLIT * group * D;
    const int64_t p0 = ((int64_t)hkv * MAX_SPLIT) * group + row;   // partial index of split 0
    // maximum over splits
    float m = -INFINITY;
    for (int i = d; i < n_split; i += D) m = fmaxf(m, part_ml[(p0 + (int64_t)i * group) * 2]);
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((d & 31) == 0) s_red[d >> 5] = m;
    __syncthreads();
    if (d == 0) {
        float M = s_red[0];
        for (int w = 1; w < D / 32; ++w) M = fmaxf(M, s_red[w]);
        s_M = M;
    }
    __syncthreads();
    const float M = s_M;
    // split weights; the sum of weighted softmax denominators in split order
    for (int i = d; i < n_split; i += D) {
        const float mi = part_ml[(p0 + (int64_t)i * group) * 2];
        s_w[i] = (mi == -INFINITY) ? 0.f : ptx::ex2(mi - M);
    }
    __syncthreads();
    if (d == 0) {
        float L = 0.f;
        for (int i = 0; i < n_split; ++i) L += s_w[i] * part_ml[(p0 + (int64_t)i * group) * 2 + 1];
        s_L = L;
    }
    float acc = 0.f;
    int i = 0;
    for (; i + 8 <= n_split; i += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = part_o[(p0 + (int64_t)(i + u) * group) * D + d];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc += s_w[i + u] * v[u];
    }
    for (; i < n_split; ++i) acc += s_w[i] * part_o[(p0 + (int64_t)i * group) * D + d];
    __syncthreads();
    out[(int64_t)h * D + d] = acc / s_L;
}

int sm_count() {
    static int n = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            n = 148;
    });
    return n;
}

template <int D, bool Q8, int DT>
int launch_t(const kvc_cache &c, int layer, int pos, const void *q, int n_head_q, float *out,
             float *scratch, cudaStream_t s) {
    DecodeArgs a;
    a.q = q;
    a.kq = c.k_q;
    a.ks = static_cast<const uint16_t *>(c.k_s);
    a.vq = c.v_q;
    a.vs = static_cast<const uint16_t *>(c.v_s);
    a.part = scratch;
    a.g = geom_of(c.d);
    a.layer = layer;
    a.n_keys = pos + 1;
    a.n_head_kv = c.d.n_head_kv;
    a.group = n_head_q / c.d.n_head_kv;
    a.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)D));
    // about three CTAs per SM in total, whole 64-key rounds per split
    const int target = (3 * sm_count() + a.n_head_kv - 1) / a.n_head_kv;
    int n_split = (a.n_keys + 63) / 64;
    if (n_split > target) n_split = target;
    if (n_split > MAX_SPLIT) n_split = MAX_SPLIT;
    if (n_split < 1) n_split = 1;
    int len = (a.n_keys + n_split - 1) / n_split;
    len = (len + 63) / 64 * 64;
    n_split = (a.n_keys + len - 1) / len;
    a.split_len = len;
    a.n_split = n_split;
    decode_split_kernel<D, Q8, DT><<<dim3(n_split, a.n_head_kv), WARPS * 32, 0, s>>>(a);
    decode_combine_kernel<D><<<n_head_q, D, 0, s>>>(scratch, n_split, a.group, a.n_head_kv, out);
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
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

// The array's device address on the current device.  In host code the symbol
// name is only a host-side stand-in, so the address is looked up once per
// device (with that device current) through cudaGetSymbolAddress and cached.
int noalloc_scratch_address(float **out) {
    constexpr int MAX_DEVICES = 64;
    static std::mutex mu;
    static float *addr[MAX_DEVICES] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return KVC_ECUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return KVC_ECUDA;
        addr[dev] = static_cast<float *>(p);
    }
    *out = addr[dev];
    return KVC_OK;
}

}  // namespace

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
