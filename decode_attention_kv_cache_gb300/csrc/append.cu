// Append kernel: quantise a chunk's K/V rows into q8_0 blocks, or round them to
// f16, and store them at their cache positions.
//
// The q8_0 block (32 values along head_dim, fp16 scale d = amax/127, int8
// codes q = round(x/d)) is the one the pages' "q8_0 device-resident cache"
// names (llama.cpp PR #58 "completion : allow the prompt to be processed
// under its own split mode", section "Why"); the f16 cache is the one of
// llama.cpp PR #59 "llama : switch the split mode of a live context",
// section "Why".  The arithmetic repeats, bit for bit, the float32 op order:
// amax exact, d = amax/127 and x/d by IEEE division, ties away from zero,
// fp16 by round to nearest even.
//
// Work split: one thread per 8 consecutive values (one 16-byte load of bf16
// or f16 input, two of f32), four neighbouring lanes per 32-value block; the
// block's amax is a 4-lane xor-shuffle reduction.  Stores are 8-byte code
// stores (16 threads cover a 128-value head row) plus one 2-byte scale per
// block, so every warp writes whole 128-byte segments.  HBM-bound.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvc_internal.h"

namespace kvc {
namespace {

template <int DT>
__device__ __forceinline__ void load8(const void *base, int64_t idx, float (&x)[8]) {
    if constexpr (DT == KVC_IN_F32) {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(base) + idx);
        float4 a = __ldg(p), b = __ldg(p + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
        uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + idx));
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (DT == KVC_IN_BF16) {
                // bf16 -> f32 is exact: the bf16 bits are the top half of the f32
                x[2 * i] = __uint_as_float(w[i] << 16);
                x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            } else {
                x[2 * i] = __half2float(__ushort_as_half((unsigned short)(w[i] & 0xFFFF)));
                x[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(w[i] >> 16)));
            }
        }
    }
}

// grid.x covers units of 8 values of one tensor; grid.y selects K (0) or V (1).
template <int DT, bool Q8>
__global__ void __launch_bounds__(256) append_kernel(
    const void *__restrict__ k, const void *__restrict__ v, int64_t n_units, int units_per_tok,
    int units_per_head, void *kq, uint16_t *ks, void *vq, uint16_t *vs, Geom g, int layer, int pos0) {
    // a kernel launched after this one as a programmatic dependent (the decode split pass) may be
    // scheduled now; it waits for this grid's completion before it reads the cache
    asm volatile("griddepcontrol.launch_dependents;");
    const bool is_v = blockIdx.y != 0;
    const void *src = is_v ? v : k;
    const int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = u < n_units;
    const int64_t uu = live ? u : 0;
    const int tok = (int)(uu / units_per_tok);
    const int rem = (int)(uu % units_per_tok);
    const int head = rem / units_per_head;
    const int c = rem % units_per_head;  // which 8-value group along head_dim
    float x[8];
    if (live) load8<DT>(src, uu * 8, x);
    else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = 0.f;
    }
    const int64_t pos = (int64_t)pos0 + tok;
    const int64_t code_off = layer * g.c_layer + pos * g.c_tok + head * g.c_head + (int64_t)c * 8;
    if constexpr (Q8) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
        // the four lanes of one 32-value block are neighbours (units of a head row are consecutive)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const float d = __fdiv_rn(amax, 127.0f);
        uint32_t packed[2] = {0u, 0u};
        if (d > 0.f) {  // codes are zero when amax/127 is zero (x/d undefined)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float r = roundf(__fdiv_rn(x[i], d));  // round half away from zero
                r = fminf(fmaxf(r, -127.f), 127.f);
                const uint32_t b = (uint32_t)(uint8_t)(int8_t)(int)r;
                packed[i >> 2] |= b << (8 * (i & 3));
            }
        }
        if (live) {
            int8_t *dst = static_cast<int8_t *>(is_v ? vq : kq) + code_off;
            *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
            if ((c & 3) == 0) {
                uint16_t *sd = is_v ? vs : ks;
                sd[layer * g.s_layer + pos * g.s_tok + head * g.s_head + (c >> 2)] =
                    __half_as_ushort(__float2half_rn(d));
            }
        }
    } else {
        if (live) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                w[i] = (uint32_t)__half_as_ushort(__float2half_rn(x[2 * i])) |
                       ((uint32_t)__half_as_ushort(__float2half_rn(x[2 * i + 1])) << 16);
            }
            uint16_t *dst = static_cast<uint16_t *>(is_v ? vq : kq) + code_off;
            *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

template <int DT>
void launch_t(const kvc_cache &c, int layer, int pos0, int n, const void *k, const void *v,
              cudaStream_t s) {
    const Geom g = geom_of(c.d);
    const int units_per_head = c.d.head_dim / 8;
    const int units_per_tok = units_per_head * c.d.n_head_kv;
    const int64_t n_units = (int64_t)n * units_per_tok;
    const int threads = 256;
    dim3 grid((unsigned)((n_units + threads - 1) / threads), 2);
    if (c.d.type == KVC_Q8_0)
        append_kernel<DT, true><<<grid, threads, 0, s>>>(
            k, v, n_units, units_per_tok, units_per_head, c.k_q, (uint16_t *)c.k_s, c.v_q,
            (uint16_t *)c.v_s, g, layer, pos0);
    else
        append_kernel<DT, false><<<grid, threads, 0, s>>>(
            k, v, n_units, units_per_tok, units_per_head, c.k_q, nullptr, c.v_q, nullptr, g, layer,
            pos0);
}

}  // namespace

int launch_append(const kvc_cache &c, int layer, int pos0, int n_tokens, const void *k,
                  const void *v, int dtype, cudaStream_t s) {
    if (n_tokens == 0) return KVC_OK;
    switch (dtype) {
        case KVC_IN_F32: launch_t<KVC_IN_F32>(c, layer, pos0, n_tokens, k, v, s); break;
        case KVC_IN_BF16: launch_t<KVC_IN_BF16>(c, layer, pos0, n_tokens, k, v, s); break;
        default: launch_t<KVC_IN_F16>(c, layer, pos0, n_tokens, k, v, s); break;
    }
    return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ECUDA;
}

}  // namespace kvc
