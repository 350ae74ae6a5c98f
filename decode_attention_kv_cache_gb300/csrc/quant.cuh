// The q8_0 block quantiser and the input loader, shared by the append kernel and the fused decode and
// prefill steps so that all of them store the same bytes.
//
// One block is 32 values along head_dim: fp16 scale d = amax / 127, int8 codes q = round(x / d)
// (llama.cpp PR #58 "completion : allow the prompt to be processed under its own split mode",
// section "Why": the q8_0 device-resident cache).  The arithmetic repeats, bit for bit, the float32
// op order: amax exact, d = amax/127 and x/d by IEEE division, ties away from zero.  The quotient x/d
// is taken as x times the IEEE reciprocal of d and rounded with a 1.5*2^23 shift; that product is
// within 5e-5 of the IEEE quotient, so the rounded code can differ from round(x/d) only when the
// product lies within that distance of a .5 boundary, and exactly those values are recomputed with
// the IEEE division (both values of a pair, the one away from the boundary giving the same code
// either way).  A non-finite block (outside the method's domain) gets zero codes.
#pragma once

#include <cuda_fp16.h>

#include "kvc_internal.h"
#include "ptx.cuh"

namespace kvc {

// 8 consecutive input values (f32, bf16 or f16: DT is a kvc_dtype) from element index idx, read through L2
// (a kernel just before the reader may have written them), as floats: bf16 and f16 widen exactly.
template <int DT>
__device__ __forceinline__ void load_inputs8(const void *base, int64_t idx, float (&x)[8]) {
    if constexpr (DT == KVC_IN_F32) {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(base) + idx);
        const float4 a = __ldcg(p), b = __ldcg(p + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
        const uint4 u = __ldcg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + idx));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (DT == KVC_IN_BF16) {
                x[2 * i] = __uint_as_float(w[i] << 16);          // the bf16 bits are the f32's top half
                x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            } else {
                x[2 * i] = __half2float(__ushort_as_half((unsigned short)(w[i] & 0xFFFF)));
                x[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(w[i] >> 16)));
            }
        }
    }
}

// Quantise x[0..31]: the 32 codes packed four to a word (byte i of word w is code 4 w + i) and the
// fp16 bits of the scale.
__device__ __forceinline__ uint16_t q8_0_quantize32(const float (&x)[32], uint32_t (&packed)[8]) {
    float m2[2] = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        m2[0] = ptx::fmax3(m2[0], fabsf(x[i]), fabsf(x[i + 1]));
        m2[1] = ptx::fmax3(m2[1], fabsf(x[i + 2]), fabsf(x[i + 3]));
    }
    const float amax = fmaxf(m2[0], m2[1]);
    const float d = __fdiv_rn(amax, 127.0f);
#pragma unroll
    for (int w = 0; w < 8; ++w) packed[w] = 0u;
    // codes are zero when amax/127 is zero (x/d undefined); |x * r| <= 127 (to an ulp) otherwise
    if (d > 0.f && amax <= 3.402823466e38f) {
        const float r = __frcp_rn(d);
        const uint64_t r2 = ptx::f2_pack(r, r), mz = ptx::f2_pack(-0.f, -0.f), M2 = ptx::f2_pack(12582912.f, 12582912.f),
                       nM2 = ptx::f2_pack(-12582912.f, -12582912.f), n1 = ptx::f2_pack(-1.f, -1.f);
        int q[32];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const uint64_t y = ptx::f2_fma(ptx::f2_pack(x[i], x[i + 1]), r2, mz);   // x * r, one rounding
            const uint64_t t = ptx::f2_add(y, M2);                                // y rounded to an integer (to even)
            const uint64_t f = ptx::f2_fma(ptx::f2_add(t, nM2), n1, y);              // y minus that integer
            float t0, t1, f0, f1;
            ptx::f2_unpack(t, t0, t1);
            ptx::f2_unpack(f, f0, f1);
            q[i] = __float_as_int(t0) - 0x4B400000;
            q[i + 1] = __float_as_int(t1) - 0x4B400000;
            if (fmaxf(fabsf(f0), fabsf(f1)) > 0.4999f) {  // near a tie: exact quotients
                q[i] = (int)roundf(__fdiv_rn(x[i], d));
                q[i + 1] = (int)roundf(__fdiv_rn(x[i + 1], d));
            }
        }
#pragma unroll
        for (int w = 0; w < 8; ++w)
            packed[w] = __byte_perm(__byte_perm(q[4 * w], q[4 * w + 1], 0x0040),
                                    __byte_perm(q[4 * w + 2], q[4 * w + 3], 0x0040), 0x5410);
    }
    return __half_as_ushort(__float2half_rn(d));
}

}  // namespace kvc
