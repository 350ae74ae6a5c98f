// The q8_0 block quantiser, shared by the append kernel and the fused decode step so that both
// store the same bytes.
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

#include "ptx.cuh"

namespace kvc {

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
