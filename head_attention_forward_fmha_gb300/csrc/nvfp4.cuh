// nvfp4.cuh -- NVFP4 quantisation of output rows, fused into the epilogues.
//
// The fused FP4 output of commit 593bc25 of the nvfp4-megamoe-kernel pages
// ("register slot for FP4 pack" in the TMEM-epilogue part; its quantiser
// part names an E2M1 element nibble, an E4M3 scale and round-to-nearest-
// even).  Format (the pages give no block size; this is the reading taken):
//   - blocks of 16 consecutive elements of a row;
//   - block scale s = E4M3(amax / (6 g)), g a global fp32 scale (> 0);
//   - element code E2M1(x / (g s)), sign in bit 3 for a nonzero magnitude;
//   - both roundings to the nearest representable value, ties to the even
//     code, saturating at the largest finite value (448, 6); s = 0 gives 0;
//   - two codes per byte, element 2i in the low nibble; one scale byte per
//     block.  A value is recovered as g * s * e.
// amax / (6 g) and x / (g s) are IEEE fp32 divisions (the products 6 g and
// g s rounded to fp32 first), so each code is decided on a well-defined fp32
// number.
#pragma once
#include <cstdint>

namespace fmha {

// E4M3 code (0 .. 0x7E) nearest to a >= 0, ties to the even code, saturating
// at 448 (0x7E).  With E = max(floor(log2 a), -6), a * 2^(3 - E) lies in
// [8, 16) for a normal E4M3 value and in [0, 8) below 2^-6 (subnormals);
// rounding it to an integer r (half to even) gives the code (E + 6) * 8 + r,
// where r = 16 carries into the next binade and r's parity is the mantissa's.
__device__ __forceinline__ uint32_t e4m3_code(float a) {
    if (!(a > 0.f)) return 0u;
    if (a >= 448.f) return 0x7Eu;
    int e = (int)((__float_as_uint(a) >> 23) & 0xffu) - 127;
    e = max(e, -6);
    const float q = __fmul_rn(a, __uint_as_float((uint32_t)(127 + 3 - e) << 23));  // exact: a power of two
    const int r = __float2int_rn(q);
    return (uint32_t)min((e + 6) * 8 + r, 0x7E);
}

// The value of an E4M3 code (exact in fp32).
__device__ __forceinline__ float e4m3_value(uint32_t c) {
    const uint32_t e = c >> 3, m = c & 7u;
    if (e == 0) return (float)m * __uint_as_float((uint32_t)(127 - 9) << 23);         // m * 2^-9
    return (float)(8u + m) * __uint_as_float((uint32_t)(127 + (int)e - 10) << 23);   // (8 + m) * 2^(e - 10)
}

// E2M1 magnitude code (0 .. 7 for 0, .5, 1, 1.5, 2, 3, 4, 6) nearest to
// a >= 0: one comparison per midpoint (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5),
// strict where the lower neighbour's code is even (a tie stays down) and
// inclusive where the upper one's is (a tie goes up); beyond 5 it saturates
// to 6.  NaN compares false everywhere and gives 0.
__device__ __forceinline__ uint32_t e2m1_code(float a) {
    return (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) + (uint32_t)(a >= 1.75f) +
           (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) + (uint32_t)(a > 5.0f);
}

// One 16-element block: returns the E4M3 scale code and packs the 16 element
// codes into two 32-bit words (element i in bits 4 (i % 8) of word i / 8).
__device__ __forceinline__ uint32_t nvfp4_block(const float (&x)[16], float g, uint32_t (&packed)[2]) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    const uint32_t sc = e4m3_code(__fdiv_rn(amax, __fmul_rn(6.f, g)));
    const float s = e4m3_value(sc);
    packed[0] = packed[1] = 0u;
    if (s > 0.f) {
        const float gs = __fmul_rn(g, s);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float y = __fdiv_rn(x[i], gs);
            uint32_t c = e2m1_code(fabsf(y));
            if (y < 0.f && c != 0u) c |= 8u;
            packed[i >> 3] |= c << (4 * (i & 7));
        }
    }
    return sc;
}

}  // namespace fmha
