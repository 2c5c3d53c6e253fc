// fd_w4_unpack.cuh - exact int4 -> fp32 conversion used by the GEMV prologue and by the
// dequantisation check kernel.
//
// A 32-bit word holds eight 4-bit two's complement integers q_0..q_7 (nibble j in bits
// 4j..4j+3). Flipping the top bit of a nibble gives u = q + 8 in [0, 15]. If the nibble
// is left where it is, at bits b..b+3 with b <= 16, and the float32 exponent field is
// set to e = 23 - b, the word reads as the float 2^e + u exactly (the nibble is the low
// part of the mantissa, one unit in the last place is 1.0). Subtracting 2^e + 8 then
// gives q exactly. Masking, flipping and setting the exponent is one lop3 per nibble:
//     bits = (word & (0xF << b)) ^ ((0x8 << b) | (127 + 23 - b) << 23)
// (the exponent bits do not meet the mask, so the xor sets them). Nibbles 5..7 sit too
// high (bit 23 belongs to the exponent) and are read from the word shifted right by 12,
// where they land at b = 8, 12, 16. The subtraction is done as packed fp32x2 adds.
#pragma once

#include "fd_internal.h"

namespace fd {

// Exponent field for 2^(23 - b), b the nibble's bit offset.
#define FD_EXP_FOR_BIT(b) ((uint32_t)(127 + 23 - (b)) << 23)
#define FD_KEY(b) ((0x8u << (b)) | FD_EXP_FOR_BIT(b))
// 2^(23 - b) + 8 as a float: the bias removed after the lop3.
#define FD_BIAS(b) ((float)(1u << (23 - (b))) + 8.0f)

// q_j for the 8 nibbles of `w`, as 4 float2 pairs (q0,q1) (q2,q3) (q4,q5) (q6,q7).
__device__ __forceinline__ void unpack_w4_f32x2(uint32_t w, float2 q[4]) {
    const uint32_t hi = w >> 12;
    float2 p0 = make_float2(__uint_as_float(and_xor(w, 0xFu << 0, FD_KEY(0))),
                            __uint_as_float(and_xor(w, 0xFu << 4, FD_KEY(4))));
    float2 p1 = make_float2(__uint_as_float(and_xor(w, 0xFu << 8, FD_KEY(8))),
                            __uint_as_float(and_xor(w, 0xFu << 12, FD_KEY(12))));
    float2 p2 = make_float2(__uint_as_float(and_xor(w, 0xFu << 16, FD_KEY(16))),
                            __uint_as_float(and_xor(hi, 0xFu << 8, FD_KEY(8))));
    float2 p3 = make_float2(__uint_as_float(and_xor(hi, 0xFu << 12, FD_KEY(12))),
                            __uint_as_float(and_xor(hi, 0xFu << 16, FD_KEY(16))));
    q[0] = fadd2(p0, make_float2(-FD_BIAS(0), -FD_BIAS(4)));
    q[1] = fadd2(p1, make_float2(-FD_BIAS(8), -FD_BIAS(12)));
    q[2] = fadd2(p2, make_float2(-FD_BIAS(16), -FD_BIAS(8)));
    q[3] = fadd2(p3, make_float2(-FD_BIAS(12), -FD_BIAS(16)));
}

}  // namespace fd
