// fd_w4_unpack.cuh - the int4 weight split shared by the GEMV kernels and the
// dequantisation check kernel.
//
// A 32-bit word holds eight 4-bit two's complement integers q_0..q_7 (nibble j in bits
// 4j..4j+3). Flipping the top bit of a nibble gives the offset value u = q + 8 in
// [0, 15]. Two lop3 split a word into byte lanes for the integer dot-product unit:
//     L = (w & 0x0F0F0F0F) ^ 0x08080808   byte b of L = u_{2b}         (even nibbles)
//     H = (w & 0xF0F0F0F0) ^ 0x80808080   byte b of H = 16 * u_{2b+1}  (odd nibbles)
// A lop3 takes one immediate operand, so the two xor keys are opaque register values
// created once per kernel (W4Keys) and the masks stay immediates: one lop3 each.
#pragma once

#include "fd_internal.h"

namespace fd {

struct W4Keys {
    uint32_t lo, hi;
};

// A register copy of `v` the compiler cannot fold back into an immediate.
__device__ __forceinline__ uint32_t opaque_u32(uint32_t v) {
    uint32_t r;
    asm volatile("mov.b32 %0, %1;" : "=r"(r) : "r"(v));
    return r;
}

__device__ __forceinline__ W4Keys w4_keys() {
    W4Keys k;
    k.lo = opaque_u32(0x08080808u);
    k.hi = opaque_u32(0x80808080u);
    return k;
}

template <uint32_t MASK>
__device__ __forceinline__ uint32_t mask_xor(uint32_t w, uint32_t key) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(w), "n"(MASK), "r"(key));
    return d;
}

__device__ __forceinline__ void split_w4(uint32_t w, const W4Keys &k, uint32_t &L, uint32_t &H) {
    L = mask_xor<0x0F0F0F0Fu>(w, k.lo);
    H = mask_xor<0xF0F0F0F0u>(w, k.hi);
}

// q_j (j = 0..7) back from the split bytes (used by the dequantisation check kernel).
__device__ __forceinline__ int q_from_split(uint32_t L, uint32_t H, int j) {
    const int b = j >> 1;
    return (j & 1) ? (int)((H >> (8 * b + 4)) & 0xF) - 8 : (int)((L >> (8 * b)) & 0xF) - 8;
}

}  // namespace fd
