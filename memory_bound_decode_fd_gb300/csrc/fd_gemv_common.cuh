// fd_gemv_common.cuh - device pieces shared by the two CUDA-core W4A16 GEMV kernels: the
// SwiGLU prologue into registers (or the plain-activation one), the 32-k integer dot
// product, the warp reduce-scatter, the cross-warp sum and the output addressing.
//
// Numerics of one 32-k slice (one 16-byte weight vector position, inside one scale
// group):
//   a_k = silu(g_k) * u_k in fp32 through the identity silu(x) = (x/2)(1 + tanh(x/2))
//   (one MUFU tanh per element; its error leaves a_k within 2^-10.5 |g_k u_k / 2|);
//   a_k is encoded as a16_k = rint(a_k * 32767 / amax) with amax = max |a_k| over the
//   slice (a block-scaled 16-bit integer: 15 magnitude bits against bf16's 8), and
//   a_k ~= a16_k * scale, scale = amax / 32767;
//   sum_k a16_k q_k is formed EXACTLY in int32 with the dp2a integer dot-product
//   instruction (16-bit x 8-bit products), from the byte split of fd_w4_unpack.cuh;
//   the slice's contribution to y[n] is float(that sum) * (scale * s[n, group]).
// Beyond fp32 rounding, the errors are tanh's and the 16-bit encoding of a (at most
// amax / 65534 per element). A plain activation x (encode_plain) is encoded the same way,
// without the tanh step.
#pragma once

#include "fd_internal.h"
#include "fd_w4_unpack.cuh"

namespace fd {

constexpr int kWindowRows = 64;  // rows whose per-warp partials are held before a flush

// Address of output (m, n): rows n < split go to out (row stride ldo); rows n >= split go
// to out2 at column n - split (the gate and up halves of a horizontal gate/up projection).
// A plain GEMV has split = ldo = N.
__device__ __forceinline__ uint16_t *out_at(uint16_t *out, uint16_t *out2, int split, int ldo,
                                            int m, int n) {
    return n < split ? out + (size_t)m * ldo + n : out2 + (size_t)m * ldo + (n - split);
}

// Sum of the n per-warp partials of one output (p[w * stride], w < n) in four
// independent chains, so the loads overlap: a single chain waits on each load in turn,
// which made the final flush of a CTA's outputs ~0.3 us long at 28 warps.
__device__ __forceinline__ float sum_partials(const float *p, int n, int stride) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int w = 0;
#pragma unroll 2
    for (; w + 3 < n; w += 4) {
        a0 += p[(size_t)w * stride];
        a1 += p[(size_t)(w + 1) * stride];
        a2 += p[(size_t)(w + 2) * stride];
        a3 += p[(size_t)(w + 3) * stride];
    }
    for (; w < n; ++w) a0 += p[(size_t)w * stride];
    return (a0 + a1) + (a2 + a3);
}

// One thread's activation slice (32 k) for one activation row, in the operand layout of
// dp2a: for word i (k = 8i .. 8i+7 of the slice),
//   e[i] = (a16[8i+0], a16[8i+2]), f[i] = (a16[8i+4], a16[8i+6])  pair with L's bytes
//   g[i] = (a16[8i+1], a16[8i+3]), h[i] = (a16[8i+5], a16[8i+7])  pair with H's bytes
// init_lo / init_hi remove the +8 offset of the nibbles (u = q + 8):
//   sum a16 u_even = sum a16 q_even + 8 S_even;  sum a16 16 u_odd = 16 sum a16 q_odd + 128 S_odd.
struct Act16 {
    uint32_t e[4], f[4], g[4], h[4];
    int init_lo, init_hi;
    float scale;
};

__device__ __forceinline__ uint32_t pack16(int lo, int hi) {
    return __byte_perm((uint32_t)lo, (uint32_t)hi, 0x5410);
}

// Round-to-nearest-even float -> int for |x| < 2^22 with two fast-pipe instructions.
__device__ __forceinline__ int rint_small(float x) {
    return (int)(__float_as_uint(x + 12582912.0f) - 0x4B400000u);
}

// Raw bf16 gate/up of one 32-element slice (issued early so the loads overlap set-up).
struct GateUp {
    uint4 g[4], u[4];
};

__device__ __forceinline__ void load_gate_up(const uint16_t *__restrict__ gate,
                                             const uint16_t *__restrict__ up, size_t offset,
                                             GateUp &gu) {
    const uint4 *g4 = reinterpret_cast<const uint4 *>(gate + offset);
    const uint4 *u4 = reinterpret_cast<const uint4 *>(up + offset);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        gu.g[i] = g4[i];
        gu.u[i] = u4[i];
    }
}

// tanh on MUFU (tanh.approx.f32: relative error about 2^-11).
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Power-of-two factor applied to a slice before its int16 encoding: 2^64 when the slice's
// largest magnitude is below 2^-64, else 1. The code of a_k is rint(a_k * 32767 / amax),
// and 32767 / amax overflows fp32 for amax below about 2^-113; scaling both by 2^64 is
// exact and keeps the quotient finite, so tiny (even subnormal) slices encode like others.
__device__ __forceinline__ float slice_prescale(float amax) {
    return amax < 0x1p-64f ? 0x1p64f : 1.0f;
}

__device__ __forceinline__ void encode_floats(const float2 (&a)[16], Act16 &act);

// Encodes one slice of a = silu(g) * u (see Act16).
__device__ __forceinline__ void encode_q16(const GateUp &gu, Act16 &act) {
    // silu(g) u = (g u / 2)(1 + tanh(g / 2)), two elements per packed instruction;
    // a[4i + j] holds elements 8i + 2j and 8i + 2j + 1
    float2 a[16];
    const float2 half2 = make_float2(0.5f, 0.5f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t gw[4] = {gu.g[i].x, gu.g[i].y, gu.g[i].z, gu.g[i].w};
        const uint32_t uw[4] = {gu.u[i].x, gu.u[i].y, gu.u[i].z, gu.u[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 h = __fmul2_rn(make_float2(bf16lo(gw[j]), bf16hi(gw[j])), half2);
            const float2 p = __fmul2_rn(h, make_float2(bf16lo(uw[j]), bf16hi(uw[j])));
            a[4 * i + j] = __ffma2_rn(p, make_float2(tanh_approx(h.x), tanh_approx(h.y)), p);
        }
    }
    encode_floats(a, act);
}

// Encodes one slice of a plain bf16 activation x (32 elements, four 16-byte words).
__device__ __forceinline__ void encode_plain(const uint4 (&x)[4], Act16 &act) {
    float2 a[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) a[4 * i + j] = make_float2(bf16lo(w[j]), bf16hi(w[j]));
    }
    encode_floats(a, act);
}

// The block-scaled int16 encoding of a slice's 32 fp32 values (see Act16).
__device__ __forceinline__ void encode_floats(const float2 (&a)[16], Act16 &act) {
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fmaxf(fabsf(a[k].x), fabsf(a[k].y)));
    const float pre = slice_prescale(amax);
    const float s_inv = amax > 0.f ? __fdividef(32767.0f, amax * pre) : 0.f;
    act.scale = amax * (1.0f / 32767.0f);
    // round(a * s_inv) by one fma with 1.5 * 2^23: the low 16 bits of the result are the
    // int16 code (two's complement), and the integer sum is the bit sum minus the bias
    const float2 sv = make_float2(s_inv, s_inv);
    const float2 mg = make_float2(12582912.0f, 12582912.0f);
    const float2 pv = make_float2(pre, pre);
    uint32_t b[32];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float2 r = __ffma2_rn(__fmul2_rn(a[k], pv), sv, mg);
        b[2 * k] = __float_as_uint(r.x);
        b[2 * k + 1] = __float_as_uint(r.y);
    }
    uint32_t s_even = 0u - 16u * 0x4B400000u, s_odd = 0u - 16u * 0x4B400000u;
#pragma unroll
    for (int k = 0; k < 32; k += 2) {
        s_even += b[k];
        s_odd += b[k + 1];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        act.e[i] = __byte_perm(b[8 * i + 0], b[8 * i + 2], 0x5410);
        act.f[i] = __byte_perm(b[8 * i + 4], b[8 * i + 6], 0x5410);
        act.g[i] = __byte_perm(b[8 * i + 1], b[8 * i + 3], 0x5410);
        act.h[i] = __byte_perm(b[8 * i + 5], b[8 * i + 7], 0x5410);
    }
    act.init_lo = -8 * (int)s_even;
    act.init_hi = -128 * (int)s_odd;
}
// Paired-lane form of encode_q16 (lanes l and l ^ 16 share one 32-k slice): this lane
// holds the slice's elements 16h .. 16h + 15 (h = half), computes their codes, and the
// pair exchanges amax, codes and offset sums by shuffles, so that both lanes end with the
// whole slice's Act16 (identical to encode_q16 on the 32 elements, up to the order of the
// amax reduction, which max makes exact).
struct GateUpHalf {
    uint4 g[2], u[2];
};

__device__ __forceinline__ void encode_floats_pair(const float2 (&a)[8], int h, Act16 &act);

__device__ __forceinline__ void encode_q16_pair(const GateUpHalf &gu, int h, Act16 &act) {
    float2 a[8];  // a[4i + j] holds elements 8i + 2j, 8i + 2j + 1 of this half
    const float2 half2 = make_float2(0.5f, 0.5f);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t gw[4] = {gu.g[i].x, gu.g[i].y, gu.g[i].z, gu.g[i].w};
        const uint32_t uw[4] = {gu.u[i].x, gu.u[i].y, gu.u[i].z, gu.u[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 hh = __fmul2_rn(make_float2(bf16lo(gw[j]), bf16hi(gw[j])), half2);
            const float2 p = __fmul2_rn(hh, make_float2(bf16lo(uw[j]), bf16hi(uw[j])));
            a[4 * i + j] = __ffma2_rn(p, make_float2(tanh_approx(hh.x), tanh_approx(hh.y)), p);
        }
    }
    encode_floats_pair(a, h, act);
}

// Paired-lane form of encode_plain: this lane holds elements 16h .. 16h + 15 of the slice
// (two 16-byte words of a plain bf16 activation).
__device__ __forceinline__ void encode_plain_pair(const uint4 (&x)[2], int h, Act16 &act) {
    float2 a[8];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t w[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) a[4 * i + j] = make_float2(bf16lo(w[j]), bf16hi(w[j]));
    }
    encode_floats_pair(a, h, act);
}

// The pair's block-scaled int16 encoding of its 32 fp32 values (16 per lane).
__device__ __forceinline__ void encode_floats_pair(const float2 (&a)[8], int h, Act16 &act) {
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fmaxf(fabsf(a[k].x), fabsf(a[k].y)));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 16));
    const float pre = slice_prescale(amax);
    const float s_inv = amax > 0.f ? __fdividef(32767.0f, amax * pre) : 0.f;
    act.scale = amax * (1.0f / 32767.0f);
    const float2 sv = make_float2(s_inv, s_inv);
    const float2 mg = make_float2(12582912.0f, 12582912.0f);
    const float2 pv = make_float2(pre, pre);
    uint32_t b[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float2 r = __ffma2_rn(__fmul2_rn(a[k], pv), sv, mg);
        b[2 * k] = __float_as_uint(r.x);
        b[2 * k + 1] = __float_as_uint(r.y);
    }
    uint32_t sum = 0u - 16u * 0x4B400000u;
#pragma unroll
    for (int k = 0; k < 16; ++k) sum += b[k];
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 16);
    // with accumulators started at 0, lo + (hi >> 4) exceeds the exact sum by 8 * sum(q)
    act.init_lo = -8 * (int)sum;
    act.init_hi = 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t mine[4] = {__byte_perm(b[8 * i + 0], b[8 * i + 2], 0x5410),
                                  __byte_perm(b[8 * i + 4], b[8 * i + 6], 0x5410),
                                  __byte_perm(b[8 * i + 1], b[8 * i + 3], 0x5410),
                                  __byte_perm(b[8 * i + 5], b[8 * i + 7], 0x5410)};
        uint32_t other[4];
#pragma unroll
        for (int f = 0; f < 4; ++f) other[f] = __shfl_xor_sync(0xFFFFFFFFu, mine[f], 16);
        // words 0-1 of the slice come from half 0, words 2-3 from half 1
        act.e[i] = h ? other[0] : mine[0];
        act.f[i] = h ? other[1] : mine[1];
        act.g[i] = h ? other[2] : mine[2];
        act.h[i] = h ? other[3] : mine[3];
        act.e[2 + i] = h ? mine[0] : other[0];
        act.f[2 + i] = h ? mine[1] : other[1];
        act.g[2 + i] = h ? mine[2] : other[2];
        act.h[2 + i] = h ? mine[3] : other[3];
    }
}

// Builds the slice's Act16 from bf16 gate/up at element `offset` (32 elements).
__device__ __forceinline__ void load_activation_q16(const uint16_t *__restrict__ gate,
                                                    const uint16_t *__restrict__ up,
                                                    size_t offset, Act16 &act) {
    GateUp gu;
    load_gate_up(gate, up, offset, gu);
    encode_q16(gu, act);
}

__device__ __forceinline__ void zero_activation(Act16 &act) {
#pragma unroll
    for (int i = 0; i < 4; ++i) act.e[i] = act.f[i] = act.g[i] = act.h[i] = 0u;
    act.init_lo = act.init_hi = 0;
    act.scale = 0.f;
}

__device__ __forceinline__ int dp2a_lo(uint32_t a16x2, uint32_t bytes, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a16x2), "r"(bytes), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a16x2, uint32_t bytes, int c) {
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a16x2), "r"(bytes), "r"(c));
    return d;
}

// Exact sum over the 32 k of one weight vector of a16_k * q_k.
__device__ __forceinline__ int dot32_q16(const Act16 &act, uint4 wv, const W4Keys &keys) {
    const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
    int lo = act.init_lo, hi = act.init_hi;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t L, H;
        split_w4(w[i], keys, L, H);
        lo = dp2a_lo(act.e[i], L, lo);
        hi = dp2a_lo(act.g[i], H, hi);
        lo = dp2a_hi(act.f[i], L, lo);
        hi = dp2a_hi(act.h[i], H, hi);
    }
    return lo + (hi >> 4);
}

// For MB activation rows: d[mb] = fp32 contribution of this vector position. The integer
// sum is scaled by the activation scale first, then by the group scale: for a slice of
// tiny activations (scale below about 2^-100) the product of the two scales alone would
// fall into the subnormal range and lose precision, the sum times the scale does not.
template <int MB>
__device__ __forceinline__ void dot32(const Act16 *act, uint4 wv, const W4Keys &keys,
                                      float group_scale, float d[MB]) {
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
        d[mb] = ((float)dot32_q16(act[mb], wv, keys) * act[mb].scale) * group_scale;
}

__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v >> 1); }

// warp_reduce_scatter within each 16-lane half of the warp: on return, lane l holds in
// v[0] the sum over its half of value index ((l & 15) >> (4 - log2 V)).
template <int V>
__device__ __forceinline__ float half_reduce_scatter(float (&v)[V], int lane) {
#pragma unroll
    for (int width = V; width > 1; width >>= 1) {
        const int half = width >> 1;
        const int offset = 8 >> (ilog2(V) - ilog2(width));
        const bool upper = (lane & offset) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, offset);
        }
    }
    float r = v[0];
#pragma unroll
    for (int offset = 8 >> ilog2(V); offset > 0; offset >>= 1)
        r += __shfl_xor_sync(0xFFFFFFFFu, r, offset);
    return r;
}

// Butterfly reduce-scatter of V values over a warp. On return, lane l holds in v[0] the
// warp-wide sum of value index (l >> (5 - log2 V)).
template <int V>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[V], int lane) {
#pragma unroll
    for (int width = V; width > 1; width >>= 1) {
        const int half = width >> 1;
        // offset for this stage: 16, 8, ... (one bit of the lane index per halving)
        const int offset = 16 >> (ilog2(V) - ilog2(width));
        const bool upper = (lane & offset) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, offset);
        }
    }
    float r = v[0];
#pragma unroll
    for (int offset = 16 >> ilog2(V); offset > 0; offset >>= 1)
        r += __shfl_xor_sync(0xFFFFFFFFu, r, offset);
    return r;
}

}  // namespace fd
