// fd_dequant_debug.cu - writes W[n, k] = q[n, k] * s[n, k / group] as fp32, reading the
// nibbles through the same byte split the GEMV kernels feed to their dot-product unit
// ("09 - Operator fusion", section 5, taxonomy item 4: dequantize weights -> matmul).
// Test support: the result is compared bit for bit with the CPU oracle's dequantised
// weights, which pins nibble order, sign handling and scale indexing of the GEMV.
#include "fd_internal.h"
#include "fd_w4_unpack.cuh"

namespace fd {
namespace {

// One thread per 32-bit word (8 weights); grid-stride over all N * K / 8 words.
__global__ void w4_dequant_kernel(const uint32_t *__restrict__ qweight,
                                  const uint16_t *__restrict__ scales, float *__restrict__ out,
                                  int K, int N, int group) {
    const size_t words_per_row = (size_t)K / 8;
    const size_t total = words_per_row * (size_t)N;
    const int ngroups = K / group;
    const W4Keys keys = w4_keys();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t n = i / words_per_row;
        const size_t p = i % words_per_row;
        const size_t k0 = p * 8;
        const uint16_t sbits = scales[n * ngroups + k0 / group];
        const float s = __uint_as_float((uint32_t)sbits << 16);
        uint32_t L, H;
        split_w4(qweight[i], keys, L, H);
        float q[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) q[j] = (float)q_from_split(L, H, j) * s;
        float4 *dst = reinterpret_cast<float4 *>(out + n * (size_t)K + k0);
        dst[0] = make_float4(q[0], q[1], q[2], q[3]);
        dst[1] = make_float4(q[4], q[5], q[6], q[7]);
    }
}

}  // namespace

cudaError_t launch_w4_dequant_debug(const void *qweight, const void *scales, float *out,
                                    int K, int N, int group, cudaStream_t stream) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const size_t total = (size_t)K / 8 * (size_t)N;
    const int threads = 256;
    size_t blocks = (total + threads - 1) / threads;
    const size_t cap = (size_t)di.sm_count * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    w4_dequant_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<const uint32_t *>(qweight), static_cast<const uint16_t *>(scales), out, K,
        N, group);
    return cudaGetLastError();
}

}  // namespace fd
