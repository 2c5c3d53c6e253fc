// fd_add_rmsnorm.cu - fused residual add + RMSNorm (one pass over HBM, two outputs).
//
// Source: "Kernel Fusion, torch.compile and CUDA Graphs, Measured", Step 2 (one program
// per row; h = bf16(x + r) stored as the new residual; rstd = 1 / sqrt(sum(h^2) / n +
// eps) on the rounded h; y = bf16(h * rstd) * w, rounded again), and "09 - Operator
// fusion", section 5 (taxonomy item 2, reduction + elementwise with a block reduction;
// "The fusion boundary problem": one kernel writes both the residual and the normalised
// row because the residual has two consumers).
//
// Design for GB300: a row is read once into registers as 16-byte bf16x8 vectors (VPT per
// thread), so the second pass of the page's compiler-generated kernel (re-reading h)
// never happens; 4 bytes are read and 4 written per element. The CTA grid is persistent
// (as many CTAs as fit on the 152 SMs, striding over rows), the sum of squares is a warp
// shuffle reduction followed by one shared-memory exchange (double-buffered, so one
// __syncthreads per row), streamed data carries an evict-first L2 policy and the weight
// row an evict-last one.
#include <atomic>

#include "fd_internal.h"

namespace fd {
namespace {

__device__ __forceinline__ float warp_allreduce_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Plain (coherent) 16-byte load with an L2 policy; x and residual may alias the outputs.
__device__ __forceinline__ uint4 ld_v4(const void *p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

template <int VPT>
__global__ void __launch_bounds__(VPT >= 8 ? 512 : 256)
    add_rmsnorm_kernel(const uint4 *x, const uint4 *residual, const uint4 *__restrict__ weight,
                       uint4 *out, uint4 *residual_out, int rows, int nvec, float inv_hidden,
                       float eps) {
    __shared__ float warp_ss[2][32];
    const int T = blockDim.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = T >> 5;
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    int parity = 0;
    // Every row is scaled by the same weight: with up to 4 vectors per thread the weight
    // lives in registers for the whole kernel, loaded once, alongside the first row.
    constexpr bool kWeightInRegs = VPT <= 4;
    uint4 wreg[kWeightInRegs ? VPT : 1];
    if (kWeightInRegs) {
#pragma unroll
        for (int i = 0; i < (kWeightInRegs ? VPT : 1); ++i) {
            const int v = tid + i * T;
            if (v < nvec) wreg[i] = ld_v4(weight + v, pol_keep);
        }
    }

    // x and residual may come from the previous kernel in the stream (programmatic
    // dependent launch): wait for it only now, after the weight row has been requested.
    grid_dep_wait();
    grid_dep_launch();

    for (int row = blockIdx.x; row < rows; row += gridDim.x) {
        const size_t base = (size_t)row * nvec;
        uint4 xv[VPT], rv[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int v = tid + i * T;
            if (v < nvec) {
                xv[i] = ld_v4(x + base + v, pol_stream);
                rv[i] = ld_v4(residual + base + v, pol_stream);
            }
        }
        // h = bf16(f32(x) + f32(r)); keep h (rounded) in registers, store it, and sum h^2.
        uint4 hv[VPT];
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int v = tid + i * T;
            if (v < nvec) {
                const uint32_t xw[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
                const uint32_t rw[4] = {rv[i].x, rv[i].y, rv[i].z, rv[i].w};
                uint32_t hw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    hw[j] = pack_bf16x2(bf16lo(xw[j]) + bf16lo(rw[j]),
                                        bf16hi(xw[j]) + bf16hi(rw[j]));
                    const float h0 = bf16lo(hw[j]), h1 = bf16hi(hw[j]);
                    ss = fmaf(h0, h0, ss);
                    ss = fmaf(h1, h1, ss);
                }
                hv[i] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                st_v4(residual_out + base + v, hv[i], pol_stream);
            }
        }
        ss = warp_allreduce_sum(ss);
        if (lane == 0) warp_ss[parity][warp] = ss;
        __syncthreads();
        float total = lane < nwarps ? warp_ss[parity][lane] : 0.f;
        total = warp_allreduce_sum(total);
        parity ^= 1;
        const float rstd = rsqrtf(fmaf(total, inv_hidden, eps));
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int v = tid + i * T;
            if (v < nvec) {
                const uint4 wv = kWeightInRegs ? wreg[kWeightInRegs ? i : 0] : ld_v4(weight + v, pol_keep);
                const uint32_t hw[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
                const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
                uint32_t yw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // bf16(h * rstd), then * w rounded to bf16 (the page's two roundings).
                    const uint32_t t = pack_bf16x2(bf16lo(hw[j]) * rstd, bf16hi(hw[j]) * rstd);
                    yw[j] = pack_bf16x2(bf16lo(t) * bf16lo(ww[j]), bf16hi(t) * bf16hi(ww[j]));
                }
                st_v4(out + base + v, make_uint4(yw[0], yw[1], yw[2], yw[3]), pol_stream);
            }
        }
    }
}

template <int VPT>
cudaError_t launch_vpt(const DeviceInfo &di, const void *x, const void *residual,
                       const void *weight, float eps, void *out, void *residual_out, int rows,
                       int hidden, cudaStream_t stream) {
    static std::atomic<int> occ_cache[64];
    const int nvec = hidden / 8;
    int T = (nvec + VPT - 1) / VPT;
    T = (T + 31) / 32 * 32;
    if (T > (VPT >= 8 ? 512 : 256)) return cudaErrorInvalidConfiguration;
    auto kern = add_rmsnorm_kernel<VPT>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    // Occupancy is cached per device and block size class (the block size is fixed per
    // hidden size in practice; recomputing on a mismatch is harmless).
    int occ = 0;
    const int cached = occ_cache[dev & 63].load(std::memory_order_relaxed);
    if ((cached >> 16) == T) {
        occ = cached & 0xFFFF;
    } else {
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, T, 0);
        if (err != cudaSuccess) return err;
        if (occ < 1) occ = 1;
        occ_cache[dev & 63].store((T << 16) | (occ & 0xFFFF), std::memory_order_relaxed);
    }
    long long grid = (long long)di.sm_count * occ;
    if (grid > rows) grid = rows;
    err = launch_kernel(add_rmsnorm_kernel<VPT>, dim3((unsigned)grid), dim3(T), 0, stream, 1,
                        static_cast<const uint4 *>(x), static_cast<const uint4 *>(residual),
                        static_cast<const uint4 *>(weight), static_cast<uint4 *>(out),
                        static_cast<uint4 *>(residual_out), rows, nvec, 1.0f / (float)hidden,
                        eps);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace

// VPT (16-byte vectors per thread per tensor) is the smallest of 1, 2, 4 that keeps the
// block at <= 256 threads, so hidden 4096 runs 256 threads x 2 vectors; above hidden 8192
// VPT is 8 with up to 512 threads (hidden <= 32768).
cudaError_t launch_add_rmsnorm(const void *x, const void *residual, const void *weight,
                               float eps, void *out, void *residual_out, int rows,
                               int hidden, cudaStream_t stream) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const int nvec = hidden / 8;
    if (nvec <= 256)
        return launch_vpt<1>(di, x, residual, weight, eps, out, residual_out, rows, hidden,
                             stream);
    if (nvec <= 512)
        return launch_vpt<2>(di, x, residual, weight, eps, out, residual_out, rows, hidden,
                             stream);
    if (nvec <= 1024)
        return launch_vpt<4>(di, x, residual, weight, eps, out, residual_out, rows, hidden,
                             stream);
    return launch_vpt<8>(di, x, residual, weight, eps, out, residual_out, rows, hidden,
                         stream);
}

}  // namespace fd
