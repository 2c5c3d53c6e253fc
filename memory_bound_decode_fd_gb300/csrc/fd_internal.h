// fd_internal.h - device helpers and launcher prototypes shared by the CUDA sources of
// the fd library (not part of the public ABI; see include/fd.h for that).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/fd.h"

namespace fd {

// ------------------------------------------------------------------------------------
// Host-side device facts (cached per device; thread-safe).
// ------------------------------------------------------------------------------------
struct DeviceInfo {
    int sm_count;
    int max_smem_optin;   // bytes of dynamic shared memory a CTA may opt in to
    int smem_per_sm;      // bytes of shared memory per SM (all resident CTAs)
    int smem_reserved;    // bytes of shared memory the system reserves per CTA
    int l2_bytes;
};
// Returns cudaSuccess and fills `info` for the current device.
cudaError_t device_info(DeviceInfo *info);

// Process-wide launch options (fd_set_launch_flags), FD_LAUNCH_* bits.
unsigned launch_flags();

// Launches `kern` on `stream`; with FD_LAUNCH_PDL set the launch allows programmatic
// dependent launch (the kernel may start while the previous kernel in the stream is
// finishing; each kernel waits on griddepcontrol before it touches data that a previous
// kernel produces).
// `cluster` > 1 launches thread-block clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, int cluster, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (launch_flags() & FD_LAUNCH_PDL) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        ++cfg.numAttrs;
    }
    if (cluster > 1) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = (unsigned)cluster;
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------------------------------------
// Launchers (host). Arguments are validated by the C-ABI layer before these run.
// ------------------------------------------------------------------------------------
// Where a GEMV's outputs go: row n < split to out[m * ldo + n], row n >= split to
// out2[m * ldo + n - split]. A plain output is {out, nullptr, N, N}.
struct GemvOut {
    void *out;
    void *out2;
    int split;
    int ldo;
};

// The next layer's residual add + RMSNorm folded into the tail of an M = 1 GEMV
// (fd_swiglu_w4a16_gemv_add_rmsnorm): each CTA writes h = bf16(y + res_in) of its rows to
// res_out and its partial sum of h^2 to partials[blockIdx.x]; the last CTA to arrive
// (atomic ticket on *counter) normalises the whole row into `normed` and resets *counter.
// A null `normed` means no fold.
struct FoldArgs {
    const uint16_t *res_in;
    uint16_t *res_out;
    const uint16_t *weight;
    uint16_t *normed;
    float *partials;
    unsigned *counter;
    float eps;
    float inv_n;
};
// Scratch of the fold: the counter, then one fp32 partial per CTA.
constexpr int kFoldPartialsOffset = 256;
constexpr int kFoldMaxCtas = (FD_FOLD_SCRATCH_BYTES - kFoldPartialsOffset) / 4;

// `up` null: the activation is gate itself (a plain W4A16 GEMV), else silu(gate) * up.
// `residual` (bf16 [M, N], may equal `out`, or null) is added to the sum before the single
// rounding to bf16 (the residual-add epilogue of the down projection). `fold` (M = 1, SwiGLU
// form, no residual) adds the next layer's add + RMSNorm; a fold the kernel cannot run
// (grid above kFoldMaxCtas) leaves *launched false.
cudaError_t launch_gemv_tma(const void *gate, const void *up, const void *qweight,
                            const void *scales, const void *residual, GemvOut o, int M, int K,
                            int N, int group, cudaStream_t stream, bool *launched,
                            const FoldArgs *fold = nullptr);
// fd_swiglu_w4a16_gemv_add_rmsnorm_noalloc's fold on the library's own static scratch
// (fd_gemv_tma.cu): *launched = false when the bulk-copy kernel does not run the shape;
// *too_big when its grid needs more per-CTA sums than the array holds.
cudaError_t launch_gemv_fold_noalloc(const void *gate, const void *up, const void *qweight,
                                     const void *scales, void *y, const void *residual,
                                     const void *rms_weight, float eps, void *normed,
                                     void *residual_out, int K, int N, int group,
                                     cudaStream_t stream, bool *launched, bool *too_big);
// Tensor-core path (tcgen05) for batched decode; sets *launched = false when the shape
// is outside its rules (K % 1024, N % 128, group % 64, (K / group) % 8).
bool gemv_tc_supported(int M, int K, int N, int group);
// The decode step as one persistent kernel (fd_decode_step.cu); *launched = false when the
// shape has no kernel or no plan (fd_step_plan.h).
cudaError_t launch_decode_step(const fd_step_layer *layers, int n_layers, const void *x0,
                               void *residual, float eps, int hidden, int inter, int group,
                               void *scratch, cudaStream_t stream, bool *launched);
cudaError_t launch_gemv_tc(const void *gate, const void *up, const void *qweight,
                           const void *scales, const void *residual, void *out, int M, int K,
                           int N, int group, cudaStream_t stream, bool *launched);
cudaError_t launch_gemv_cc(const void *gate, const void *up, const void *qweight,
                           const void *scales, const void *residual, GemvOut o, int M, int K,
                           int N, int group, cudaStream_t stream);
cudaError_t launch_add_rmsnorm(const void *x, const void *residual, const void *weight,
                               float eps, void *out, void *residual_out, int rows,
                               int hidden, cudaStream_t stream);
// NVFP4 scaled matmul with the output multiplier folded in (fd_nvfp4.cu); the shape has
// passed plan_nvfp4's rules for every 128-row batch chunk.
cudaError_t launch_nvfp4_mm(const void *x, const void *x_sf, const void *w, const void *w_sf,
                            const float *alpha, void *out, int M, int K, int N,
                            cudaStream_t stream);
cudaError_t launch_w4_dequant_debug(const void *qweight, const void *scales, float *out,
                                    int K, int N, int group, cudaStream_t stream);

// Host accessors of the device status words of the files whose kernels have bounded waits
// (FD_DEFINE_STATUS_ACCESSOR in fd_tma.cuh): copy the word to *out on `stream`, then zero it
// if `clear`.
cudaError_t status_gemv_tma(cudaStream_t stream, unsigned *out, bool clear);
cudaError_t status_gemv_tc(cudaStream_t stream, unsigned *out, bool clear);
cudaError_t status_nvfp4(cudaStream_t stream, unsigned *out, bool clear);
cudaError_t status_decode_step(cudaStream_t stream, unsigned *out, bool clear);

// ------------------------------------------------------------------------------------
// Device helpers.
// ------------------------------------------------------------------------------------

// Programmatic dependent launch: wait until the previous kernel in the stream has
// completed and its writes are visible (a no-op for an ordinary launch), and allow the
// next kernel to begin launching.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2 policy for data touched once per call (activations, streamed weights, outputs).
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// L2 policy for data every CTA re-reads (the RMSNorm weight row).
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16-byte read-only load that bypasses L1 and carries an L2 eviction policy.
__device__ __forceinline__ uint4 ld_nc_v4(const void *p, uint64_t pol) {
    uint4 v;
    asm volatile(
        "ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p), "l"(pol));
    return v;
}

// 16-byte store with an L2 eviction policy.
__device__ __forceinline__ void st_v4(void *p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
                 :
                 : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

// Two bf16 in one 32-bit word -> two floats (exact).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two floats -> two bf16 (round to nearest even) packed low/high.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Packed fp32x2 arithmetic (one instruction for two lanes of work on sm_100+).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }

// (a & b) ^ c: one lop3 (the compiler folds the constant operands).
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c) {
    return (a & b) ^ c;
}

}  // namespace fd
