// fd_api.cu - the C ABI (include/fd.h): argument checks, dispatch, status strings.
//
// Every check runs on the host before any CUDA call, so a rejected call launches nothing
// and touches no device state (it also works on a machine without a GPU).
#include <atomic>
#include <cmath>
#include <cstdint>

#include "fd_copy.h"
#include "fd_gemv_plan.h"
#include "fd_gemv_tc_plan.h"
#include "fd_internal.h"
#include "fd_nvfp4_plan.h"
#include "fd_step_plan.h"

namespace fd {

namespace {

constexpr int kMaxDevices = 64;
// Smallest M that FD_GEMV_AUTO sends to the tensor-core path.
constexpr int kTensorCoreMinM = 16;
std::atomic<int> g_info_ready[kMaxDevices];
DeviceInfo g_info[kMaxDevices];
thread_local int g_last_cuda_error = 0;
std::atomic<int> g_gemv_path{FD_GEMV_AUTO};
std::atomic<unsigned> g_launch_flags{0u};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t a_bytes, const void *b, size_t b_bytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + b_bytes && b0 < a0 + a_bytes;
}

// FD_LAUNCH_TEST_FAIL: the launch is reported as failed without calling CUDA.
bool fake_launch_failure() {
    return (g_launch_flags.load(std::memory_order_relaxed) & FD_LAUNCH_TEST_FAIL) != 0;
}

int from_cuda(cudaError_t err) {
    if (err == cudaSuccess) return FD_OK;
    g_last_cuda_error = static_cast<int>(err);
    return FD_ERR_CUDA;
}

// Sizes of a W4 GEMV call apart from its pointers: FD_OK, an error, or kEmpty when there is
// nothing to compute (M == 0 or N == 0), in which case no pointer is read.
constexpr int kEmpty = -1;
int check_w4_sizes(int M, int K, int N, int group) {
    if (M < 0 || N < 0 || K <= 0 || group <= 0) return FD_ERR_SHAPE;
    if (K % 32 != 0 || group % 32 != 0 || K % group != 0) return FD_ERR_SHAPE;
    if (K > FD_MAX_K || M > FD_MAX_M) return FD_ERR_UNSUPPORTED;
    return (M == 0 || N == 0) ? kEmpty : FD_OK;
}

int check_w4_layout(const void *qweight, const void *scales, int K, int N, int group) {
    if (!qweight || !scales) return FD_ERR_NULL;
    if (K <= 0 || N <= 0 || group <= 0) return FD_ERR_SHAPE;
    if (K % 32 != 0 || group % 32 != 0 || K % group != 0) return FD_ERR_SHAPE;
    if (K > FD_MAX_K) return FD_ERR_UNSUPPORTED;
    if (!aligned16(qweight) || !aligned16(scales)) return FD_ERR_ALIGN;
    return FD_OK;
}

}  // namespace

cudaError_t device_info(DeviceInfo *info) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const int slot = dev % kMaxDevices;
    if (g_info_ready[slot].load(std::memory_order_acquire) == dev + 1) {
        *info = g_info[slot];
        return cudaSuccess;
    }
    DeviceInfo di{};
    err = cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                 dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                 dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&di.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&di.l2_bytes, cudaDevAttrL2CacheSize, dev);
    if (err != cudaSuccess) return err;
    // Benign race: concurrent first calls write identical values.
    g_info[slot] = di;
    g_info_ready[slot].store(dev + 1, std::memory_order_release);
    *info = di;
    return cudaSuccess;
}

unsigned launch_flags() { return g_launch_flags.load(std::memory_order_relaxed); }

}  // namespace fd

using namespace fd;

namespace {

// Validation and kernel choice shared by both GEMV entry points; `residual` may be null.
int swiglu_gemv(const void *gate, const void *up, const void *qweight, const void *scales,
                const void *residual, void *out, int M, int K, int N, int group,
                fd_stream_t stream) {
    const int sz = check_w4_sizes(M, K, N, group);
    if (sz == kEmpty) return FD_OK;
    if (!gate || !up || !out) return FD_ERR_NULL;
    if (sz != FD_OK) return sz;
    int st = check_w4_layout(qweight, scales, K, N, group);
    if (st != FD_OK) return st;
    if (!aligned16(gate) || !aligned16(up) || !aligned16(out)) return FD_ERR_ALIGN;
    if (residual && !aligned16(residual)) return FD_ERR_ALIGN;
    const size_t act_bytes = (size_t)M * K * 2;
    const size_t out_bytes = (size_t)M * N * 2;
    const size_t w_bytes = (size_t)N * K / 2;
    const size_t s_bytes = (size_t)N * (K / group) * 2;
    if (overlaps(out, out_bytes, gate, act_bytes) || overlaps(out, out_bytes, up, act_bytes) ||
        overlaps(out, out_bytes, qweight, w_bytes) || overlaps(out, out_bytes, scales, s_bytes))
        return FD_ERR_OVERLAP;
    // the residual may be the output itself (in place), or apart from every other buffer
    if (residual && residual != out &&
        (overlaps(residual, out_bytes, out, out_bytes) ||
         overlaps(residual, out_bytes, gate, act_bytes) ||
         overlaps(residual, out_bytes, up, act_bytes) ||
         overlaps(residual, out_bytes, qweight, w_bytes) ||
         overlaps(residual, out_bytes, scales, s_bytes)))
        return FD_ERR_OVERLAP;
    if (fake_launch_failure()) return from_cuda(cudaErrorLaunchOutOfResources);
    cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
    const int path = g_gemv_path.load(std::memory_order_relaxed);
    if (fd_gemv_uses_tensor_cores(M, K, N, group)) {
        bool launched = false;
        cudaError_t err = launch_gemv_tc(gate, up, qweight, scales, residual, out, M, K, N,
                                         group, st_, &launched);
        if (err != cudaSuccess || launched) return from_cuda(err);
    }
    const GemvOut o{out, nullptr, N, N};
    if (path == FD_GEMV_AUTO || path == FD_GEMV_BULK) {
        bool launched = false;
        cudaError_t err = launch_gemv_tma(gate, up, qweight, scales, residual, o, M, K, N,
                                          group, st_, &launched);
        if (err != cudaSuccess || launched) return from_cuda(err);
    }
    return from_cuda(launch_gemv_cc(gate, up, qweight, scales, residual, o, M, K, N, group, st_));
}

}  // namespace

extern "C" {


int fd_swiglu_w4a16_gemv(const void *gate, const void *up, const void *qweight,
                         const void *scales, void *out, int M, int K, int N, int group,
                         fd_stream_t stream) {
    return swiglu_gemv(gate, up, qweight, scales, nullptr, out, M, K, N, group, stream);
}

int fd_swiglu_w4a16_gemv_residual(const void *gate, const void *up, const void *qweight,
                                  const void *scales, const void *residual, void *out, int M,
                                  int K, int N, int group, fd_stream_t stream) {
    if (check_w4_sizes(M, K, N, group) == kEmpty) return FD_OK;
    if (!residual) return FD_ERR_NULL;
    return swiglu_gemv(gate, up, qweight, scales, residual, out, M, K, N, group, stream);
}

int fd_swiglu_w4a16_gemv_add_rmsnorm(const void *gate, const void *up, const void *qweight,
                                     const void *scales, void *y, const void *residual,
                                     const void *rms_weight, float eps, void *normed,
                                     void *residual_out, void *scratch, int K, int N, int group,
                                     fd_stream_t stream) {
    const int sz = check_w4_sizes(1, K, N, group);
    if (sz == kEmpty) return FD_OK;
    if (!(eps >= 0.0f) || !std::isfinite(eps) || N % 8 != 0) return FD_ERR_SHAPE;
    if (!gate || !up || !y || !residual || !rms_weight || !normed || !residual_out || !scratch)
        return FD_ERR_NULL;
    if (sz != FD_OK) return sz;
    int st = check_w4_layout(qweight, scales, K, N, group);
    if (st != FD_OK) return st;
    if (!aligned16(gate) || !aligned16(up) || !aligned16(y) || !aligned16(residual) ||
        !aligned16(rms_weight) || !aligned16(normed) || !aligned16(residual_out) ||
        !aligned16(scratch))
        return FD_ERR_ALIGN;
    const size_t act = (size_t)K * 2, row = (size_t)N * 2;
    const size_t w_bytes = (size_t)N * K / 2, s_bytes = (size_t)N * (K / group) * 2;
    const void *ins[] = {gate, up, qweight, scales, rms_weight};
    const size_t in_bytes[] = {act, act, w_bytes, s_bytes, row};
    // outputs: y, normed, residual_out (== residual allowed), scratch
    const void *outs[] = {y, normed, residual_out, scratch};
    const size_t out_bytes[] = {row, row, row, (size_t)FD_FOLD_SCRATCH_BYTES};
    for (int i = 0; i < 4; ++i) {
        for (int j = 0; j < 5; ++j)
            if (overlaps(outs[i], out_bytes[i], ins[j], in_bytes[j])) return FD_ERR_OVERLAP;
        for (int j = i + 1; j < 4; ++j)
            if (overlaps(outs[i], out_bytes[i], outs[j], out_bytes[j])) return FD_ERR_OVERLAP;
        if (outs[i] != residual_out && overlaps(outs[i], out_bytes[i], residual, row))
            return FD_ERR_OVERLAP;
    }
    if (residual_out != residual && overlaps(residual_out, row, residual, row)) return FD_ERR_OVERLAP;
    if (fake_launch_failure()) return from_cuda(cudaErrorLaunchOutOfResources);
    cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
    const int path = g_gemv_path.load(std::memory_order_relaxed);
    if (path == FD_GEMV_AUTO || path == FD_GEMV_BULK) {
        unsigned char *sc = static_cast<unsigned char *>(scratch);
        const FoldArgs fold{static_cast<const uint16_t *>(residual),
                            static_cast<uint16_t *>(residual_out),
                            static_cast<const uint16_t *>(rms_weight),
                            static_cast<uint16_t *>(normed),
                            reinterpret_cast<float *>(sc + kFoldPartialsOffset),
                            reinterpret_cast<unsigned *>(sc), eps, 1.0f / (float)N};
        bool launched = false;
        cudaError_t err = launch_gemv_tma(gate, up, qweight, scales, nullptr,
                                          GemvOut{y, nullptr, N, N}, 1, K, N, group, st_,
                                          &launched, &fold);
        if (err != cudaSuccess || launched) return from_cuda(err);
    }
    // the GEMV on the selected kernel, then the separate add-RMSNorm kernel
    st = swiglu_gemv(gate, up, qweight, scales, nullptr, y, 1, K, N, group, stream);
    if (st != FD_OK) return st;
    return from_cuda(launch_add_rmsnorm(y, residual, rms_weight, eps, normed, residual_out, 1, N,
                                        st_));
}

int fd_swiglu_w4a16_gemv_add_rmsnorm_noalloc(const void *gate, const void *up,
                                             const void *qweight, const void *scales, void *y,
                                             const void *residual, const void *rms_weight,
                                             float eps, void *normed, void *residual_out, int K,
                                             int N, int group, fd_stream_t stream) {
    const int sz = check_w4_sizes(1, K, N, group);
    if (sz == kEmpty) return FD_OK;
    if (!(eps >= 0.0f) || !std::isfinite(eps) || N % 8 != 0) return FD_ERR_SHAPE;
    if (!gate || !up || !y || !residual || !rms_weight || !normed || !residual_out)
        return FD_ERR_NULL;
    if (sz != FD_OK) return sz;
    int st = check_w4_layout(qweight, scales, K, N, group);
    if (st != FD_OK) return st;
    if (!aligned16(gate) || !aligned16(up) || !aligned16(y) || !aligned16(residual) ||
        !aligned16(rms_weight) || !aligned16(normed) || !aligned16(residual_out))
        return FD_ERR_ALIGN;
    const size_t act = (size_t)K * 2, row = (size_t)N * 2;
    const size_t w_bytes = (size_t)N * K / 2, s_bytes = (size_t)N * (K / group) * 2;
    const void *ins[] = {gate, up, qweight, scales, rms_weight};
    const size_t in_bytes[] = {act, act, w_bytes, s_bytes, row};
    const void *outs[] = {y, normed, residual_out};
    for (int i = 0; i < 3; ++i) {
        for (int j = 0; j < 5; ++j)
            if (overlaps(outs[i], row, ins[j], in_bytes[j])) return FD_ERR_OVERLAP;
        for (int j = i + 1; j < 3; ++j)
            if (overlaps(outs[i], row, outs[j], row)) return FD_ERR_OVERLAP;
        if (outs[i] != residual_out && overlaps(outs[i], row, residual, row)) return FD_ERR_OVERLAP;
    }
    if (residual_out != residual && overlaps(residual_out, row, residual, row)) return FD_ERR_OVERLAP;
    if (fake_launch_failure()) return from_cuda(cudaErrorLaunchOutOfResources);
    cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
    const int path = g_gemv_path.load(std::memory_order_relaxed);
    if (path == FD_GEMV_AUTO || path == FD_GEMV_BULK) {
        bool launched = false, too_big = false;
        cudaError_t err = launch_gemv_fold_noalloc(gate, up, qweight, scales, y, residual,
                                                   rms_weight, eps, normed, residual_out, K, N,
                                                   group, st_, &launched, &too_big);
        if (err != cudaSuccess || launched) return from_cuda(err);
        if (too_big) return FD_ERR_UNSUPPORTED;
    }
    // the selected GEMV kernel, then the separate add-RMSNorm kernel: no scratch at all
    st = swiglu_gemv(gate, up, qweight, scales, nullptr, y, 1, K, N, group, stream);
    if (st != FD_OK) return st;
    return from_cuda(launch_add_rmsnorm(y, residual, rms_weight, eps, normed, residual_out, 1, N,
                                        st_));
}

int fd_w4a16_gate_up_gemv(const void *x, const void *qweight, const void *scales,
                          void *gate_out, void *up_out, int M, int K, int I, int group,
                          fd_stream_t stream) {
    if (I < 0) return FD_ERR_SHAPE;
    if (I > (INT32_MAX - 1) / 2) return FD_ERR_UNSUPPORTED;
    const int N = 2 * I;  // gate rows, then up rows
    const int sz = check_w4_sizes(M, K, N, group);
    if (sz == kEmpty) return FD_OK;
    if (!x || !gate_out || !up_out) return FD_ERR_NULL;
    if (sz != FD_OK) return sz;
    int st = check_w4_layout(qweight, scales, K, N, group);
    if (st != FD_OK) return st;
    if (!aligned16(x) || !aligned16(gate_out) || !aligned16(up_out)) return FD_ERR_ALIGN;
    const size_t x_bytes = (size_t)M * K * 2;
    const size_t o_bytes = (size_t)M * I * 2;
    const size_t w_bytes = (size_t)N * K / 2;
    const size_t s_bytes = (size_t)N * (K / group) * 2;
    for (const void *o : {static_cast<const void *>(gate_out), static_cast<const void *>(up_out)}) {
        if (overlaps(o, o_bytes, x, x_bytes) || overlaps(o, o_bytes, qweight, w_bytes) ||
            overlaps(o, o_bytes, scales, s_bytes))
            return FD_ERR_OVERLAP;
    }
    if (overlaps(gate_out, o_bytes, up_out, o_bytes)) return FD_ERR_OVERLAP;
    if (fake_launch_failure()) return from_cuda(cudaErrorLaunchOutOfResources);
    cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
    const GemvOut o{gate_out, up_out, I, I};
    const int path = g_gemv_path.load(std::memory_order_relaxed);
    if (path != FD_GEMV_CUDA_CORE) {  // the bulk-copy kernel where its layout rules hold
        bool launched = false;
        cudaError_t err = launch_gemv_tma(x, nullptr, qweight, scales, nullptr, o, M, K, N,
                                          group, st_, &launched);
        if (err != cudaSuccess || launched) return from_cuda(err);
    }
    return from_cuda(launch_gemv_cc(x, nullptr, qweight, scales, nullptr, o, M, K, N, group, st_));
}

int fd_nvfp4_scaled_mm(const void *x, const void *x_sf, const void *w, const void *w_sf,
                       const float *alpha, void *out, int M, int K, int N, fd_stream_t stream) {
    if (M < 0 || N < 0 || K <= 0 || K % kNfStageK != 0) return FD_ERR_SHAPE;
    if (M > FD_MAX_M || K > FD_NVFP4_MAX_K) return FD_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return FD_OK;  // empty: nothing read or written
    if (!x || !x_sf || !w || !w_sf || !alpha || !out) return FD_ERR_NULL;
    if (!aligned16(x) || !aligned16(x_sf) || !aligned16(w) || !aligned16(w_sf) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(alpha) & 3u) != 0)
        return FD_ERR_ALIGN;
    const size_t out_bytes = (size_t)M * N * 2;
    if (overlaps(out, out_bytes, x, (size_t)M * K / 2) ||
        overlaps(out, out_bytes, x_sf, (size_t)M * K / 16) ||
        overlaps(out, out_bytes, w, (size_t)N * K / 2) ||
        overlaps(out, out_bytes, w_sf, (size_t)N * K / 16) || overlaps(out, out_bytes, alpha, 4))
        return FD_ERR_OVERLAP;
    if (fake_launch_failure()) return from_cuda(cudaErrorLaunchOutOfResources);
    return from_cuda(launch_nvfp4_mm(x, x_sf, w, w_sf, alpha, out, M, K, N,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int fd_debug_plan_nvfp4(int M, int K, int N, int smem_budget, int *plan) {
    if (!plan) return FD_ERR_NULL;
    Nvfp4Plan p{};
    if (!plan_nvfp4(M, K, N, smem_budget, &p)) return FD_ERR_UNSUPPORTED;
    const int v[13] = {p.split, p.s_total, p.max_stages, p.npad, p.n_tiles, p.tmem_cols,
                       p.cols_own, (int)p.sf_row, (int)p.off_x, (int)p.off_wsf, (int)p.off_xsf,
                       (int)p.recv_bytes, (int)p.smem};
    for (int i = 0; i < 13; ++i) plan[i] = v[i];
    return FD_OK;
}

int fd_copy(void *dst, const void *src, size_t bytes, fd_stream_t stream) {
    if (bytes == 0) return FD_OK;  // empty: nothing read or written
    if (!dst || !src) return FD_ERR_NULL;
    if (bytes % 16 != 0) return FD_ERR_SHAPE;
    if (!aligned16(dst) || !aligned16(src)) return FD_ERR_ALIGN;
    if (overlaps(dst, bytes, src, bytes)) return FD_ERR_OVERLAP;
    if (fake_launch_failure()) return from_cuda(cudaErrorLaunchOutOfResources);
    return from_cuda(launch_copy(dst, src, bytes, reinterpret_cast<cudaStream_t>(stream)));
}

int fd_copy_rows(void *dst, size_t dst_pitch, const void *src, size_t src_pitch,
                 size_t row_bytes, size_t rows, fd_stream_t stream) {
    if (row_bytes == 0 || rows == 0) return FD_OK;  // empty: nothing read or written
    if (!dst || !src) return FD_ERR_NULL;
    if (row_bytes % 16 != 0 || dst_pitch % 16 != 0 || src_pitch % 16 != 0 ||
        dst_pitch < row_bytes || src_pitch < row_bytes)
        return FD_ERR_SHAPE;
    if (!aligned16(dst) || !aligned16(src)) return FD_ERR_ALIGN;
    // the spans the rows lie in (conservative: no interleaving of the two is allowed)
    if (overlaps(dst, (rows - 1) * dst_pitch + row_bytes, src, (rows - 1) * src_pitch + row_bytes))
        return FD_ERR_OVERLAP;
    if (fake_launch_failure()) return from_cuda(cudaErrorLaunchOutOfResources);
    return from_cuda(launch_copy_rows(dst, dst_pitch, src, src_pitch, row_bytes, rows,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

int fd_debug_plan_gemv(const int *device, int M, int K, int N, int group, int plain, int *plan) {
    if (!device || !plan) return FD_ERR_NULL;
    if (M <= 0 || K <= 0 || N <= 0 || group <= 0 || K % 32 != 0 || K % group != 0)
        return FD_ERR_SHAPE;
    // the bulk-copy kernel's compile-time shape: one activation row per pass with two lanes
    // per 32-k slice at M = 1, else two rows per pass with one lane; 8-row chunks, 8 slots
    const int MB = M == 1 ? 1 : 2;
    TmaPlanInput in{device[0], device[1], device[2], device[3], device[4], device[5],
                    M, K, N, group, MB, MB == 1 ? 2 : 1, 8, 8, plain ? 1 : 0};
    TmaPlan p{};
    if (!plan_gemv_tma(in, &p)) return FD_ERR_UNSUPPORTED;
    const int v[9] = {p.grid, p.rows_base, p.rows_extra, p.S, p.w_rows, p.act_first_stage,
                      p.ring, p.per_sm, (int)p.smem};
    for (int i = 0; i < 9; ++i) plan[i] = v[i];
    return FD_OK;
}

int fd_debug_plan_tc(int M, int K, int N, int group, int smem_budget, int *plan) {
    if (!plan) return FD_ERR_NULL;
    if (M <= 0 || K <= 0 || N <= 0 || group <= 0) return FD_ERR_SHAPE;
    if (!gemv_tc_supported(M, K, N, group) || smem_budget <= 0) return FD_ERR_UNSUPPORTED;
    // the first launch's row block (up to 128 activation rows)
    const int npad = tc_npad(M < 128 ? M : 128);
    int stepk = 0;
    TcPlan p{};
    if (!plan_tc(npad, K / kTcSplit, group, (size_t)smem_budget, &stepk, &p))
        return FD_ERR_UNSUPPORTED;
    const int v[10] = {npad, stepk, p.s_w, p.s_gu, p.s_op, p.sg, (int)p.off_gu, (int)p.off_op,
                       (int)p.off_sc, (int)p.smem};
    for (int i = 0; i < 10; ++i) plan[i] = v[i];
    return FD_OK;
}

int fd_debug_plan_step(const int *device, int hidden, int inter, int group, int *plan) {
    if (!device || !plan) return FD_ERR_NULL;
    if (hidden <= 0 || hidden % 8 != 0 || inter <= 0 || group <= 0) return FD_ERR_SHAPE;
    if (!step_shape_supported(hidden, inter, group)) return FD_ERR_UNSUPPORTED;
    int vpt = 0, threads = 0;
    if (!step_rms_shape(hidden, &vpt, &threads)) return FD_ERR_UNSUPPORTED;
    // the launcher's budget: the opt-in shared memory less the kernel's static shared memory
    const long long budget = (long long)device[1] - (long long)device[4];
    StepPlan p{};
    if (budget <= 0 || !plan_step(device[0], (size_t)budget, inter, hidden, group, &p))
        return FD_ERR_UNSUPPORTED;
    const int v[8] = {p.grid, p.rows_base, p.rows_extra, p.S, p.w_rows, (int)p.smem, vpt, threads};
    for (int i = 0; i < 8; ++i) plan[i] = v[i];
    return FD_OK;
}

int fd_gemv_uses_tensor_cores(int M, int K, int N, int group) {
    if (M <= 0 || K <= 0 || N <= 0 || group <= 0) return 0;
    const int path = g_gemv_path.load(std::memory_order_relaxed);
    const bool wanted = (path == FD_GEMV_AUTO && M >= kTensorCoreMinM) || path == FD_GEMV_TENSOR;
    return wanted && gemv_tc_supported(M, K, N, group) ? 1 : 0;
}

int fd_set_gemv_path(int path) {
    if (path < FD_GEMV_AUTO || path > FD_GEMV_TENSOR) return FD_ERR_UNSUPPORTED;
    g_gemv_path.store(path, std::memory_order_relaxed);
    return FD_OK;
}

int fd_get_gemv_path(void) { return g_gemv_path.load(std::memory_order_relaxed); }

int fd_set_launch_flags(unsigned flags) {
    if (flags & ~(FD_LAUNCH_PDL | FD_LAUNCH_TEST_FAIL | FD_LAUNCH_TEST_WAIT_TIMEOUT))
        return FD_ERR_UNSUPPORTED;
    g_launch_flags.store(flags, std::memory_order_relaxed);
    return FD_OK;
}

unsigned fd_get_launch_flags(void) { return g_launch_flags.load(std::memory_order_relaxed); }

int fd_add_rmsnorm(const void *x, const void *residual, const void *weight, float eps,
                   void *out, void *residual_out, int rows, int hidden, fd_stream_t stream) {
    if (rows < 0 || hidden <= 0 || hidden % 8 != 0) return FD_ERR_SHAPE;
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return FD_ERR_SHAPE;
    if (hidden > FD_MAX_HIDDEN) return FD_ERR_UNSUPPORTED;
    if (rows == 0) return FD_OK;  // empty: nothing read or written
    if (!x || !residual || !weight || !out || !residual_out) return FD_ERR_NULL;
    if (!aligned16(x) || !aligned16(residual) || !aligned16(weight) || !aligned16(out) ||
        !aligned16(residual_out))
        return FD_ERR_ALIGN;
    const size_t bytes = (size_t)rows * hidden * 2;
    const size_t w_bytes = (size_t)hidden * 2;
    // Allowed aliasing: out == x, residual_out == residual (same pointer, in place).
    if (overlaps(out, bytes, residual_out, bytes)) return FD_ERR_OVERLAP;
    if (out != x && (overlaps(out, bytes, x, bytes) || overlaps(out, bytes, residual, bytes)))
        return FD_ERR_OVERLAP;
    if (out == x && overlaps(out, bytes, residual, bytes)) return FD_ERR_OVERLAP;
    if (residual_out != residual && (overlaps(residual_out, bytes, residual, bytes) ||
                                     overlaps(residual_out, bytes, x, bytes)))
        return FD_ERR_OVERLAP;
    if (residual_out == residual && overlaps(residual_out, bytes, x, bytes))
        return FD_ERR_OVERLAP;
    if (overlaps(weight, w_bytes, out, bytes) || overlaps(weight, w_bytes, residual_out, bytes))
        return FD_ERR_OVERLAP;
    if (fake_launch_failure()) return from_cuda(cudaErrorLaunchOutOfResources);
    return from_cuda(launch_add_rmsnorm(x, residual, weight, eps, out, residual_out, rows,
                                        hidden, reinterpret_cast<cudaStream_t>(stream)));
}

int fd_w4_dequant_debug(const void *qweight, const void *scales, float *out, int K, int N,
                        int group, fd_stream_t stream) {
    const int sz = check_w4_sizes(1, K, N, group);
    if (sz == kEmpty) return FD_OK;
    if (!out) return FD_ERR_NULL;
    if (sz != FD_OK) return sz;
    int st = check_w4_layout(qweight, scales, K, N, group);
    if (st != FD_OK) return st;
    if (!aligned16(out)) return FD_ERR_ALIGN;
    const size_t out_bytes = (size_t)N * K * 4;
    if (overlaps(out, out_bytes, qweight, (size_t)N * K / 2) ||
        overlaps(out, out_bytes, scales, (size_t)N * (K / group) * 2))
        return FD_ERR_OVERLAP;
    if (fake_launch_failure()) return from_cuda(cudaErrorLaunchOutOfResources);
    return from_cuda(launch_w4_dequant_debug(qweight, scales, out, K, N, group,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

const char *fd_status_string(int status) {
    switch (status) {
        case FD_OK: return "FD_OK: success";
        case FD_ERR_NULL: return "FD_ERR_NULL: a required pointer is NULL";
        case FD_ERR_SHAPE: return "FD_ERR_SHAPE: a size is invalid (<= 0 or breaks a divisibility rule)";
        case FD_ERR_ALIGN: return "FD_ERR_ALIGN: a pointer is not 16-byte aligned";
        case FD_ERR_UNSUPPORTED: return "FD_ERR_UNSUPPORTED: a size is above the supported maximum";
        case FD_ERR_CUDA: return "FD_ERR_CUDA: the CUDA runtime reported an error";
        case FD_ERR_OVERLAP: return "FD_ERR_OVERLAP: an output overlaps an input in a way the kernel does not allow";
        default: return "fd: unknown status";
    }
}

int fd_decode_mlp_step(const fd_step_layer *layers, int n_layers, const void *x0,
                       void *residual, float eps, int hidden, int inter, int group,
                       void *scratch, fd_stream_t stream) {
    if (!layers || !x0 || !residual || !scratch) return FD_ERR_NULL;
    if (n_layers < 1 || n_layers > FD_STEP_MAX_LAYERS || hidden <= 0 || hidden % 8 != 0 ||
        inter <= 0 || group <= 0 || !(eps >= 0.0f) || !std::isfinite(eps))
        return FD_ERR_SHAPE;
    if (!aligned16(x0) || !aligned16(residual) || !aligned16(scratch) ||
        !aligned16(layers))
        return FD_ERR_ALIGN;
    const size_t row = (size_t)hidden * 2;
    const size_t sync_bytes = FD_STEP_SCRATCH_BYTES(n_layers, hidden);
    if (overlaps(x0, row, residual, row) || overlaps(scratch, sync_bytes, residual, row) ||
        overlaps(scratch, sync_bytes, x0, row))
        return FD_ERR_OVERLAP;
    if (!step_shape_supported(hidden, inter, group)) return FD_ERR_UNSUPPORTED;
    if (fake_launch_failure()) return from_cuda(cudaErrorLaunchOutOfResources);
    bool launched = false;
    cudaError_t err = launch_decode_step(layers, n_layers, x0, residual, eps, hidden, inter, group,
                                         scratch, reinterpret_cast<cudaStream_t>(stream), &launched);
    if (err != cudaSuccess) return from_cuda(err);
    return launched ? FD_OK : FD_ERR_UNSUPPORTED;
}

int fd_device_status(fd_stream_t stream, unsigned *status, int clear) {
    if (!status) return FD_ERR_NULL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // one word per file with bounded waits; pinned so the copies are truly asynchronous
    static thread_local unsigned *words = nullptr;
    if (!words) {
        cudaError_t err = cudaMallocHost(&words, 4 * sizeof(unsigned));
        if (err != cudaSuccess) return from_cuda(err);
    }
    cudaError_t (*const readers[4])(cudaStream_t, unsigned *, bool) = {
        status_gemv_tma, status_gemv_tc, status_nvfp4, status_decode_step};
    for (int i = 0; i < 4; ++i) {
        words[i] = 0;
        cudaError_t err = readers[i](st, &words[i], clear != 0);
        if (err != cudaSuccess) return from_cuda(err);
    }
    cudaError_t err = cudaStreamSynchronize(st);
    if (err != cudaSuccess) return from_cuda(err);
    *status = words[0] | words[1] | words[2] | words[3];
    return FD_OK;
}

int fd_last_cuda_error(void) { return g_last_cuda_error; }

int fd_version(void) { return 1 * 10000 + 0 * 100 + 0; }

}  // extern "C"
