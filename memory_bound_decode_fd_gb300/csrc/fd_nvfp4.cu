// fd_nvfp4.cu - NVFP4 scaled matmul with the fp32 output multiplier folded in, on the
// fifth-generation tensor cores' block-scaled MMA (tcgen05.mma kind::mxf4nvf4).
//
//   out[m, n] = bf16( alpha * sum_k X[m, k] * W[n, k] ),
//   X[m, k] = e2m1(x[m, k]) * e4m3(x_sf[m, k / 16]),  W[n, k] = e2m1(w[n, k]) * e4m3(w_sf[n, k / 16])
//
// Source: "PyTorch folds NVFP4 output scaling into NVGEMM candidates for decode workloads"
// (body and metrics table): a scaled matmul of two packed-FP4 operands with E4M3 1x16
// block scales, whose zero-dimensional fp32 output multiplier is applied inside the GEMM
// instead of by a separate multiplication kernel; decode at batch 64.
//
// Design for GB300:
//   * A CTA owns 128 weight rows (the MMA's M) and a slice of K; the `split` CTAs of a
//     thread-block cluster hold the slices of the same rows and combine their fp32 partial
//     sums through distributed shared memory (no global scratch, one bf16 store per
//     output). The activation rows (the batch, padded to NPAD) are the MMA's N.
//   * The whole K slice of both operands and both scale tiles fit in shared memory, so
//     warp 0 issues every tensor-map copy at once: per 256-k stage one 128-byte-swizzled
//     box of 128 weight rows and one of NPAD activation rows, already in the tensor core's
//     K-major operand layout (no transform on the CUDA cores).
//   * Four warps copy the E4M3 scale factors into tensor memory (tcgen05.st), one 256-k
//     stage at a time: for each K = 64 step, 4 columns for the weights and 4 for the
//     activations; lane l of every 32-lane quarter holds, in column c, the four
//     16-element scales of row l + 32c.
//   * Warp 1 lane 0 issues one block-scaled MMA per K = 64 step (M = 128, N = NPAD) into a
//     TMEM accumulator as each stage's operands and scales are ready, then commits.
//   * The same four warps read the accumulator (lane = weight row), exchange partial sums
//     through the cluster, and the owner of each row range applies alpha (read from device
//     memory, the page's 0-dim multiplier) to the fp32 sum and rounds once to bf16.
//   * Every wait is bounded (fd_tma.cuh); a CTA that gives up still takes part in both
//     cluster barriers and frees its TMEM, and its cluster writes NaN to the outputs.
#include <atomic>

#include <cudaTypedefs.h>

#include "fd_nvfp4_plan.h"
#include "fd_tc.cuh"

namespace fd {
namespace {

constexpr int kNfThreads = 6 * 32;   // producer, MMA, four scale / epilogue warps
constexpr int kNfFirstEpi = 2;

// Bounded wait that ignores the abort flag: used where the CTA must not go on before the
// hardware is done (copies landing, MMAs completing), even after a failure.
__device__ __forceinline__ void nf_wait_hw(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_test_parity(bar, parity) && clock64() - t0 < kWaitLimitCycles) __nanosleep(64);
}

template <int NPAD>
__global__ void __launch_bounds__(kNfThreads, 1)
    nvfp4_mm_kernel(const __grid_constant__ CUtensorMap map_w,
                    const __grid_constant__ CUtensorMap map_x,
                    const __grid_constant__ CUtensorMap map_wsf,
                    const __grid_constant__ CUtensorMap map_xsf, const float *alpha,
                    uint16_t *out, int M, int N, int s_total, uint32_t sf_row, int rows_own,
                    uint32_t tmem_cols, uint32_t off_x, uint32_t off_wsf, uint32_t off_xsf) {
    static_assert(NPAD == 16 || NPAD == 32 || NPAD == 64 || NPAD == 128, "MMA N");
    constexpr uint32_t kXStage = NPAD * kNfStageK / 2;    // activation bytes per stage
    __shared__ __align__(8) uint64_t full_bar[kNfMaxStages];  // a stage's operands
    __shared__ __align__(8) uint64_t sf_ready[kNfMaxStages];  // a stage's scales are in TMEM
    __shared__ __align__(8) uint64_t sf_full, acc_full;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ uint32_t peer_abort[kNfMaxSplit];
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base (128-byte-swizzled tensor-map destinations need it)
    unsigned char *smem = smem_raw + (((smem_u32(smem_raw) + 1023u) & ~1023u) - smem_u32(smem_raw));

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int split = (int)gridDim.x;
    const int n0 = blockIdx.y * kNfRows;
    // this rank's K slice: stages [s_begin, s_end) of the s_total 256-k stages
    const int s_begin = nvfp4_first_stage((int)rank, s_total, split);
    const int S = nvfp4_first_stage((int)rank + 1, s_total, split) - s_begin;
    const int k0 = s_begin * kNfStageK;

    if (tid == 0) {
        for (int s = 0; s < kNfMaxStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&sf_ready[s], 4);
        }
        mbar_init(&sf_full, 1);
        mbar_init(&acc_full, 1);
        abort_flag = 0;
        for (int p = 0; p < kNfMaxSplit; ++p) peer_abort[p] = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // -------------------------------------------------- every copy, issued at once
        if (lane == 0) {
            prefetch_tensormap(&map_w);
            prefetch_tensormap(&map_x);
            prefetch_tensormap(&map_wsf);
            prefetch_tensormap(&map_xsf);
        }
        grid_dep_wait();  // the activations may come from the previous kernel
        grid_dep_launch();
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();  // each weight byte is read once
            const uint64_t pol_x = policy_evict_last();   // every weight tile reads them
            // the scale boxes are max_stages wide: a shorter slice copies a few unused (or
            // out-of-range, zero-filled) columns past its end
            mbar_arrive_expect_tx(&sf_full, (uint32_t)(kNfRows + NPAD) * sf_row);
            tma_load_2d(smem + off_wsf, &map_wsf, k0 / 16, n0, &sf_full, pol_w);
            tma_load_2d(smem + off_xsf, &map_xsf, k0 / 16, 0, &sf_full, pol_x);
            for (int s = 0; s < S; ++s) {
                const int xb = (k0 + s * kNfStageK) / 2;  // byte column, a multiple of 128
                mbar_arrive_expect_tx(&full_bar[s], kNfWStage + kXStage);
                tma_load_2d(smem + (size_t)s * kNfWStage, &map_w, xb, n0, &full_bar[s], pol_w);
                tma_load_2d(smem + off_x + (size_t)s * kXStage, &map_x, xb, 0, &full_bar[s], pol_x);
            }
            // every copy must land before the CTA reuses the memory or exits
            nf_wait_hw(&sf_full, 0);
            for (int s = 0; s < S; ++s) nf_wait_hw(&full_bar[s], 0);
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------- MMA issue
        grid_dep_wait();
        grid_dep_launch();
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_nvf4(kNfRows, NPAD);
            const uint32_t w_base = smem_u32(smem);
            const uint32_t x_base = smem_u32(smem + off_x);
            for (int s = 0; s < S; ++s) {
                if (!mbar_wait_bounded(&sf_ready[s], 0, &abort_flag)) break;
                if (!mbar_wait_bounded(&full_bar[s], 0, &abort_flag)) break;
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < kNfStageK / kNfMmaK; ++j) {
                    const int kb = s * (kNfStageK / kNfMmaK) + j;
                    // a K = 64 step is 32 bytes of each 128-byte operand row
                    const uint64_t ad = smem_desc_sw128(w_base + (uint32_t)s * kNfWStage + 32u * j);
                    const uint64_t bd = smem_desc_sw128(x_base + (uint32_t)s * kXStage + 32u * j);
                    const uint32_t sfa = tmem + kNfSfCol0 + 8u * kb;
                    tc_mma_nvf4(tmem, ad, bd, idesc, sfa, sfa + 4u, (uint32_t)(s | j));
                }
            }
            tc_commit(&acc_full);  // fires once every MMA issued above has completed
        }
        __syncwarp();
    } else {
        // -------------------------------------------------- scale factors into TMEM
        grid_dep_wait();
        grid_dep_launch();
        const uint32_t q = (uint32_t)(warp & 3);  // this warp's TMEM lane quarter
        const bool ok = mbar_wait_bounded(&sf_full, 0, &abort_flag);
        const unsigned char *wsf = smem + off_wsf;
        const unsigned char *xsf = smem + off_xsf;
        const uint32_t lane_addr = tmem + ((32u * q) << 16);
        // One stage (4 K = 64 steps) at a time: a 16-byte load gives a row's scales of all
        // 4 steps, so each lane loads its 4 weight rows and 4 activation rows once per
        // stage (rows 64 bytes apart: at most 4-way bank conflicts), and the MMA thread may
        // start on a stage as soon as its scales are in TMEM.
        for (int s = 0; s < S; ++s) {
            if (ok) {
                uint4 a[4], b[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int r = lane + 32 * c;
                    a[c] = *reinterpret_cast<const uint4 *>(wsf + (size_t)r * sf_row + 16 * s);
                    b[c] = r < NPAD ? *reinterpret_cast<const uint4 *>(xsf + (size_t)r * sf_row + 16 * s)
                                    : make_uint4(0, 0, 0, 0);
                }
                const uint32_t col = kNfSfCol0 + kNfSfColsPerStage * s;  // 8 per K = 64 step
                tmem_st_x4(lane_addr + col + 0u, a[0].x, a[1].x, a[2].x, a[3].x);
                tmem_st_x4(lane_addr + col + 4u, b[0].x, b[1].x, b[2].x, b[3].x);
                tmem_st_x4(lane_addr + col + 8u, a[0].y, a[1].y, a[2].y, a[3].y);
                tmem_st_x4(lane_addr + col + 12u, b[0].y, b[1].y, b[2].y, b[3].y);
                tmem_st_x4(lane_addr + col + 16u, a[0].z, a[1].z, a[2].z, a[3].z);
                tmem_st_x4(lane_addr + col + 20u, b[0].z, b[1].z, b[2].z, b[3].z);
                tmem_st_x4(lane_addr + col + 24u, a[0].w, a[1].w, a[2].w, a[3].w);
                tmem_st_x4(lane_addr + col + 28u, b[0].w, b[1].w, b[2].w, b[3].w);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sf_ready[s]);
        }
        // the accumulator is complete once the MMA thread's commit fires
        if (lane == 0) nf_wait_hw(&acc_full, 0);
        __syncwarp();
        tc_fence_after();
    }

    // ------------------------------------------------------ cluster reduction + store
    // #1: every CTA of the cluster is done with its operand memory (copies landed, MMAs
    // complete), so it can take the partial sums: [src rank][NPAD][rows_own] fp32.
    cluster_sync_all();
    const uint32_t recv = smem_u32(smem);
    if (warp >= kNfFirstEpi) {
        const int q = warp & 3;
        const int r = 32 * q + lane;  // this thread's weight row in the tile
        const int owner = r / rows_own, rr = r % rows_own;
        const uint32_t dst = map_to_rank(recv, (uint32_t)owner);
#pragma unroll 1
        for (int c8 = 0; c8 < NPAD / 8; ++c8) {
            uint32_t v[8];
            tmem_ld_x8(tmem + ((uint32_t)(32 * q) << 16) + 8u * c8, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int j = 8 * c8 + i;
                st_cluster_f32(dst + (uint32_t)(((int)rank * NPAD + j) * rows_own + rr) * 4u,
                               __uint_as_float(v[i]));
            }
        }
    }
    if (tid == 0) {
        for (int p = 0; p < split; ++p)
            st_cluster_u32(map_to_rank(smem_u32(&peer_abort[rank]), (uint32_t)p), (uint32_t)abort_flag);
    }
    __syncwarp();
    // #2: all partial sums and failure flags have arrived.
    cluster_sync_all();
    if (warp >= kNfFirstEpi) {
        grid_dep_wait();  // alpha may be written, and `out` read, by the previous kernel
        const float a = *alpha;
        bool failed = false;
        for (int p = 0; p < split; ++p) failed |= peer_abort[p] != 0;
        const float *rv = reinterpret_cast<const float *>(smem);
        const int et = tid - kNfFirstEpi * 32;
        for (int i = et; i < NPAD * rows_own; i += 4 * 32) {
            const int j = i / rows_own, rr = i % rows_own;
            float acc = 0.f;
            for (int src = 0; src < split; ++src) acc += rv[(src * NPAD + j) * rows_own + rr];
            const int row = (int)rank * rows_own + rr;
            const int n = n0 + row;
            if (j < M && n < N && row < kNfRows) {
                const __nv_bfloat16 y = __float2bfloat16_rn(a * acc);
                out[(size_t)j * N + n] = failed ? (uint16_t)0x7FC0 : *reinterpret_cast<const uint16_t *>(&y);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

// ------------------------------------------------------------------ host side

using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiled encode_fn() {
    static std::atomic<void *> fn{nullptr};
    void *f = fn.load(std::memory_order_acquire);
    if (!f) {
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !f)
            return nullptr;
        fn.store(f, std::memory_order_release);
    }
    return reinterpret_cast<EncodeTiled>(f);
}

// A row-major byte matrix [rows, row_bytes] as a 2D tensor map with boxes of
// box_bytes x box_rows (rows past `rows` read as zero).
bool encode_bytes_2d(CUtensorMap *map, const void *base, uint64_t row_bytes, uint64_t rows,
                     uint32_t box_bytes, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
    EncodeTiled enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {row_bytes, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_bytes, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <int NPAD>
cudaError_t launch_npad(const DeviceInfo &di, const unsigned char *x, const unsigned char *x_sf,
                        const void *w, const void *w_sf, const float *alpha, uint16_t *out,
                        int mc, int K, int N, cudaStream_t stream) {
    static std::atomic<uint64_t> attr_done{0};
    static std::atomic<int> static_smem_cache{-1};
    auto kern = nvfp4_mm_kernel<NPAD>;
    int static_smem = static_smem_cache.load(std::memory_order_relaxed);
    if (static_smem < 0) {
        cudaFuncAttributes fa;
        cudaError_t err = cudaFuncGetAttributes(&fa, kern);
        if (err != cudaSuccess) return err;
        static_smem = (int)fa.sharedSizeBytes;
        static_smem_cache.store(static_smem, std::memory_order_relaxed);
    }
    const int budget = di.max_smem_optin - static_smem;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, budget);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
        attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    Nvfp4Plan p{};
    if (!plan_nvfp4(mc, K, N, budget, &p) || p.npad != NPAD) return cudaErrorInvalidValue;
    CUtensorMap mw, mx, mwsf, mxsf;
    if (!encode_bytes_2d(&mw, w, (uint64_t)K / 2, (uint64_t)N, kNfStageK / 2, kNfRows,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_bytes_2d(&mx, x, (uint64_t)K / 2, (uint64_t)mc, kNfStageK / 2, NPAD,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_bytes_2d(&mwsf, w_sf, (uint64_t)K / 16, (uint64_t)N, p.sf_row, kNfRows,
                         CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_bytes_2d(&mxsf, x_sf, (uint64_t)K / 16, (uint64_t)mc, p.sf_row, NPAD,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    err = launch_kernel(kern, dim3((unsigned)p.split, (unsigned)p.n_tiles), dim3(kNfThreads),
                        (size_t)p.smem, stream, p.split, mw, mx, mwsf, mxsf, alpha, out, mc, N,
                        p.s_total, p.sf_row, p.rows_own, (uint32_t)p.tmem_cols, p.off_x,
                        p.off_wsf, p.off_xsf);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_nvfp4_mm(const void *x, const void *x_sf, const void *w, const void *w_sf,
                            const float *alpha, void *out, int M, int K, int N,
                            cudaStream_t stream) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    // batches above 128 rows run in launches of 128 activation rows; where 128 padded rows
    // do not fit shared memory (K above 12288) in launches of 64
    Nvfp4Plan probe{};
    const int widest = K / kNfStageK < kNfMaxSplit ? K / kNfStageK : kNfMaxSplit;
    const int chunk = plan_nvfp4_split(kNfMaxBatch, K, N, widest, di.max_smem_optin - 1024, &probe)
                          ? kNfMaxBatch
                          : kNfMaxBatch / 2;
    for (int m0 = 0; m0 < M; m0 += chunk) {
        const int mc = M - m0 < chunk ? M - m0 : chunk;
        const unsigned char *xm = static_cast<const unsigned char *>(x) + (size_t)m0 * (K / 2);
        const unsigned char *xsfm = static_cast<const unsigned char *>(x_sf) + (size_t)m0 * (K / 16);
        uint16_t *om = static_cast<uint16_t *>(out) + (size_t)m0 * N;
        const int npad = nvfp4_npad(mc);
        if (npad == 16)
            err = launch_npad<16>(di, xm, xsfm, w, w_sf, alpha, om, mc, K, N, stream);
        else if (npad == 32)
            err = launch_npad<32>(di, xm, xsfm, w, w_sf, alpha, om, mc, K, N, stream);
        else if (npad == 64)
            err = launch_npad<64>(di, xm, xsfm, w, w_sf, alpha, om, mc, K, N, stream);
        else
            err = launch_npad<128>(di, xm, xsfm, w, w_sf, alpha, om, mc, K, N, stream);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

FD_DEFINE_STATUS_ACCESSOR(status_nvfp4)

}  // namespace fd
