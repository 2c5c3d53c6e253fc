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
//   * The same four warps copy the accumulator (lane = weight row, 32 columns per wait) to
//     shared memory as [column][row]; each cluster rank owns a range of output columns
//     (activation rows), and one bulk copy per rank moves that range's partial sums into the
//     owner's shared memory (distributed shared memory, completion on the owner's
//     mbarrier). The owner adds the ranks' partials in rank order, applies alpha (read from
//     device memory, the page's 0-dim multiplier, early in the kernel) and rounds once to
//     bf16.
//   * Thread 0 initialises the barriers and issues every copy before the block-wide
//     barrier, so the copies are in flight while warp 1 allocates the tensor memory.
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
// hardware is done (copies landing, MMAs completing), even after a failure. try_wait
// suspends the thread until the phase completes or a hardware time limit passes.
__device__ __forceinline__ void nf_wait_hw(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_parity(bar, parity) && clock64() - t0 < kWaitLimitCycles) {
    }
}
// The same, returning whether the phase completed (a timeout is recorded in the status word).
__device__ __forceinline__ bool nf_wait_hw_ok(uint64_t *bar, uint32_t parity) {
    nf_wait_hw(bar, parity);
    if (mbar_test_parity(bar, parity)) return true;
    record_wait_timeout();
    return false;
}

// TCOLS, the TMEM columns a CTA allocates (256 or 512, as the launch plan asks), is a
// compile-time constant. (The occupancy API reports one CTA per SM for any kernel that
// allocates tensor memory, whatever the count; on GB300 two CTAs of 256 columns were seen
// resident on one SM at run time, which is what the plan's shared-memory floor allows.)
template <int NPAD, uint32_t TCOLS>
__global__ void __launch_bounds__(kNfThreads, 1)
    nvfp4_mm_kernel(const __grid_constant__ CUtensorMap map_w,
                    const __grid_constant__ CUtensorMap map_x,
                    const __grid_constant__ CUtensorMap map_wsf,
                    const __grid_constant__ CUtensorMap map_xsf, const float *alpha,
                    uint16_t *out, int M, int N, int s_total, uint32_t sf_row, int cols_own,
                    uint32_t off_x, uint32_t off_wsf, uint32_t off_xsf) {
    static_assert(NPAD == 16 || NPAD == 32 || NPAD == 64 || NPAD == 128, "MMA N");
    static_assert(TCOLS == 256 || TCOLS == 512, "TMEM columns");
    constexpr uint32_t kXStage = NPAD * kNfStageK / 2;    // activation bytes per stage
    __shared__ __align__(8) uint64_t full_bar[kNfMaxStages];  // a stage's operands
    __shared__ __align__(8) uint64_t sf_ready[kNfMaxStages];  // a stage's scales are in TMEM
    __shared__ __align__(8) uint64_t sf_full, acc_full;
    __shared__ __align__(8) uint64_t red_bar;  // the other ranks' partial sums have landed
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
    // The cluster reduction: rank p finishes the output columns (activation rows)
    // [p c, (p + 1) c), c = cols_own. Once the operands are dead, shared memory from offset
    // 0 holds `split` receive slots [src rank][c][128 rows] fp32 and then this CTA's
    // accumulator as [column][128 rows] fp32, in which rank p's columns are one contiguous
    // chunk: one bulk copy per rank sends it, completing on that rank's red_bar.
    const uint32_t chunk = (uint32_t)cols_own * kNfRows * 4;
    const uint32_t recv_base = smem_u32(smem);
    const uint32_t acc_base = recv_base + (uint32_t)split * chunk;

    if (tid == 0) {
        prefetch_tensormap(&map_w);
        prefetch_tensormap(&map_x);
        prefetch_tensormap(&map_wsf);
        prefetch_tensormap(&map_xsf);
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&sf_ready[s], 4);
        }
        mbar_init(&sf_full, 1);
        mbar_init(&acc_full, 1);
        mbar_init(&red_bar, 1);
        mbar_arrive_expect_tx(&red_bar, (uint32_t)(split - 1) * chunk);
        abort_flag = 0;
        for (int p = 0; p < kNfMaxSplit; ++p) peer_abort[p] = 0;
        fence_mbar_init();
        // -------------------------------------------------- every copy, issued at once,
        // while warp 1 allocates the tensor memory
        grid_dep_wait();  // the activations may come from the previous kernel
        grid_dep_launch();
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
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, TCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    float out_scale = 0.f;  // alpha, read by the epilogue warps once they may

    if (warp == 0) {
        grid_dep_wait();
        grid_dep_launch();
        if (lane == 0) {  // every copy must land before the CTA reuses the memory or exits
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
        grid_dep_wait();  // alpha may be written, and `out` read, by the previous kernel
        grid_dep_launch();
        out_scale = *alpha;
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
    if (tid == 0) {  // this CTA's failure flag, to every rank
        for (int p = 0; p < split; ++p)
            st_cluster_u32(map_to_rank(smem_u32(&peer_abort[rank]), (uint32_t)p), (uint32_t)abort_flag);
    }
    __syncwarp();
    // #1: every CTA of the cluster is done with its operand memory (copies landed, MMAs
    // complete) and has published its failure flag.
    cluster_sync_all();
    const int mcols = M < NPAD ? M : NPAD;  // columns past the batch are never stored
    if (warp >= kNfFirstEpi) {
        const int q = warp & 3;
        const int r = 32 * q + lane;  // this thread's weight row in the tile (its TMEM lane)
        float *acc_col = reinterpret_cast<float *>(smem + (size_t)split * chunk) + r;
        constexpr int kChunk = NPAD < 32 ? NPAD : 32;
#pragma unroll 1
        for (int c0 = 0; c0 < mcols; c0 += kChunk) {
            uint32_t v[kChunk];
            const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0;
            tmem_ld_x16(ta, v);
            if constexpr (kChunk == 32) tmem_ld_x16(ta + 16u, v + 16);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < kChunk; ++i)  // a warp stores 128 contiguous bytes
                if (c0 + i < mcols) acc_col[(c0 + i) * kNfRows] = __uint_as_float(v[i]);
        }
        fence_proxy_async_smem();  // the stores above, before the bulk copies read them
        named_bar_sync(1, 4 * 32);
        if (tid == kNfFirstEpi * 32) {
            for (int p = 0; p < split; ++p)
                if (p != (int)rank)
                    bulk_s2cluster(map_to_rank(recv_base + rank * chunk, (uint32_t)p),
                                   acc_base + (uint32_t)p * chunk, chunk,
                                   map_to_rank(smem_u32(&red_bar), (uint32_t)p));
        }
        // every other rank's partial sums of this rank's columns
        bool failed = split > 1 && !nf_wait_hw_ok(&red_bar, 0);
        for (int p = 0; p < split; ++p) failed |= peer_abort[p] != 0;
        // lane l finishes rows 4l .. 4l + 3 of the columns j0 + q, j0 + q + 4, ...
        const int j0 = (int)rank * cols_own;
        const int own = mcols - j0 < cols_own ? mcols - j0 : cols_own;
        const int n = n0 + 4 * lane;
        const bool vec = (N & 3) == 0 && n + 3 < N;
        for (int jj = q; jj < own; jj += 4) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};  // partial sums in rank order
#pragma unroll
            for (int src = 0; src < kNfMaxSplit; ++src) {
                if (src < split) {
                    const uint32_t a = src == (int)rank
                        ? acc_base + (uint32_t)(((j0 + jj) * kNfRows + 4 * lane) * 4)
                        : recv_base + (uint32_t)src * chunk + (uint32_t)((jj * kNfRows + 4 * lane) * 4);
                    const uint4 v = lds_v4(a);
                    acc[0] += __uint_as_float(v.x);
                    acc[1] += __uint_as_float(v.y);
                    acc[2] += __uint_as_float(v.z);
                    acc[3] += __uint_as_float(v.w);
                }
            }
            uint16_t y[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                y[e] = failed ? (uint16_t)0x7FC0 : __bfloat16_as_ushort(__float2bfloat16_rn(out_scale * acc[e]));
            uint16_t *o = out + (size_t)(j0 + jj) * N + n;
            if (vec) {
                *reinterpret_cast<uint2 *>(o) = make_uint2((uint32_t)y[0] | ((uint32_t)y[1] << 16),
                                                           (uint32_t)y[2] | ((uint32_t)y[3] << 16));
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (n + e < N) o[e] = y[e];
            }
        }
    }
    // #2: no CTA leaves while a bulk copy may still read from or write to its memory
    // (each rank passes this barrier only after its own copies in have landed).
    __syncwarp();
    cluster_sync_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TCOLS);
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

template <int NPAD, uint32_t TCOLS>
cudaError_t launch_plan(const Nvfp4Plan &p, int budget, const unsigned char *x,
                        const unsigned char *x_sf, const void *w, const void *w_sf,
                        const float *alpha, uint16_t *out, int mc, int K, int N,
                        cudaStream_t stream) {
    static std::atomic<uint64_t> attr_done{0};
    auto kern = nvfp4_mm_kernel<NPAD, TCOLS>;
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
                        p.s_total, p.sf_row, p.cols_own, p.off_x, p.off_wsf, p.off_xsf);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

template <int NPAD>
cudaError_t launch_npad(const DeviceInfo &di, const unsigned char *x, const unsigned char *x_sf,
                        const void *w, const void *w_sf, const float *alpha, uint16_t *out,
                        int mc, int K, int N, cudaStream_t stream) {
    // both column variants declare the same static shared memory
    static std::atomic<int> static_smem_cache{-1};
    int static_smem = static_smem_cache.load(std::memory_order_relaxed);
    if (static_smem < 0) {
        cudaFuncAttributes fa;
        cudaError_t err = cudaFuncGetAttributes(&fa, nvfp4_mm_kernel<NPAD, 512>);
        if (err != cudaSuccess) return err;
        static_smem = (int)fa.sharedSizeBytes;
        static_smem_cache.store(static_smem, std::memory_order_relaxed);
    }
    const int budget = di.max_smem_optin - static_smem;
    Nvfp4Plan p{};
    if (!plan_nvfp4(mc, K, N, budget, &p) || p.npad != NPAD) return cudaErrorInvalidValue;
    if (p.tmem_cols == 256)
        return launch_plan<NPAD, 256>(p, budget, x, x_sf, w, w_sf, alpha, out, mc, K, N, stream);
    return launch_plan<NPAD, 512>(p, budget, x, x_sf, w, w_sf, alpha, out, mc, K, N, stream);
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
