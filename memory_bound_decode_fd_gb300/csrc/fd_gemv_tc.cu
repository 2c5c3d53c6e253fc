// fd_gemv_tc.cu - SwiGLU-prologue W4A16 product for batched decode (M >= 16) on the
// fifth-generation tensor cores (tcgen05.mma, accumulator in tensor memory).
//
// y[m, n] = bf16( [residual[m, n] +] sum_k a[m, k] * w[n, k] ),  a = silu(g) * u,
//           w = q * s[n, k / group]   (the residual: the down projection's residual-add
//           epilogue, added to the fp32 sum before the one rounding)
//
// Sources: "09 - Operator fusion", section 5 (taxonomy item 4, GEMM prologue fusion:
// the int4 weights are dequantised on chip as they stream in; "The fusion boundary
// problem": act = silu(gate) * up feeds act @ W_down); "PyTorch Community Proposes Fusion
// Fix ..." ("Fix proposal": the activation and the dequantised weights are never written
// to memory).
//
// At M = 64 a weight byte feeds 256 flops, at the tensor-core ridge of this GPU, so the
// product runs on the tensor cores while the CUDA cores do the two prologues:
//   * A CTA owns 128 weight rows (the MMA's M) and a quarter of K; the four CTAs of a
//     thread-block cluster hold the four quarters of the same rows and combine their
//     fp32 partial sums through distributed shared memory at the end (no global
//     scratch, one bf16 store per output).
//   * Warp 0 streams int4 weight tiles (128 rows x 256 k: one 128-byte line per row,
//     16 KB) and the CTA's scales with tensor-map bulk copies; warp 1 streams the gate/up
//     tiles (M rows x 64 k) of each 64-k step.
//   * Sixteen worker warps turn each step into MMA operands in shared memory (eight
//     for each operand, so the ALU-heavy and the MUFU-heavy work interleave):
//       A = bf16(q * s) for the 128 x 64 weight tile (packed bf16x2 arithmetic: the
//           nibble is placed in the mantissa of 128.0, 136 is subtracted exactly and the
//           product with the group scale is rounded once), and
//       B = bf16(silu(g) * u) for the M x 64 activation tile (fp32, tanh form of silu).
//     Both use the same order of k inside each 8-k core matrix (k0 k4 k1 k5 k2 k6 k3 k7),
//     which leaves the dot product unchanged.
//   * Warp 2 lane 0 issues four tcgen05.mma (M = 128, N = M padded, K = 16) per step
//     into one TMEM accumulator and returns the operand stage through tcgen05.commit.
//   * Every wait is bounded (fd_tma.cuh); a CTA that gives up still takes part in both
//     cluster barriers, frees its TMEM, and its cluster writes NaN to the outputs.
#include <atomic>

#include <cudaTypedefs.h>

#include "fd_gemv_common.cuh"
#include "fd_gemv_tc_plan.h"
#include "fd_tc.cuh"

namespace fd {
namespace {

constexpr int kTcFirstWorker = 3;            // warps 0, 1, 2: weights, gate/up, MMA
constexpr int kTcDequantWarps = 8;           // then the A-operand (weight) warps
constexpr int kTcSiluWarps = 8;              // then the B-operand (activation) warps
constexpr int kTcFirstSilu = kTcFirstWorker + kTcDequantWarps;
constexpr int kTcThreads = (kTcFirstSilu + kTcSiluWarps) * 32;
constexpr int kTcSiluThreads = kTcSiluWarps * 32;
constexpr int kTcEpilogueThreads = kTcDequantWarps * 32;  // the dequant warps
constexpr int kTcMaxStages = 16;
constexpr uint32_t kCoreBytes = 128;                       // 8 rows x 16 bytes

// Bias of the nibble trick: bf16 0x4300 | u is 128 + u, and u = q + 8.
constexpr uint32_t kMagic136x2 = 0x43084308u;

// Bounded wait that ignores the abort flag: used where the CTA must not go on before the
// hardware is done (copies landing, MMAs completing), even after a failure.
__device__ __forceinline__ void wait_parity_hw(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_test_parity(bar, parity) && clock64() - t0 < kWaitLimitCycles) __nanosleep(64);
}

template <int NPAD, int STEPK>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemv_tc_kernel(const __grid_constant__ CUtensorMap map_w,
                   const __grid_constant__ CUtensorMap map_s,
                   const __grid_constant__ CUtensorMap map_g,
                   const __grid_constant__ CUtensorMap map_u, const uint16_t *residual,
                   uint16_t *out, int M, int N, int group, int k_cta, int s_w, int s_gu, int s_op,
                   uint32_t off_gu, uint32_t off_op, uint32_t off_sc, int sg) {
    static_assert(NPAD % 16 == 0 && NPAD >= 16 && NPAD <= 128, "N of the MMA");
    static_assert(STEPK == 64 || STEPK == 128, "k per step");
    constexpr int kCols = NPAD < 32 ? 32 : NPAD;  // TMEM columns (power of two)
    constexpr int kBoxes = STEPK / kTcGuBoxK;     // gate (or up) boxes per step
    constexpr uint32_t kGuTile = NPAD * 128;      // one box: NPAD x 64 bf16
    constexpr uint32_t kGuStage = 2 * kBoxes * kGuTile;  // gate boxes, then up boxes
    constexpr uint32_t kATileBytes = kTcRows * STEPK * 2;  // bf16 A tile
    constexpr uint32_t kGroupBytes = (STEPK / 8) * kCoreBytes;  // 8-row group of a tile
    constexpr uint32_t kOpStage = kATileBytes + NPAD * STEPK * 2;
    constexpr int kStepsPerWTile = kTcWTileK / STEPK;
    constexpr int kChunks = STEPK / 64;           // 32-k weight chunks per thread per step
    constexpr int kHalf = NPAD / 2;               // accumulator columns per epilogue warp

    __shared__ __align__(8) uint64_t w_full[kTcMaxStages], w_empty[kTcMaxStages];
    __shared__ __align__(8) uint64_t gu_full[kTcMaxStages], gu_empty[kTcMaxStages];
    __shared__ __align__(8) uint64_t op_full[kTcMaxStages], op_empty[kTcMaxStages];
    __shared__ __align__(8) uint64_t sc_full, acc_full;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ uint32_t peer_abort[kTcSplit];
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base (swizzled tensor-map destinations need it).
    unsigned char *smem = smem_raw + (((smem_u32(smem_raw) + 1023u) & ~1023u) - smem_u32(smem_raw));

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int n0 = blockIdx.y * kTcRows;
    const int k0 = (int)rank * k_cta;
    const int n_steps = k_cta / STEPK;
    const int g_op = s_op / 2;  // operand stages per commit (the ring has two halves)
    const int x0_scale = (k0 / group) & ~7;

    if (tid == 0) {
        for (int s = 0; s < kTcMaxStages; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_empty[s], kTcDequantWarps);
            mbar_init(&gu_full[s], 1);
            mbar_init(&gu_empty[s], kTcSiluWarps);
            mbar_init(&op_full[s], kTcDequantWarps + kTcSiluWarps);
            mbar_init(&op_empty[s], 1);
        }
        mbar_init(&sc_full, 1);
        mbar_init(&acc_full, 1);
        abort_flag = 0;
        for (int p = 0; p < kTcSplit; ++p) peer_abort[p] = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(&tmem_slot, kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    grid_dep_launch();

    // The three single-issue roles run their loops with the whole warp (warp-uniform
    // values, no divergent single-thread path); lane 0 waits and issues, and a shuffle
    // keeps the warp's decision uniform.
    if (warp == 0) {
        // -------------------------------------------------- weights + scales (constant)
        const uint64_t pol_w = policy_evict_first();
        if (lane == 0) {
            prefetch_tensormap(&map_w);
            prefetch_tensormap(&map_s);
        }
        // Weight traffic ahead of the gate/up copies would delay them (measured on the
        // decode step with the CUDA-core kernel), so the weights also wait for the previous
        // kernel under programmatic dependent launch.
        grid_dep_wait();
        if (lane == 0) {
            mbar_arrive_expect_tx(&sc_full, (uint32_t)kTcRows * sg * 2);
            tma_load_2d(smem + off_sc, &map_s, x0_scale, n0, &sc_full, pol_w);
        }
        int s = 0, round = 0, issued = 0;
        const int n_tiles = k_cta / kTcWTileK;
        for (int t = 0; t < n_tiles; ++t) {
            bool ok = true;
            if (lane == 0 && round > 0) ok = mbar_wait_bounded(&w_empty[s], (round - 1) & 1, &abort_flag);
            if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&w_full[s], kWStageBytes);
                tma_load_2d(smem + (size_t)s * kWStageBytes, &map_w, (k0 + t * kTcWTileK) / 2, n0,
                            &w_full[s], pol_w);
            }
            issued = t + 1;
            if (++s == s_w) { s = 0; ++round; }
        }
        if (lane == 0) {
            for (int t = issued > s_w ? issued - s_w : 0; t < issued; ++t)
                wait_parity_hw(&w_full[t % s_w], (t / s_w) & 1);
            wait_parity_hw(&sc_full, 0);
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------- gate / up tiles
        if (lane == 0) {
            prefetch_tensormap(&map_g);
            prefetch_tensormap(&map_u);
        }
        grid_dep_wait();  // gate/up may be written by the previous kernel
        const uint64_t pol = policy_evict_last();  // every n-tile re-reads them
        int s = 0, round = 0, issued = 0;
        for (int t = 0; t < n_steps; ++t) {
            bool ok = true;
            if (lane == 0 && round > 0) ok = mbar_wait_bounded(&gu_empty[s], (round - 1) & 1, &abort_flag);
            if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
            if (lane == 0) {
                unsigned char *st = smem + off_gu + (size_t)s * kGuStage;
                mbar_arrive_expect_tx(&gu_full[s], kGuStage);
#pragma unroll
                for (int bx = 0; bx < kBoxes; ++bx) {
                    const int kx = k0 + t * STEPK + bx * kTcGuBoxK;
                    tma_load_2d(st + bx * kGuTile, &map_g, kx, 0, &gu_full[s], pol);
                    tma_load_2d(st + (kBoxes + bx) * kGuTile, &map_u, kx, 0, &gu_full[s], pol);
                }
            }
            issued = t + 1;
            if (++s == s_gu) { s = 0; ++round; }
        }
        if (lane == 0) {
            for (int t = issued > s_gu ? issued - s_gu : 0; t < issued; ++t)
                wait_parity_hw(&gu_full[t % s_gu], (t / s_gu) & 1);
        }
        __syncwarp();
    } else if (warp == 2) {
        // -------------------------------------------------- MMA issue
        // One thread (fastest measured issue loop). The operand ring is released in two
        // halves of g_op stages: one tcgen05.commit per half instead of one per stage (a
        // commit costs the issuing thread about as much as four MMAs).
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kTcRows, NPAD);
            // Descriptors of stage 0, first K = 16 step; the start-address field (bits 0-13,
            // address / 16) advances by 2 core matrices per step and by a stage per stage.
            const uint32_t a0 = smem_u32(smem + off_op);
            const uint64_t adesc0 = smem_desc_interleaved(a0, kCoreBytes, kGroupBytes);
            const uint64_t bdesc0 = smem_desc_interleaved(a0 + kATileBytes, kCoreBytes, kGroupBytes);
            constexpr uint64_t kStepField = (2 * kCoreBytes) >> 4;
            constexpr uint64_t kStageField = kOpStage >> 4;
            uint64_t ad = adesc0, bd = bdesc0;
            int s = 0, phase = 0, gpos = 0, gcount = 0;
            for (int t = 0; t < n_steps; ++t) {
                if (!mbar_wait_bounded(&op_full[s], phase, &abort_flag)) break;
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < STEPK / 16; ++j)
                    tc_mma_f16(tmem, ad + j * kStepField, bd + j * kStepField, idesc, (t | j) != 0);
                if (++gpos == g_op || t == n_steps - 1) {
                    tc_commit(&op_empty[gcount & 1]);
                    gpos = 0;
                    ++gcount;
                }
                if (++s == s_op) {
                    s = 0;
                    phase ^= 1;
                    ad = adesc0;
                    bd = bdesc0;
                } else {
                    ad += kStageField;
                    bd += kStageField;
                }
            }
            tc_commit(&acc_full);  // fires once every MMA issued above has completed
        }
        __syncwarp();
    } else if (warp < kTcFirstSilu) {
        // -------------------------------------------------- dequant warps: A operand
        // Every shared-memory address below is a 32-bit shared-window address; the stage
        // addresses advance with the ring instead of being recomputed.
        const int wt = tid - kTcFirstWorker * 32;
        const uint32_t key = opaque_u32(kMagic136x2);
        const uint32_t magic = opaque_u32(kMagic136x2);
        const int row = wt & (kTcRows - 1);  // weight row and k half of each step
        const int h = wt >> 7;
        // 128-byte swizzle of the tensor-map copy: 16-byte chunk c of row r sits at c ^ (r & 7);
        // this thread's chunks of step q of a tile: 2 q kChunks + h kChunks + j
        const uint32_t w_row0 = smem_u32(smem) + row * 128;
        uint32_t chunk_off[kStepsPerWTile][kChunks];
#pragma unroll
        for (int q = 0; q < kStepsPerWTile; ++q)
#pragma unroll
            for (int j = 0; j < kChunks; ++j)
                chunk_off[q][j] = ((uint32_t)(2 * q * kChunks + h * kChunks + j) ^ (row & 7)) << 4;
        const uint32_t a_row0 = smem_u32(smem + off_op) + (row >> 3) * kGroupBytes + (row & 7) * 16 +
                                h * (STEPK / 16) * kCoreBytes;
        // the group scale of this thread's k range (STEPK / 2 k, never across a group: group is
        // a multiple of 64 and the range starts at a multiple of STEPK / 2)
        int gk = k0 % group + h * (STEPK / 2);
        uint32_t sc_at = smem_u32(smem + off_sc) +
                         (uint32_t)(row * sg + (k0 / group - x0_scale) + gk / group) * 2;
        gk %= group;
        const uint32_t w_full0 = smem_u32(&w_full[0]), w_empty0 = smem_u32(&w_empty[0]);
        const uint32_t op_full0 = smem_u32(&op_full[0]), op_empty0 = smem_u32(&op_empty[0]);
        bool ok = mbar_wait_bounded(&sc_full, 0, &abort_flag);
        int ws = 0, wph = 0, os = 0, gpos = 0, gcount = 0;
        uint32_t w_at = w_row0, a_at = a_row0;
        for (int t = 0; t < n_steps && ok; ++t) {
            const int wsub = t & (kStepsPerWTile - 1);
            // entering a ring half: wait for the commit of its previous use
            ok = (wsub != 0 || mbar_wait_bounded_at(w_full0 + 8 * ws, wph, &abort_flag)) &&
                 (gpos != 0 || gcount < 2 ||
                  mbar_wait_bounded_at(op_empty0 + 8 * (gcount & 1), ((gcount >> 1) - 1) & 1,
                                       &abort_flag));
            if (!ok) break;
            uint4 wv[kChunks];
#pragma unroll
            for (int j = 0; j < kChunks; ++j) wv[j] = lds_v4(w_at + chunk_off[wsub][j]);
            const uint32_t sc = lds_u16(sc_at);
            const uint32_t s2 = sc | (sc << 16);
#pragma unroll
            for (int j = 0; j < kChunks; ++j) {
                const uint32_t wd[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    // pairs (k_j, k_j+4) of the word's 8 k: 136 + q as bf16, exact
                    const uint32_t w = wd[i];
                    const uint32_t t0 = mask_xor<0x000F000Fu>(w, key);
                    const uint32_t t1 = mask_xor<0x000F000Fu>(w >> 4, key);
                    const uint32_t t2 = mask_xor<0x000F000Fu>(w >> 8, key);
                    const uint32_t t3 = mask_xor<0x000F000Fu>(w >> 12, key);
                    uint4 o;
                    o.x = bf16x2_mul(bf16x2_sub(t0, magic), s2);
                    o.y = bf16x2_mul(bf16x2_sub(t1, magic), s2);
                    o.z = bf16x2_mul(bf16x2_sub(t2, magic), s2);
                    o.w = bf16x2_mul(bf16x2_sub(t3, magic), s2);
                    sts_v4(a_at + (4 * j + i) * kCoreBytes, o);
                }
            }
            // generic writes of A before the tensor core reads them; generic reads of the
            // weight stage before the next bulk copy overwrites it
            fence_proxy_async_smem();
            __syncwarp();
            const bool tile_done = (wsub == kStepsPerWTile - 1);
            if (lane == 0) {
                if (tile_done) mbar_arrive_at(w_empty0 + 8 * ws);
                mbar_arrive_at(op_full0 + 8 * os);
            }
            if (tile_done) {
                if (++ws == s_w) { ws = 0; wph ^= 1; w_at = w_row0; } else { w_at += kWStageBytes; }
            }
            if (++os == s_op) { os = 0; a_at = a_row0; } else { a_at += kOpStage; }
            if (++gpos == g_op) { gpos = 0; ++gcount; }
            for (gk += STEPK; gk >= group; gk -= group) sc_at += 2;
        }
        __syncwarp();
    } else {
        // -------------------------------------------------- SwiGLU warps: B operand
        constexpr int kC = STEPK / 8;                 // 16-byte chunks per row of a step
        constexpr int kCBits = STEPK == 128 ? 4 : 3;
        constexpr int kItems = (NPAD * kC + kTcSiluThreads - 1) / kTcSiluThreads;
        const int st = tid - kTcFirstSilu * 32;
        const float2 half2 = make_float2(0.5f, 0.5f);
        // lanes 0..7 take rows 0..7 of one core matrix: conflict-free reads (128-byte
        // swizzle: chunk c of row m at c ^ (m & 7)) and writes
        uint32_t src_off[kItems], dst_off[kItems];
        bool active[kItems];
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            const int item = st + j * kTcSiluThreads;
            const int m = (item & 7) | ((item >> (3 + kCBits)) << 3);
            const int c = (item >> 3) & (kC - 1);
            active[j] = item < NPAD * kC;
            // box c / 8 of the step, chunk c % 8 of its 128-byte row
            src_off[j] = (c >> 3) * kGuTile + m * 128 + (((c & 7) ^ (m & 7)) << 4);
            dst_off[j] = (m >> 3) * kGroupBytes + c * kCoreBytes + (m & 7) * 16;
        }
        const uint32_t g_row0 = smem_u32(smem + off_gu);
        const uint32_t b_row0 = smem_u32(smem + off_op) + kATileBytes;
        const uint32_t gu_full0 = smem_u32(&gu_full[0]), gu_empty0 = smem_u32(&gu_empty[0]);
        const uint32_t op_full0 = smem_u32(&op_full[0]), op_empty0 = smem_u32(&op_empty[0]);
        bool ok = true;
        int gs = 0, gph = 0, os = 0, gpos = 0, gcount = 0;
        uint32_t g_at = g_row0, b_at = b_row0;
        for (int t = 0; t < n_steps && ok; ++t) {
            ok = mbar_wait_bounded_at(gu_full0 + 8 * gs, gph, &abort_flag) &&
                 (gpos != 0 || gcount < 2 ||
                  mbar_wait_bounded_at(op_empty0 + 8 * (gcount & 1), ((gcount >> 1) - 1) & 1,
                                       &abort_flag));
            if (!ok) break;
#pragma unroll
            for (int j = 0; j < kItems; ++j) {
                if (active[j]) {
                    const uint4 gv = lds_v4(g_at + src_off[j]);
                    const uint4 uv = lds_v4(g_at + kBoxes * kGuTile + src_off[j]);
                    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
                    const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
                    float2 a[4];  // a[i] = (element 2i, element 2i + 1)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        // silu(g) u = (g u / 2)(1 + tanh(g / 2)), two elements at a time
                        const float2 hv = __fmul2_rn(make_float2(bf16lo(gw[i]), bf16hi(gw[i])), half2);
                        const float2 p = __fmul2_rn(hv, make_float2(bf16lo(uw[i]), bf16hi(uw[i])));
                        const float2 th = make_float2(tanh_approx(hv.x), tanh_approx(hv.y));
                        a[i] = __ffma2_rn(p, th, p);
                    }
                    uint4 o;  // k order 0 4 1 5 2 6 3 7, as the dequantised weights
                    o.x = pack_bf16x2(a[0].x, a[2].x);
                    o.y = pack_bf16x2(a[0].y, a[2].y);
                    o.z = pack_bf16x2(a[1].x, a[3].x);
                    o.w = pack_bf16x2(a[1].y, a[3].y);
                    sts_v4(b_at + dst_off[j], o);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_at(gu_empty0 + 8 * gs);
                mbar_arrive_at(op_full0 + 8 * os);
            }
            if (++gs == s_gu) { gs = 0; gph ^= 1; g_at = g_row0; } else { g_at += kGuStage; }
            if (++os == s_op) { os = 0; b_at = b_row0; } else { b_at += kOpStage; }
            if (++gpos == g_op) { gpos = 0; ++gcount; }
        }
        __syncwarp();
    }

    // ------------------------------------------------------ epilogue
    uint32_t v[kHalf];
    const bool worker = warp >= kTcFirstWorker && warp < kTcFirstSilu;
    const int quarter = warp & 3;                       // TMEM lanes 32q .. 32q + 31
    const int col0 = ((warp - kTcFirstWorker) >> 2) * kHalf;
    if (worker) {
        wait_parity_hw(&acc_full, 0);
        __syncwarp();
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kHalf / 8; ++c) {
            uint32_t r[8];
            tmem_ld_x8(tmem + ((uint32_t)(32 * quarter) << 16) + col0 + 8 * c, r);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[8 * c + i] = r[i];
        }
        tmem_ld_wait();
    }
    tc_fence_before();
    __syncwarp();
    // #1: every CTA of the cluster is done with its rings (copies landed, MMAs complete),
    // so the ring memory can take the partial sums.
    cluster_sync_all();
    const uint32_t recv = smem_u32(smem + off_gu);  // [src rank][NPAD][32] fp32
    if (worker) {
        const uint32_t dst = map_to_rank(recv, (uint32_t)quarter);
#pragma unroll
        for (int j = 0; j < kHalf; ++j)
            st_cluster_f32(dst + (((rank * NPAD) + col0 + j) * 32 + lane) * 4,
                           __uint_as_float(v[j]));
    }
    if (tid == 0) {
        for (int p = 0; p < kTcSplit; ++p)
            st_cluster_u32(map_to_rank(smem_u32(&peer_abort[rank]), (uint32_t)p),
                           (uint32_t)abort_flag);
    }
    __syncwarp();
    // #2: all partial sums and failure flags have arrived.
    cluster_sync_all();
    if (worker) {
        grid_dep_wait();  // the previous kernel in the stream may still use `out`
        const float *rv = reinterpret_cast<const float *>(smem + off_gu);
        const bool failed = (peer_abort[0] | peer_abort[1] | peer_abort[2] | peer_abort[3]) != 0;
        const int wt = tid - kTcFirstWorker * 32;
        for (int i = wt; i < M * 16; i += kTcEpilogueThreads) {
            const int m = i >> 4, rp = (i & 15) * 2;
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int src = 0; src < kTcSplit; ++src) {
                const float2 p = *reinterpret_cast<const float2 *>(rv + ((src * NPAD) + m) * 32 + rp);
                s0 += p.x;
                s1 += p.y;
            }
            const size_t oi = (size_t)m * N + n0 + 32 * rank + rp;
            if (residual) {
                const uint32_t r = *reinterpret_cast<const uint32_t *>(residual + oi);
                s0 += bf16lo(r);
                s1 += bf16hi(r);
            }
            const uint32_t o = failed ? 0x7FC07FC0u : pack_bf16x2(s0, s1);
            *reinterpret_cast<uint32_t *>(out + oi) = o;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kCols);
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

bool encode_2d(CUtensorMap *map, CUtensorMapDataType type, const void *base, uint64_t dim0,
               uint64_t dim1, uint64_t row_bytes, uint32_t box0, uint32_t box1,
               CUtensorMapSwizzle swizzle) {
    EncodeTiled enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {dim0, dim1};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box0, box1};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, type, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One kernel instantiation: its cached static shared memory and opt-in attribute.
template <int NPAD, int STEPK>
struct TcKernel {
    static cudaError_t prepare(const DeviceInfo &di, size_t *budget) {
        static std::atomic<int> static_smem_cache{-1};
        static std::atomic<uint64_t> attr_done{0};
        auto kern = gemv_tc_kernel<NPAD, STEPK>;
        int static_smem = static_smem_cache.load(std::memory_order_relaxed);
        if (static_smem < 0) {
            cudaFuncAttributes fa;
            cudaError_t err = cudaFuncGetAttributes(&fa, kern);
            if (err != cudaSuccess) return err;
            static_smem = (int)fa.sharedSizeBytes;
            static_smem_cache.store(static_smem, std::memory_order_relaxed);
        }
        *budget = (size_t)di.max_smem_optin - (size_t)static_smem;
        int dev = 0;
        cudaError_t err = cudaGetDevice(&dev);
        if (err != cudaSuccess) return err;
        const uint64_t bit = 1ull << (dev & 63);
        if (!(attr_done.load(std::memory_order_acquire) & bit)) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)*budget);
            if (err != cudaSuccess) return err;
            attr_done.fetch_or(bit, std::memory_order_acq_rel);
        }
        return cudaSuccess;
    }
    static cudaError_t launch(const TcPlan &plan, const CUtensorMap &mw, const CUtensorMap &ms,
                              const CUtensorMap &mg, const CUtensorMap &mu,
                              const void *residual, void *out, int mc, int N, int group,
                              int k_cta, cudaStream_t stream) {
        return launch_kernel(gemv_tc_kernel<NPAD, STEPK>, dim3(kTcSplit, N / kTcRows),
                             dim3(kTcThreads), plan.smem, stream, kTcSplit, mw, ms, mg, mu,
                             static_cast<const uint16_t *>(residual), static_cast<uint16_t *>(out),
                             mc, N, group, k_cta, plan.s_w, plan.s_gu, plan.s_op, plan.off_gu,
                             plan.off_op, plan.off_sc, plan.sg);
    }
};

template <int NPAD>
cudaError_t launch_npad(const DeviceInfo &di, const void *gate, const void *up,
                        const void *qweight, const void *scales, const void *residual,
                        void *out, int mc, int K, int N, int group, cudaStream_t stream,
                        bool *launched) {
    constexpr int kStepK = tc_step_k(NPAD);
    using Primary = TcKernel<NPAD, kStepK>;
    using Fallback = TcKernel<NPAD, 64>;  // the same kernel at 64-k steps (see plan_tc)
    const int k_cta = K / kTcSplit;
    size_t budget = 0;
    cudaError_t err = Primary::prepare(di, &budget);
    if (err != cudaSuccess) return err;
    TcPlan plan;
    int stepk = 0;
    if (!plan_tc(NPAD, k_cta, group, budget, &stepk, &plan)) return cudaSuccess;  // not launched
    if (stepk != kStepK) {
        size_t b64 = 0;
        err = Fallback::prepare(di, &b64);
        if (err != cudaSuccess) return err;
        if (b64 < plan.smem) return cudaSuccess;  // not launched
    }

    CUtensorMap mw, ms, mg, mu;
    if (!encode_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, qweight, (uint64_t)K / 2, (uint64_t)N,
                   (uint64_t)K / 2, kTcWTileK / 2, kTcRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&ms, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, scales, (uint64_t)K / group,
                   (uint64_t)N, (uint64_t)(K / group) * 2, (uint32_t)plan.sg, kTcRows,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&mg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, gate, (uint64_t)K, (uint64_t)mc,
                   (uint64_t)K * 2, kTcGuBoxK, NPAD, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&mu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, up, (uint64_t)K, (uint64_t)mc,
                   (uint64_t)K * 2, kTcGuBoxK, NPAD, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;

    *launched = true;
    err = stepk == kStepK
              ? Primary::launch(plan, mw, ms, mg, mu, residual, out, mc, N, group, k_cta, stream)
              : Fallback::launch(plan, mw, ms, mg, mu, residual, out, mc, N, group, k_cta, stream);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace

bool gemv_tc_supported(int M, int K, int N, int group) {
    if (M < 1 || K % (kTcSplit * 256) != 0 || N % kTcRows != 0) return false;
    if (group % kTcGuBoxK != 0 || K % group != 0 || (K / group) % 8 != 0) return false;
    const int k_cta = K / kTcSplit;
    return ((k_cta + group - 1) / group + 14) <= 256;
}

cudaError_t launch_gemv_tc(const void *gate, const void *up, const void *qweight,
                           const void *scales, const void *residual, void *out, int M, int K,
                           int N, int group, cudaStream_t stream, bool *launched) {
    *launched = false;
    if (!gemv_tc_supported(M, K, N, group)) return cudaSuccess;
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const uint16_t *g = static_cast<const uint16_t *>(gate);
    const uint16_t *u = static_cast<const uint16_t *>(up);
    uint16_t *o = static_cast<uint16_t *>(out);
    const uint16_t *r = static_cast<const uint16_t *>(residual);
    // Up to 128 activation rows per launch (the MMA's N); larger M runs in row blocks.
    for (int m0 = 0; m0 < M; m0 += 128) {
        const int mc = M - m0 < 128 ? M - m0 : 128;
        const size_t ao = (size_t)m0 * K, oo = (size_t)m0 * N;
        const uint16_t *ro = r ? r + oo : nullptr;
        bool done = false;
        if (mc <= 16)
            err = launch_npad<16>(di, g + ao, u + ao, qweight, scales, ro, o + oo, mc, K, N, group, stream, &done);
        else if (mc <= 32)
            err = launch_npad<32>(di, g + ao, u + ao, qweight, scales, ro, o + oo, mc, K, N, group, stream, &done);
        else if (mc <= 64)
            err = launch_npad<64>(di, g + ao, u + ao, qweight, scales, ro, o + oo, mc, K, N, group, stream, &done);
        else
            err = launch_npad<128>(di, g + ao, u + ao, qweight, scales, ro, o + oo, mc, K, N, group, stream, &done);
        if (err != cudaSuccess) return err;
        if (!done) {
            if (m0 == 0) return cudaSuccess;  // nothing launched: the caller falls back
            return cudaErrorInvalidConfiguration;
        }
        *launched = true;
    }
    return cudaSuccess;
}

FD_DEFINE_STATUS_ACCESSOR(status_gemv_tc)

}  // namespace fd
