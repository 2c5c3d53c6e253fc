// fd_gemv_tma.cu - SwiGLU-prologue W4A16 GEMV, bulk-copy (TMA) weight stream.
//
// y[m, n] = bf16( [residual[m, n] +] sum_k silu(g[m, k]) * u[m, k] * q[n, k] * s[n, k / group] )
//
// The same kernel in its PLAIN form (template flag) takes a plain activation x instead of
// silu(g) * u: the horizontal gate/up projection, whose stacked output rows go to two
// tensors (rows n < split to out, the rest to out2).
//
// Sources: "09 - Operator fusion", section 5 (taxonomy item 4: dequantisation as the
// weights are loaded, only int4 crosses HBM; "The fusion boundary problem": act =
// silu(gate) * up feeds act @ W_down); "PyTorch Community Proposes Fusion Fix ..."
// ("Reproduction and analysis", "Fix proposal": the M = 1 product is never materialised,
// the small input a = silu(g) * u is formed first - here in registers).
//
// The fast path for K % 1024 == 0, K <= 15360 and (K / group) % 8 == 0 (every
// decode shape of interest). Design for GB300:
//   * Persistent CTAs, each owning a contiguous range of output rows n: one per SM, or
//     several per SM when a CTA is small (K=4096: three CTAs of 288 threads), as many as
//     the registers, threads and shared memory allow.
//   * Warp specialisation: the last warp is a producer whose lane 0 streams chunks of 8
//     consecutive weight rows (8 * K/2 bytes, one contiguous bulk copy) and their scales
//     (8 * K/group * 2 bytes, a second bulk copy) into shared-memory stages, completion
//     tracked by "full" mbarriers. When a CTA's whole share of rows fits (27 rows at
//     K=14336 N=4096, 17 at K=9216 N=2560), every chunk has a stage of its own and all
//     are in flight from the start; otherwise the stages form a ring (up to 8) and
//     consumers release a stage through an "empty" mbarrier (one arrival per warp).
//   * Each 32-k slice of K is owned by LPS consumer lanes (K/32 * LPS threads): a =
//     silu(g) * u for its k lives in registers as block-scaled int16
//     (fd_gemv_common.cuh); per row a lane reads its 16-byte slot (conflict-free), splits
//     each word into even/odd nibble bytes (2 lop3) and accumulates exactly in int32 with
//     4 dp2a per word; the 32-k sum is converted once and scaled by the activation and
//     group scales.
//   * LPS = 2 at M = 1: lanes l and l + 16 of a warp share a slice (16 slices per warp)
//     and take alternate rows of each chunk, so K = 9216 runs 18 consumer warps instead of
//     9 and every lane has half the rows; the encoding of the slice is split between them
//     (each converts 16 of its 32 k and they swap halves with one shuffle).
//   * Per chunk a butterfly reduce-scatter (over 16 lanes when LPS = 2) leaves one warp
//     sum per (row, m) in shared memory; every 64 rows the consumers sum over warps, add
//     the residual if one is given (the down projection's residual-add epilogue) and
//     store bf16 once per output.
//   * Every mbarrier wait is bounded (fd_tma.cuh). If one gives up, the CTA records the
//     timeout in the device status word (fd_device_status), stops computing, waits
//     (bounded) for the copies it issued, writes NaN to all of its outputs and exits.
#include <atomic>
#include <mutex>

#include "fd_gemv_common.cuh"
#include "fd_gemv_plan.h"
#include "fd_tma.cuh"

namespace fd {
namespace {

constexpr int kMaxStages = 8;
constexpr int kChunkRows = 8;  // rows per bulk-copy chunk

// The fold's tail, run by every thread of every CTA after its rows are stored. Each CTA
// publishes the sum of h^2 over its rows (warp sums, then warps in order) and takes a
// ticket; the CTA that draws the last one sums the partials in CTA order (so the result
// does not depend on arrival order), forms rstd = 1/sqrt(mean h^2 + eps) and writes the
// whole normalised row, bf16(bf16(h * rstd) * w) (the two roundings of the separate
// add-RMSNorm kernel), then resets the counter for the next call. No CTA waits for another.
__device__ __forceinline__ void fold_tail(const FoldArgs &fold, float ss, int N, float *red,
                                          int *last, bool failed) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < nwarps; ++w) t += red[w];
        // a CTA that gave up poisons the sum, so the normalised row is NaN like its outputs
        fold.partials[blockIdx.x] = failed ? __int_as_float(0x7FC00000) : t;
        __threadfence();  // the h rows and the partial before the ticket
        const unsigned ticket = atomicAdd(fold.counter, 1u);
        *last = (ticket == gridDim.x - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!*last) return;
    __threadfence();  // every other CTA's h rows and partial are visible after its ticket
    if (warp == 0) {
        float t = 0.f;
        for (int b = lane; b < (int)gridDim.x; b += 32) t += __ldcg(&fold.partials[b]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
        if (lane == 0) red[0] = t;
    }
    __syncthreads();
    const float rstd = rsqrtf(fmaf(red[0], fold.inv_n, fold.eps));
    const uint4 *h4 = reinterpret_cast<const uint4 *>(fold.res_out);
    const uint4 *w4 = reinterpret_cast<const uint4 *>(fold.weight);
    uint4 *o4 = reinterpret_cast<uint4 *>(fold.normed);
    for (int v = tid; v < N / 8; v += blockDim.x) {
        const uint4 hv = __ldcg(h4 + v);
        const uint4 wv = w4[v];
        const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t yw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t t = pack_bf16x2(bf16lo(hw[j]) * rstd, bf16hi(hw[j]) * rstd);
            yw[j] = pack_bf16x2(bf16lo(t) * bf16lo(ww[j]), bf16hi(t) * bf16hi(ww[j]));
        }
        o4[v] = make_uint4(yw[0], yw[1], yw[2], yw[3]);
    }
    if (tid == 0) *fold.counter = 0u;  // ready for the next call in the stream
}

// NVEC_C / NG_C: compile-time K/32 and K/group for the common shapes (0 = runtime), so
// the per-row shared-memory offsets fold into instruction immediates.
//
// Shared memory: w_rows weight rows (stage s holds rows [sR, sR + R)), the scales of S
// stages, then the per-warp partial sums. With one SwiGLU activation row (M == 1) the
// producer first bulk-copies gate and up (2 * K * 2 bytes = 8 weight rows) into the last
// 8 weight rows, ahead of the weight stream, so the consumers' activation reads do not
// queue behind it (loaded from global memory instead, they arrived behind the weights and
// the call took 10-25 % longer on GB300); stages from act_first_stage on are filled only
// after every consumer warp has read its slice. A small activation (at most 16 KB for the
// call: the gate/up projection's x at K = 4096, gate and up up to K = 4096 at M = 1) is
// loaded by the lanes straight from global memory instead, and the free stages' weight
// chunks go out before the dependency wait (the gate/up GEMV measured 64 -> 69 % of HBM
// with this on GB300; with 57 KB of gate/up the same order slowed the decode step).
// FOLD: the next layer's add-RMSNorm in the tail (M = 1, SwiGLU form only); a separate
// instantiation, so the other kernels' code is unchanged by it.
template <int MB, int R, int NVEC_C, int NG_C, int LPS, bool PLAIN, bool FOLD>
__global__ void __launch_bounds__(LPS == 2 ? 1024 : 512, 1)
    gemv_tma_kernel(const uint16_t *__restrict__ gate, const uint16_t *__restrict__ up,
                    const unsigned char *__restrict__ qweight,
                    const uint16_t *__restrict__ scales, const uint16_t *residual,
                    uint16_t *out, uint16_t *out2, int split, int ldo, int M, int K, int N,
                    int group, int rows_base, int rows_extra, int S,
                    int w_rows, int act_first_stage, int weights_evict_first,
                    int test_timeout, const FoldArgs fold) {
    static_assert(R * MB <= 32 && (R * MB & (R * MB - 1)) == 0, "R*MB: power of 2, <= 32");
    static_assert(LPS == 1 || (LPS == 2 && MB == 1 && R % 2 == 0), "paired lanes: M = 1 only");
    static_assert(!FOLD || (MB == 1 && LPS == 2 && !PLAIN), "the fold: M = 1, SwiGLU form");
    static_assert(kWindowRows % R == 0, "window must hold whole chunks");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full_bar[kMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
    __shared__ __align__(8) uint64_t act_full_bar;
    __shared__ __align__(8) uint64_t act_free_bar;
    __shared__ int abort_flag;
    __shared__ float fold_red[FOLD ? 32 : 1];
    __shared__ int fold_last;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nvec = NVEC_C ? NVEC_C : (K >> 5);  // 32-k slices, a multiple of 32
    const int ncons = LPS * nvec;                  // consumer threads (LPS lanes per slice)
    const int ncw = ncons >> 5;                    // consumer warps
    const int ngroups = NG_C ? NG_C : K / group;
    const uint32_t w_row_bytes = (uint32_t)nvec * 16;
    const uint32_t s_row_bytes = (uint32_t)ngroups * 2;
    const uint32_t w_stage_bytes = (uint32_t)R * w_row_bytes;
    const uint32_t s_stage_bytes = (uint32_t)R * s_row_bytes;
    unsigned char *s_region = smem + (size_t)w_rows * w_row_bytes;
    float *red = reinterpret_cast<float *>(s_region + (size_t)S * s_stage_bytes);
    // gate then up, each K bf16 (4K bytes = 8 weight rows; PLAIN: x alone, 2K bytes = 4
    // rows), in the last weight rows (M == 1 only); stages from act_first_stage on are
    // filled only after its release
    const bool direct_act = (long long)M * K * (PLAIN ? 2 : 4) <= 16384;
    const bool act_in_smem = (M == 1) && !direct_act;
    const uint32_t act_bytes = (uint32_t)K * (PLAIN ? 2 : 4);
    uint16_t *act_smem =
        reinterpret_cast<uint16_t *>(smem + (size_t)w_rows * w_row_bytes - act_bytes);

    const int b = blockIdx.x;
    const int n_begin = b * rows_base + min(b, rows_extra);
    const int n_cnt = rows_base + (b < rows_extra ? 1 : 0);
    const int n_chunks = (n_cnt + R - 1) / R;
    const int m_chunks = (M + MB - 1) / MB;
    const int total = n_chunks * m_chunks;

    // Lane 0 of the last warp is the producer. It initialises the barriers itself and
    // issues the activation copy and the chunks that fit in free stages before the
    // CTA-wide barrier, so they are in flight while the other warps start up.
    // test_timeout (FD_LAUNCH_TEST_WAIT_TIMEOUT): short waits, and chunk 0 is never copied,
    // so the consumers' wait for it runs out
    const long long limit = test_timeout ? kTestWaitLimitCycles : kWaitLimitCycles;
    const int skip_chunk = test_timeout ? 0 : -1;
    const bool producer = (warp == ncw && lane == 0);
    float fold_ss = 0.f;  // the fold: this thread's sum of h^2 over the rows it stores
    uint64_t pol_w = 0, pol_s = 0;
    int issued = 0, ps = 0, pround = 0, pnc = 0, pc = 0;
    bool pok = true;
    auto issue_chunk = [&](int c) {
        if (act_in_smem && c == act_first_stage)
            pok = mbar_wait_bounded(&act_free_bar, 0, &abort_flag, limit);
        if (pok && pround > 0)
            pok = mbar_wait_bounded(&empty_bar[ps], (pround - 1) & 1, &abort_flag, limit);
        if (!pok) return;
        if (c != skip_chunk) {
            const int rows = min(R, n_cnt - pnc * R);
            const size_t n0 = (size_t)n_begin + (size_t)pnc * R;
            const uint32_t wb = (uint32_t)rows * w_row_bytes;
            const uint32_t sb = (uint32_t)rows * s_row_bytes;
            mbar_arrive_expect_tx(&full_bar[ps], wb + sb);
            bulk_g2s(smem + (size_t)ps * w_stage_bytes, qweight + n0 * w_row_bytes, wb,
                     &full_bar[ps], pol_w);
            bulk_g2s(s_region + (size_t)ps * s_stage_bytes, scales + n0 * ngroups, sb,
                     &full_bar[ps], pol_s);
        }
        issued = c + 1;
        if (++ps == S) { ps = 0; ++pround; }
        if (++pnc == n_chunks) pnc = 0;
    };
    if (producer) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], ncw);
        }
        mbar_init(&act_full_bar, 1);
        mbar_init(&act_free_bar, ncw);
        abort_flag = 0;
        fence_mbar_init();
        pol_w = weights_evict_first ? policy_evict_first() : policy_evict_last();
        pol_s = policy_evict_first();
        if (direct_act) {
            // The weights never come from the previous kernel, and the consumers read the
            // small activation from global memory: the free stages' chunks go out before
            // the dependency wait.
            for (; pc < total && pc < S; ++pc) issue_chunk(pc);
            grid_dep_wait();
            grid_dep_launch();
        } else {
            // Nothing is issued before the dependency wait: the activation copy is what
            // every consumer waits for first, and weight traffic issued ahead of it (copies
            // into the ring or L2 prefetches) delayed it and cost the 32-layer decode step
            // 15-25 % in measurements on GB300.
            grid_dep_wait();
            grid_dep_launch();
            if (act_in_smem) {
                const uint32_t ab = (uint32_t)K * 2;
                mbar_arrive_expect_tx(&act_full_bar, act_bytes);
                const uint64_t pol_a = policy_evict_last();  // every CTA reads it
                bulk_g2s(act_smem, gate, ab, &act_full_bar, pol_a);
                if (!PLAIN) bulk_g2s(act_smem + K, up, ab, &act_full_bar, pol_a);
            }
            // stages that are free from the start: no waits
            for (; pc < total && pc < act_first_stage; ++pc) issue_chunk(pc);
        }
    }
    __syncthreads();

    if (warp == ncw) {
        // ------------------------------------------------------------ producer warp
        if (lane != 0) {
            grid_dep_wait();
            grid_dep_launch();
        } else {
            for (; pc < total && pok; ++pc) issue_chunk(pc);
            // Every issued copy must land before the CTA exits: wait (bounded) on the
            // last phase of each stage that was used, and on the activation copy.
            for (int c = max(0, issued - S); c < issued; ++c) {
                if (c == skip_chunk) continue;
                const int st_idx = c % S;
                const long long t0 = clock64();
                while (!mbar_test_parity(&full_bar[st_idx], (c / S) & 1)) {
                    if (clock64() - t0 > limit) {
                        record_wait_timeout();
                        break;
                    }
                    __nanosleep(64);
                }
            }
            if (act_in_smem) {
                const long long t0 = clock64();
                while (!mbar_test_parity(&act_full_bar, 0)) {
                    if (clock64() - t0 > limit) {
                        record_wait_timeout();
                        break;
                    }
                    __nanosleep(64);
                }
            }
        }
    } else if constexpr (LPS == 2) {
        // ------------------------------------------------------ consumer warps, paired
        // Lanes l and l ^ 16 share one 32-k slice: lane l owns slice 16 * warp + (l & 15)
        // and, in every chunk, the rows r = 2i + h (h = l >> 4). So a CTA runs twice the
        // warps of the one-lane form on the same rows, and each lane encodes 16 elements.
        grid_dep_wait();
        grid_dep_launch();
        // The residual of the first window's rows (thread i stores row i, below), requested
        // now so that the final store does not wait on its load.
        float res0 = 0.f;
        if (residual && tid < min(n_cnt, kWindowRows)) res0 = bf16lo(residual[n_begin + tid]);
        // the fold's residual stream of the same rows, likewise requested early
        float fres0 = 0.f;
        if constexpr (FOLD) {
            if (tid < min(n_cnt, kWindowRows)) fres0 = bf16lo(fold.res_in[n_begin + tid]);
        }
        const int hh = lane >> 4;
        const int slice = 16 * warp + (lane & 15);
        const int col = (slice * 32) / group;  // this lane's scale column
        const W4Keys keys = w4_keys();
        Act16 act;
        {
            GateUpHalf gu;
            bool act_ok = true;
            if (act_in_smem) {
                act_ok = mbar_wait_bounded(&act_full_bar, 0, &abort_flag, limit);
                if (act_ok) {
                    const uint4 *g4 = reinterpret_cast<const uint4 *>(act_smem + slice * 32 + 16 * hh);
                    gu.g[0] = g4[0];
                    gu.g[1] = g4[1];
                    if (!PLAIN) {
                        const uint4 *u4 = reinterpret_cast<const uint4 *>(act_smem + K + slice * 32 + 16 * hh);
                        gu.u[0] = u4[0];
                        gu.u[1] = u4[1];
                    }
                }
            } else {
                const uint4 *g4 = reinterpret_cast<const uint4 *>(gate + slice * 32 + 16 * hh);
                gu.g[0] = g4[0];
                gu.g[1] = g4[1];
                if (!PLAIN) {
                    const uint4 *u4 = reinterpret_cast<const uint4 *>(up + slice * 32 + 16 * hh);
                    gu.u[0] = u4[0];
                    gu.u[1] = u4[1];
                }
            }
            if (!act_ok) gu.g[0] = gu.g[1] = gu.u[0] = gu.u[1] = make_uint4(0, 0, 0, 0);
            if constexpr (PLAIN)
                encode_plain_pair(gu.g, hh, act);
            else
                encode_q16_pair(gu, hh, act);
            // When weight chunks overlay the area, it is released after the encode (released
            // before it, the encode ran ~0.4 us longer at K=14336 and the call gained
            // nothing, the weight stream being the bound), with a proxy fence: the
            // producer's bulk copy writes it next.
            if (act_in_smem && act_first_stage < total) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&act_free_bar);
            }
        }
        constexpr int kRowsPerLane = R / 2;
        constexpr int kLanesPerValue = 16 / kRowsPerLane;
        int window_base = 0;
        int s = 0, phase = 0, nc = 0;
        for (int c = 0; c < total; ++c) {
            float part[kRowsPerLane];
            const bool ok = mbar_wait_bounded(&full_bar[s], phase, &abort_flag, limit);
            const int rows_valid = min(R, n_cnt - nc * R);
            const uint4 *wst =
                reinterpret_cast<const uint4 *>(smem + (size_t)s * w_stage_bytes) + slice + hh * nvec;
            const uint16_t *sst = reinterpret_cast<const uint16_t *>(s_region + (size_t)s * s_stage_bytes) +
                                  col + hh * ngroups;
            if (ok && rows_valid == R) {
#pragma unroll
                for (int i = 0; i < kRowsPerLane; ++i) {
                    const uint4 wv = wst[2 * i * nvec];
                    const float sc = __uint_as_float((uint32_t)sst[2 * i * ngroups] << 16);
                    float d[1];
                    dot32<1>(&act, wv, keys, sc, d);
                    part[i] = d[0];
                }
            } else {
                // last, partial chunk (or a failed wait): rows past the range are skipped
#pragma unroll
                for (int i = 0; i < kRowsPerLane; ++i) {
                    if (ok && 2 * i + hh < rows_valid) {
                        const uint4 wv = wst[2 * i * nvec];
                        const float sc = __uint_as_float((uint32_t)sst[2 * i * ngroups] << 16);
                        float d[1];
                        dot32<1>(&act, wv, keys, sc, d);
                        part[i] = d[0];
                    } else {
                        part[i] = 0.f;
                    }
                }
            }
            if (total > S) {  // the stage is reused: its reads before the next bulk copy
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty_bar[s]);
            }

            const float wsum = half_reduce_scatter<kRowsPerLane>(part, lane);
            if (((lane & 15) & (kLanesPerValue - 1)) == 0) {
                const int r = 2 * ((lane & 15) / kLanesPerValue) + hh;
                red[(size_t)warp * kWindowRows + (nc * R + r - window_base)] = wsum;
            }
            const int rows_done = (nc + 1) * R;
            const bool last_chunk = (nc == n_chunks - 1);
            if (rows_done - window_base == kWindowRows || last_chunk) {
                named_bar_sync(1, ncons);
                const int rows_in_window = min(rows_done, n_cnt) - window_base;
                for (int i = tid; i < rows_in_window; i += ncons) {
                    const int n = n_begin + window_base + i;
                    float acc = sum_partials(red + i, ncw, kWindowRows);
                    if (residual) acc += window_base == 0 ? res0 : bf16lo(residual[n]);
                    __nv_bfloat16 y = __float2bfloat16_rn(acc);
                    // The split output (gate/up halves) only where it is used: in the SwiGLU
                    // kernel the extra select changed the register allocation of the row
                    // loop and cost 2.8 % per call at K=14336 on GB300.
                    if constexpr (PLAIN) {
                        *out_at(out, out2, split, ldo, 0, n) = *reinterpret_cast<uint16_t *>(&y);
                    } else {
                        const uint16_t yb = *reinterpret_cast<uint16_t *>(&y);
                        out[n] = yb;
                        if constexpr (FOLD) {
                            // the next layer's add: h = bf16(f32(y) + f32(residual)), the
                            // rounded y as the separate kernel would read it
                            const float r = window_base == 0 ? fres0 : bf16lo(fold.res_in[n]);
                            const __nv_bfloat16 h = __float2bfloat16_rn(bf16lo(yb) + r);
                            const uint16_t hb = *reinterpret_cast<const uint16_t *>(&h);
                            fold.res_out[n] = hb;
                            const float hf = bf16lo(hb);
                            fold_ss = fmaf(hf, hf, fold_ss);
                        }
                    }
                }
                named_bar_sync(1, ncons);
                window_base = last_chunk ? 0 : rows_done;
            }
            if (++s == S) { s = 0; phase ^= 1; }
            if (++nc == n_chunks) nc = 0;
        }
    } else {
        // ------------------------------------------------------------ consumer warps
        // (one lane per 32-k slice)
        // gate/up and the output may be shared with the previous kernel in the stream.
        grid_dep_wait();
        grid_dep_launch();
        const int col = (tid * 32) / group;  // this thread's scale column
        const W4Keys keys = w4_keys();
        Act16 act[MB];
        int window_base = 0;
        int s = 0, phase = 0, nc = 0, m0 = 0;
        constexpr int kLanesPerValue = 32 / (R * MB);
        for (int c = 0; c < total; ++c) {
            if (nc == 0) {
#pragma unroll
                for (int mb = 0; mb < MB; ++mb) {
                    if (m0 + mb < M) {
                        GateUp gu;
                        if (act_in_smem) {
                            if (mbar_wait_bounded(&act_full_bar, 0, &abort_flag, limit)) {
                                // Each lane's slice is 64 contiguous bytes, read in order.
                                // (The reads are 4-way bank conflicted; rotating their order
                                // by lane avoids that but needs per-lane register selects,
                                // which measured ~0.5 us slower per call.)
                                const uint4 *g4 = reinterpret_cast<const uint4 *>(act_smem + tid * 32);
                                const uint4 *u4 = reinterpret_cast<const uint4 *>(act_smem + K + tid * 32);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    gu.g[i] = g4[i];
                                    if (!PLAIN) gu.u[i] = u4[i];
                                }
                            } else {
#pragma unroll
                                for (int i = 0; i < 4; ++i) gu.g[i] = gu.u[i] = make_uint4(0, 0, 0, 0);
                            }
                            // The area is released after the encode (when chunks overlay
                            // it), with a proxy fence: the next bulk copy writes it.
                            if constexpr (PLAIN)
                                encode_plain(gu.g, act[mb]);
                            else
                                encode_q16(gu, act[mb]);
                            if (act_first_stage < total) {
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) mbar_arrive(&act_free_bar);
                            }
                        } else {
                            const size_t off = (size_t)(m0 + mb) * K + (size_t)tid * 32;
                            if constexpr (PLAIN) {
                                const uint4 *x4 = reinterpret_cast<const uint4 *>(gate + off);
#pragma unroll
                                for (int i = 0; i < 4; ++i) gu.g[i] = x4[i];
                                encode_plain(gu.g, act[mb]);
                            } else {
                                load_gate_up(gate, up, off, gu);
                                encode_q16(gu, act[mb]);
                            }
                        }
                    } else {
                        zero_activation(act[mb]);
                    }
                }
            }
            float part[R * MB];
            const bool ok = mbar_wait_bounded(&full_bar[s], phase, &abort_flag, limit);
            const int rows_valid = min(R, n_cnt - nc * R);
            const uint4 *wst = reinterpret_cast<const uint4 *>(smem + (size_t)s * w_stage_bytes) + tid;
            const uint16_t *sst =
                reinterpret_cast<const uint16_t *>(s_region + (size_t)s * s_stage_bytes) + col;
            if (ok && rows_valid == R) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint4 wv = wst[r * nvec];
                    const float sc = __uint_as_float((uint32_t)sst[r * ngroups] << 16);
                    float d[MB];
                    dot32<MB>(act, wv, keys, sc, d);
#pragma unroll
                    for (int mb = 0; mb < MB; ++mb) part[r * MB + mb] = d[mb];
                }
            } else {
                // last, partial chunk (or a failed wait): rows past the range are skipped
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (ok && r < rows_valid) {
                        const uint4 wv = wst[r * nvec];
                        const float sc = __uint_as_float((uint32_t)sst[r * ngroups] << 16);
                        float d[MB];
                        dot32<MB>(act, wv, keys, sc, d);
#pragma unroll
                        for (int mb = 0; mb < MB; ++mb) part[r * MB + mb] = d[mb];
                    } else {
#pragma unroll
                        for (int mb = 0; mb < MB; ++mb) part[r * MB + mb] = 0.f;
                    }
                }
            }
            if (total > S) {  // the stage is reused: its reads before the next bulk copy
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty_bar[s]);
            }

            const float wsum = warp_reduce_scatter<R * MB>(part, lane);
            if ((lane & (kLanesPerValue - 1)) == 0) {
                const int idx = lane / kLanesPerValue;
                const int r = idx / MB, mb = idx % MB;
                red[((size_t)warp * kWindowRows + (nc * R + r - window_base)) * MB + mb] = wsum;
            }
            const int rows_done = (nc + 1) * R;
            const bool last_chunk = (nc == n_chunks - 1);
            if (rows_done - window_base == kWindowRows || last_chunk) {
                named_bar_sync(1, ncons);
                const int rows_in_window = min(rows_done, n_cnt) - window_base;
                for (int i = tid; i < rows_in_window * MB; i += ncons) {
                    const int row = i / MB, mb = i % MB;
                    float acc = sum_partials(red + (size_t)row * MB + mb, ncw, kWindowRows * MB);
                    if (m0 + mb < M) {
                        const int n = n_begin + window_base + row;
                        if (residual) acc += bf16lo(residual[(size_t)(m0 + mb) * N + n]);
                        __nv_bfloat16 y = __float2bfloat16_rn(acc);
                        if constexpr (PLAIN)
                            *out_at(out, out2, split, ldo, m0 + mb, n) = *reinterpret_cast<uint16_t *>(&y);
                        else
                            out[(size_t)(m0 + mb) * N + n] = *reinterpret_cast<uint16_t *>(&y);
                    }
                }
                named_bar_sync(1, ncons);
                window_base = last_chunk ? 0 : rows_done;
            }
            if (++s == S) { s = 0; phase ^= 1; }
            if (++nc == n_chunks) { nc = 0; m0 += MB; }
        }
    }

    __syncthreads();
    if (abort_flag) {
        // A wait gave up: make the failure visible in every output this CTA owns.
        for (int i = tid; i < n_cnt * M; i += blockDim.x) {
            const int m = i / n_cnt, r = i % n_cnt;
            if constexpr (PLAIN)
                *out_at(out, out2, split, ldo, m, n_begin + r) = 0x7FC0;  // bf16 quiet NaN
            else
                out[(size_t)m * N + n_begin + r] = 0x7FC0;
        }
    }
    if constexpr (FOLD) fold_tail(fold, fold_ss, N, fold_red, &fold_last, abort_flag != 0);
}

template <int MB, int R, int NVEC_C, int NG_C, int LPS, bool PLAIN, bool FOLD>
cudaError_t launch_cfg(const DeviceInfo &di, const void *gate, const void *up,
                       const void *qweight, const void *scales, const void *residual,
                       GemvOut o, int M, int K, int N, int group, cudaStream_t stream,
                       bool *launched, const FoldArgs *fold) {
    static std::atomic<uint64_t> attr_done{0};
    static std::atomic<int> func_cache{-1};  // static shared memory | registers << 20
    auto kern = gemv_tma_kernel<MB, R, NVEC_C, NG_C, LPS, PLAIN, FOLD>;
    int fc = func_cache.load(std::memory_order_relaxed);
    if (fc < 0) {
        cudaFuncAttributes fa;
        cudaError_t err = cudaFuncGetAttributes(&fa, kern);
        if (err != cudaSuccess) return err;
        fc = (fa.sharedSizeBytes & 0xFFFFF) | (fa.numRegs << 20);
        func_cache.store(fc, std::memory_order_relaxed);
    }
    const int nvec = K / 32;
    TmaPlanInput in{di.sm_count, di.max_smem_optin, di.smem_per_sm, di.smem_reserved,
                    fc & 0xFFFFF, fc >> 20, M, K, N, group, MB, LPS, R, kMaxStages, PLAIN ? 1 : 0};
    TmaPlan plan{};
    if (!plan_gemv_tma(in, &plan)) return cudaSuccess;  // not launched
    if (fold && plan.grid > kFoldMaxCtas) return cudaSuccess;  // not launched: no room for partials
    const FoldArgs fa = fold ? *fold : FoldArgs{};
    const int S = plan.S, w_rows = plan.w_rows, act_first_stage = plan.act_first_stage;
    const int grid = plan.grid, rows_base = plan.rows_base, rows_extra = plan.rows_extra;
    const size_t smem = plan.smem;
    const size_t budget = (size_t)di.max_smem_optin - (size_t)(fc & 0xFFFFF);
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)budget);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
        attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    err = launch_kernel(kern, dim3(grid), dim3(LPS * nvec + 32), smem, stream, 1,
                        static_cast<const uint16_t *>(gate), static_cast<const uint16_t *>(up),
                        static_cast<const unsigned char *>(qweight),
                        static_cast<const uint16_t *>(scales),
                        static_cast<const uint16_t *>(residual), static_cast<uint16_t *>(o.out),
                        static_cast<uint16_t *>(o.out2), o.split, o.ldo, M, K, N, group,
                        rows_base, rows_extra, S, w_rows, act_first_stage,
                        M <= MB ? 1 : 0, (launch_flags() & FD_LAUNCH_TEST_WAIT_TIMEOUT) ? 1 : 0, fa);
    *launched = true;
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

// LPS = 2 (two lanes per 32-k slice) for one activation row, else one lane per slice.
// The SwiGLU form is specialised for the down-projection widths, the plain form for the
// model width (the gate/up projection's K).
template <int MB, bool PLAIN, bool FOLD>
cudaError_t launch_mb(const DeviceInfo &di, const void *gate, const void *up,
                      const void *qweight, const void *scales, const void *residual, GemvOut o,
                      int M, int K, int N, int group, cudaStream_t stream, bool *launched,
                      const FoldArgs *fold) {
    constexpr int R = kChunkRows;
    constexpr int LPS = MB == 1 ? 2 : 1;
#define FD_SHAPE(KK, GG)                                                                          \
    if (K == KK && group == GG)                                                                   \
        return launch_cfg<MB, R, KK / 32, KK / GG, LPS, PLAIN, FOLD>(di, gate, up, qweight, scales,\
                                                              residual, o, M, K, N, group, stream, \
                                                              launched, fold);
    if constexpr (PLAIN) {
        FD_SHAPE(4096, 128)
    } else {
        FD_SHAPE(14336, 128)
        FD_SHAPE(9216, 128)
        FD_SHAPE(4096, 128)
        FD_SHAPE(1024, 128)
    }
#undef FD_SHAPE
    return launch_cfg<MB, R, 0, 0, LPS, PLAIN, FOLD>(di, gate, up, qweight, scales, residual, o,
                                                     M, K, N, group, stream, launched, fold);
}

// The grid the FOLD kernel would launch for an M = 1 call (0: the kernel does not run the
// shape), from the same plan as launch_cfg.
template <int NVEC_C, int NG_C>
cudaError_t fold_grid_cfg(const DeviceInfo &di, int K, int N, int group, int *grid) {
    static std::atomic<int> func_cache{-1};
    auto kern = gemv_tma_kernel<1, kChunkRows, NVEC_C, NG_C, 2, false, true>;
    int fc = func_cache.load(std::memory_order_relaxed);
    if (fc < 0) {
        cudaFuncAttributes fa;
        cudaError_t err = cudaFuncGetAttributes(&fa, kern);
        if (err != cudaSuccess) return err;
        fc = (fa.sharedSizeBytes & 0xFFFFF) | (fa.numRegs << 20);
        func_cache.store(fc, std::memory_order_relaxed);
    }
    TmaPlanInput in{di.sm_count, di.max_smem_optin, di.smem_per_sm, di.smem_reserved,
                    fc & 0xFFFFF, fc >> 20, 1, K, N, group, 1, 2, kChunkRows, kMaxStages, 0};
    TmaPlan plan{};
    *grid = plan_gemv_tma(in, &plan) ? plan.grid : 0;
    return cudaSuccess;
}

// The library's own scratch for fd_swiglu_w4a16_gemv_add_rmsnorm_noalloc: the fold's
// counter and per-CTA partial sums (FD_FOLD_SCRATCH_BYTES). Every GPU that loads this
// library holds it until the process exits; every call of the entry point shares it.
static __device__ __align__(256) unsigned char g_fold_scratch[FD_FOLD_SCRATCH_BYTES];

// Set-up, once per device, with that device current: the array's device address (in host
// code its name is only a stand-in, not a device address) and one zeroing of it on
// `stream`, ordered before the call's kernel. Every completed call leaves the counter at
// zero again.
cudaError_t fold_scratch_address(cudaStream_t stream, void **ptr) {
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev & 63]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_fold_scratch);
        if (err != cudaSuccess) return err;
        err = cudaMemsetAsync(p, 0, FD_FOLD_SCRATCH_BYTES, stream);
        if (err != cudaSuccess) return err;
        addr[dev & 63] = p;
    }
    *ptr = addr[dev & 63];
    return cudaSuccess;
}

}  // namespace

bool gemv_tma_supported(int M, int K, int group);

cudaError_t launch_gemv_fold_noalloc(const void *gate, const void *up, const void *qweight,
                                     const void *scales, void *y, const void *residual,
                                     const void *rms_weight, float eps, void *normed,
                                     void *residual_out, int K, int N, int group,
                                     cudaStream_t stream, bool *launched, bool *too_big) {
    *launched = false;
    *too_big = false;
    if (!gemv_tma_supported(1, K, group)) return cudaSuccess;
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    int grid = 0;
    if (K == 14336 && group == 128)
        err = fold_grid_cfg<14336 / 32, 14336 / 128>(di, K, N, group, &grid);
    else if (K == 9216 && group == 128)
        err = fold_grid_cfg<9216 / 32, 9216 / 128>(di, K, N, group, &grid);
    else if (K == 4096 && group == 128)
        err = fold_grid_cfg<4096 / 32, 4096 / 128>(di, K, N, group, &grid);
    else if (K == 1024 && group == 128)
        err = fold_grid_cfg<1024 / 32, 1024 / 128>(di, K, N, group, &grid);
    else
        err = fold_grid_cfg<0, 0>(di, K, N, group, &grid);
    if (err != cudaSuccess || grid == 0) return err;
    if (grid > kFoldMaxCtas) {  // more per-CTA sums than the array holds
        *too_big = true;
        return cudaSuccess;
    }
    void *scratch = nullptr;
    err = fold_scratch_address(stream, &scratch);
    if (err != cudaSuccess) return err;
    unsigned char *sc = static_cast<unsigned char *>(scratch);
    const FoldArgs fold{static_cast<const uint16_t *>(residual),
                        static_cast<uint16_t *>(residual_out),
                        static_cast<const uint16_t *>(rms_weight), static_cast<uint16_t *>(normed),
                        reinterpret_cast<float *>(sc + kFoldPartialsOffset),
                        reinterpret_cast<unsigned *>(sc), eps, 1.0f / (float)N};
    return launch_gemv_tma(gate, up, qweight, scales, nullptr, GemvOut{y, nullptr, N, N}, 1, K,
                           N, group, stream, launched, &fold);
}

bool gemv_tma_supported(int M, int K, int group) {
    (void)M;
    const int nvec = K / 32;
    return K % 1024 == 0 && nvec + 32 <= 512 && (K / group) % 8 == 0;
}

cudaError_t launch_gemv_tma(const void *gate, const void *up, const void *qweight,
                            const void *scales, const void *residual, GemvOut o, int M, int K,
                            int N, int group, cudaStream_t stream, bool *launched,
                            const FoldArgs *fold) {
    *launched = false;
    if (!gemv_tma_supported(M, K, group)) return cudaSuccess;
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    if (fold) {
        if (M != 1 || up == nullptr || residual != nullptr) return cudaSuccess;
        return launch_mb<1, false, true>(di, gate, up, qweight, scales, residual, o, M, K, N,
                                         group, stream, launched, fold);
    }
    if (up == nullptr) {
        if (M == 1)
            return launch_mb<1, true, false>(di, gate, up, qweight, scales, residual, o, M, K, N,
                                             group, stream, launched, nullptr);
        return launch_mb<2, true, false>(di, gate, up, qweight, scales, residual, o, M, K, N,
                                         group, stream, launched, nullptr);
    }
    if (M == 1)
        return launch_mb<1, false, false>(di, gate, up, qweight, scales, residual, o, M, K, N,
                                          group, stream, launched, nullptr);
    return launch_mb<2, false, false>(di, gate, up, qweight, scales, residual, o, M, K, N, group,
                                      stream, launched, nullptr);
}

FD_DEFINE_STATUS_ACCESSOR(status_gemv_tma)

}  // namespace fd
