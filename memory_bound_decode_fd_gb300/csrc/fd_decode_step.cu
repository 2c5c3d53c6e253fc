// fd_decode_step.cu - the decode step (L layers of add-RMSNorm then the SwiGLU-W4A16 down
// projection, M = 1) as one persistent cooperative kernel.
//
//   per layer l:  (normed_l, residual) = add_rmsnorm(x_l, residual, w_l)
//                 y_l = swiglu_w4a16_gemv(g_l, u_l, W_l, s_l);  x_{l+1} = y_l
//
// Sources: "Kernel Fusion, torch.compile and CUDA Graphs, Measured", Step 4 (in decode the
// per-kernel fixed costs exceed the kernels' own time; the step is recorded once and
// replayed) and Step 2 (the add-RMSNorm row kernel); "09 - Operator fusion", section 5
// (the down projection with its SwiGLU prologue and dequantisation on chip).
//
// Design for GB300. The separate kernels of a step are each bounded by HBM while they
// stream weights, but every GEMV launch also pays ~3.5 us with no weight bytes arriving:
// its activation copy and encode, the DRAM latency of its first chunk, and its tail. That
// head cannot overlap the previous kernel: weight requests queued ahead of a kernel's
// activation copy delay it by their own transfer time. Here one CTA per SM stays resident
// for all layers and keeps the rows of the bulk-copy GEMV's partition (the same rows, chunks
// and consumer layout, so every output is bit-identical to the separate kernels):
//   * The producer lane streams each layer's weight and scale chunks into the CTA's stages
//     as soon as the consumers release the previous layer's chunk in that stage, so the
//     next layer's weights arrive while this layer finishes and the next add-RMSNorm runs.
//   * A CTA owns the residual of its rows: it forms h = bf16(y + residual) for them, keeps
//     h in registers and publishes each element as one 32-bit word, the layer's tag in the
//     high half and the bf16 in the low half, into one of two h rows in the scratch
//     (alternating by layer), then adds one to the layer's counter (no fence: the tags,
//     not the counter, make the data safe to use). When the counter reaches the grid,
//     every CTA reads the whole h row, re-reading a 16-byte vector in the rare case that
//     not all its words carry the layer's tag yet. (Polling the tagged row itself, with no
//     counter, measured slower: 152 CTAs re-reading the same lines.) It computes the next
//     layer's add-RMSNorm for the whole row exactly as the row kernel does (the same
//     thread count, vector layout and reduction order) into shared memory and stores its
//     own rows of the normalised row. So each CTA holds the complete normalised row before
//     it reads the next layer's activations, as the next kernel of a chain starts only
//     after add-RMSNorm has finished. The first layer's add-RMSNorm needs no wait: every
//     CTA computes it from x0 and the residual.
//   * A CTA writes h row l + 2 into the buffer that held h row l only after it has read
//     the whole h row l + 1, which every CTA writes only after it has read h row l. The
//     call zeroes the rows first, so no tag of an earlier call is taken for this one.
//   * The activations (gate, up) are loaded straight into registers (no shared-memory
//     copy, which would have to wait behind the next layer's weights) and encoded as in the
//     GEMV kernel.
//   * Every wait is bounded (fd_tma.cuh). A wait that gives up records the status word; the
//     CTA keeps taking part in every count (so no other CTA waits on it) and writes NaN
//     where its results would have gone. FD_LAUNCH_TEST_WAIT_TIMEOUT makes the first
//     count's waits run out on purpose, on a short limit.
#include <atomic>

#include "fd_gemv_common.cuh"
#include "fd_step_plan.h"
#include "fd_tma.cuh"

namespace fd {
namespace {

static_assert(kStepWindowRows == kWindowRows, "the cross-warp sums of the GEMV kernel");

// Bounded spin until *p >= target, with acquire ordering at GPU scope.
__device__ __forceinline__ bool wait_counter(const unsigned *p, unsigned target, long long limit) {
    const long long t0 = clock64();
    while (true) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        if (v >= target) return true;
        if (clock64() - t0 > limit) {
            record_wait_timeout();
            return false;
        }
        __nanosleep(32);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Plain 16-byte global load, bypassing L1.
__device__ __forceinline__ uint4 ldg_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Tagged h words: relaxed GPU-scope accesses (each 32-bit word is read and written whole;
// the words of one vector load are checked one by one).
__device__ __forceinline__ uint4 ld_relaxed_v4(const void *p) {
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u32(void *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded re-read of the 8 tagged words of h vector v until all carry `tag`; returns the
// 8 bf16 as one 16-byte vector (false if the wait gave up).
__device__ __forceinline__ bool read_tagged_vec(const uint32_t *row, int v, uint32_t tag,
                                                uint4 *out, long long limit) {
    const uint4 *p = reinterpret_cast<const uint4 *>(row + 8 * v);
    const long long t0 = clock64();
    while (true) {
        const uint4 a = ld_relaxed_v4(p), c = ld_relaxed_v4(p + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
        bool ok = true;
#pragma unroll
        for (int k = 0; k < 8; ++k) ok &= (w[k] >> 16) == tag;
        if (ok) {
            *out = make_uint4(__byte_perm(w[0], w[1], 0x5410), __byte_perm(w[2], w[3], 0x5410),
                              __byte_perm(w[4], w[5], 0x5410), __byte_perm(w[6], w[7], 0x5410));
            return true;
        }
        if (clock64() - t0 > limit) {
            *out = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
            return false;
        }
        __nanosleep(20);
    }
}

// The add-RMSNorm row kernel's arithmetic on one whole row (fd_add_rmsnorm.cu with T
// threads and vpt 16-byte vectors per thread, vector v = t + i T): thread t < T holds the
// h vectors hv[i] and the weight vectors wv[i]. The sum of h^2 per thread in vector order,
// a warp butterfly, a butterfly over the warps' sums; rstd = rsqrt(sum / hidden + eps);
// the row bf16(bf16(h rstd) w) into s_normed. Every consumer thread calls it (it meets
// named barrier 1 once); s_normed is complete when the next barrier 1 is passed.
__device__ __forceinline__ void norm_row(const uint4 (&hv)[kStepRmsMaxVpt],
                                         const uint4 (&wv)[kStepRmsMaxVpt], int nvec, int vpt,
                                         int T, float inv_hidden, float eps, float *warp_ss,
                                         uint4 *s_normed, int ncons) {
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = T >> 5;
    float ss = 0.f;
    if (tid < T) {
#pragma unroll
        for (int i = 0; i < kStepRmsMaxVpt; ++i) {
            if (i < vpt && tid + i * T < nvec) {
                const uint32_t hw[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float h0 = bf16lo(hw[j]), h1 = bf16hi(hw[j]);
                    ss = fmaf(h0, h0, ss);
                    ss = fmaf(h1, h1, ss);
                }
            }
        }
    }
    ss = warp_sum(ss);
    if (lane == 0 && warp < nwarps) warp_ss[warp] = ss;
    named_bar_sync(1, ncons);
    if (tid < T) {
        float total = lane < nwarps ? warp_ss[lane] : 0.f;
        total = warp_sum(total);
        const float rstd = rsqrtf(fmaf(total, inv_hidden, eps));
#pragma unroll
        for (int i = 0; i < kStepRmsMaxVpt; ++i) {
            const int v = tid + i * T;
            if (i < vpt && v < nvec) {
                const uint32_t hw[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
                const uint32_t ww[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
                uint32_t yw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t t = pack_bf16x2(bf16lo(hw[j]) * rstd, bf16hi(hw[j]) * rstd);
                    yw[j] = pack_bf16x2(bf16lo(t) * bf16lo(ww[j]), bf16hi(t) * bf16hi(ww[j]));
                }
                s_normed[v] = make_uint4(yw[0], yw[1], yw[2], yw[3]);
            }
        }
    }
}

// Thread t < T: the weight vectors of its part of the row (read-only data).
__device__ __forceinline__ void load_norm_weight(const void *w, int nvec, int vpt, int T,
                                                 uint4 (&wv)[kStepRmsMaxVpt]) {
    const int tid = threadIdx.x;
#pragma unroll
    for (int i = 0; i < kStepRmsMaxVpt; ++i) {
        const int v = tid + i * T;
        wv[i] = make_uint4(0u, 0u, 0u, 0u);
        if (tid < T && i < vpt && v < nvec) wv[i] = __ldg(static_cast<const uint4 *>(w) + v);
    }
}

template <int NVEC_C, int NG_C>
__global__ void __launch_bounds__(1024, 1)
    decode_step_kernel(const fd_step_layer *__restrict__ layers, int n_layers,
                       const uint16_t *x0, uint16_t *residual, float eps, int N,
                       int rows_base, int rows_extra, int S, int w_rows, int rms_vpt,
                       int rms_threads, unsigned *count, uint32_t *hrows, int test_timeout) {
    constexpr int nvec = NVEC_C;      // 32-k slices
    constexpr int ngroups = NG_C;
    constexpr int ncons = 2 * nvec;   // two lanes per slice
    constexpr int ncw = ncons / 32;   // consumer warps
    constexpr int kRowsPerLane = kStepR / 2;
    constexpr int kLanesPerValue = 16 / kRowsPerLane;
    static_assert(ncons % 32 == 0 && ncons + 32 <= 1024, "consumer threads");
    static_assert(ncons >= kWindowRows && ncons >= 256, "one output row per consumer thread");
    constexpr uint32_t w_row_bytes = nvec * 16;
    constexpr uint32_t s_row_bytes = ngroups * 2;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full_bar[kStepMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kStepMaxStages];
    __shared__ int abort_flag;
    __shared__ float warp_ss[32];
    unsigned char *s_region = smem + (size_t)w_rows * w_row_bytes;
    float *red = reinterpret_cast<float *>(s_region + (size_t)S * kStepR * s_row_bytes);
    // the whole normalised row of the current layer (16-byte aligned: red is a multiple of 16)
    uint4 *s_normed = reinterpret_cast<uint4 *>(red + (size_t)ncw * kWindowRows);
    const uint16_t *s_normed16 = reinterpret_cast<const uint16_t *>(s_normed);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int b = blockIdx.x;
    const int grid = (int)gridDim.x;
    const int n_begin = b * rows_base + min(b, rows_extra);
    const int n_cnt = rows_base + (b < rows_extra ? 1 : 0);
    const int n_chunks = (n_cnt + kStepR - 1) / kStepR;
    const int nvec_h = N / 8;          // 16-byte vectors of a hidden row
    const float inv_hidden = 1.0f / (float)N;
    // hrows[(l & 1) * N ..]: h_{l+1} as tagged words (tag l + 1), written at the end of
    // layer l; count[l]: the CTAs that have written theirs (count[0] is also the exit
    // count of a single-layer call).
    // test_timeout (FD_LAUNCH_TEST_WAIT_TIMEOUT): short waits, and CTA 0 never adds itself
    // to count[0], so every CTA's wait for it runs out; the CTAs carry on (every count
    // after it is complete) and write NaN from the first normalised row that needed it.
    const long long limit = test_timeout ? kTestWaitLimitCycles : kWaitLimitCycles;
    const bool withhold = test_timeout && b == 0;

    if (tid == 0) {
        for (int s = 0; s < n_chunks; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], ncw);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == ncw) {
        // ------------------------------------------------------------ producer warp
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();  // each weight byte is read once
            bool ok = true;
            for (int l = 0; l < n_layers; ++l) {
                const unsigned char *qw = static_cast<const unsigned char *>(layers[l].qweight);
                const uint16_t *sc = static_cast<const uint16_t *>(layers[l].scales);
                for (int c = 0; c < n_chunks; ++c) {
                    // the consumers have read chunk c of the previous layer
                    if (ok && l > 0) ok = mbar_wait_bounded(&empty_bar[c], (l - 1) & 1, &abort_flag, limit);
                    if (!ok) break;
                    const int rows = min(kStepR, n_cnt - c * kStepR);
                    const size_t n0 = (size_t)n_begin + (size_t)c * kStepR;
                    const uint32_t wb = (uint32_t)rows * w_row_bytes, sb = (uint32_t)rows * s_row_bytes;
                    mbar_arrive_expect_tx(&full_bar[c], wb + sb);
                    bulk_g2s(smem + (size_t)c * kStepR * w_row_bytes, qw + n0 * w_row_bytes, wb,
                             &full_bar[c], pol_w);
                    bulk_g2s(s_region + (size_t)c * kStepR * s_row_bytes, sc + n0 * ngroups, sb,
                             &full_bar[c], pol_w);
                }
                if (!ok) break;
            }
            // every issued copy must land before the CTA exits (the last layer's chunks,
            // or after a failure whatever was issued)
            for (int c = 0; c < n_chunks; ++c) {
                const long long t0 = clock64();
                while (!mbar_try_parity(&full_bar[c], (n_layers - 1) & 1) && clock64() - t0 < limit) {
                }
            }
        }
        __syncwarp();
        return;  // the producer warp takes no part in the named barriers below
    }

    // ---------------------------------------------------------------- consumer warps
    // Lanes l and l ^ 16 share one 32-k slice (slice 16 * warp + (l & 15)); in every chunk
    // lane l takes the rows 2i + (l >> 4), as in the bulk-copy GEMV kernel.
    const int hh = lane >> 4;
    const int slice = 16 * warp + (lane & 15);
    const int col = (slice * 32) / (nvec * 32 / ngroups);  // this lane's scale column
    const W4Keys keys = w4_keys();

    // ------------------------------------------------- add-RMSNorm 0, by every CTA
    float hres = 0.f;  // thread tid < n_cnt: h of row n_begin + tid (float of bf16)
    {
        uint4 hv[kStepRmsMaxVpt], wv[kStepRmsMaxVpt];
        load_norm_weight(layers[0].rms_weight, nvec_h, rms_vpt, rms_threads, wv);
#pragma unroll
        for (int i = 0; i < kStepRmsMaxVpt; ++i) {
            const int v = tid + i * rms_threads;
            hv[i] = make_uint4(0u, 0u, 0u, 0u);
            if (tid < rms_threads && i < rms_vpt && v < nvec_h) {
                const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(x0) + v);
                const uint4 rv = __ldcg(reinterpret_cast<const uint4 *>(residual) + v);
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
                uint32_t hw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    hw[j] = pack_bf16x2(bf16lo(xw[j]) + bf16lo(rw[j]), bf16hi(xw[j]) + bf16hi(rw[j]));
                hv[i] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            }
        }
        if (tid < n_cnt) {
            const int n = n_begin + tid;
            const __nv_bfloat16 h = __float2bfloat16_rn(bf16lo(x0[n]) + bf16lo(__ldcg(residual + n)));
            hres = __bfloat162float(h);
        }
        norm_row(hv, wv, nvec_h, rms_vpt, rms_threads, inv_hidden, eps, warp_ss, s_normed, ncons);
        named_bar_sync(1, ncons);
        if (tid < n_cnt) static_cast<uint16_t *>(layers[0].normed)[n_begin + tid] = s_normed16[n_begin + tid];
    }

    for (int l = 0; l < n_layers; ++l) {
        const fd_step_layer &Ly = layers[l];
        const bool fold = l + 1 < n_layers;
        const bool failed_in = abort_flag != 0;
        // ------------------------------------------------- the activation slice
        Act16 act;
        {
            GateUpHalf gu;
            const uint16_t *g = static_cast<const uint16_t *>(Ly.gate);
            const uint16_t *u = static_cast<const uint16_t *>(Ly.up);
            const uint4 *g4 = reinterpret_cast<const uint4 *>(g + slice * 32 + 16 * hh);
            const uint4 *u4 = reinterpret_cast<const uint4 *>(u + slice * 32 + 16 * hh);
            gu.g[0] = ldg_v4(g4);
            gu.g[1] = ldg_v4(g4 + 1);
            gu.u[0] = ldg_v4(u4);
            gu.u[1] = ldg_v4(u4 + 1);
            encode_q16_pair(gu, hh, act);
        }
        // ------------------------------------------------- the CTA's rows of y_l
        for (int c = 0; c < n_chunks; ++c) {
            float part[kRowsPerLane];
            const bool ok = mbar_wait_bounded(&full_bar[c], l & 1, &abort_flag, limit);
            const int rows_valid = min(kStepR, n_cnt - c * kStepR);
            const uint4 *wst = reinterpret_cast<const uint4 *>(smem + (size_t)c * kStepR * w_row_bytes) +
                               slice + hh * nvec;
            const uint16_t *sst = reinterpret_cast<const uint16_t *>(s_region + (size_t)c * kStepR * s_row_bytes) +
                                  col + hh * ngroups;
            if (ok && rows_valid == kStepR) {
#pragma unroll
                for (int i = 0; i < kRowsPerLane; ++i) {
                    const uint4 wv = wst[2 * i * nvec];
                    const float scv = __uint_as_float((uint32_t)sst[2 * i * ngroups] << 16);
                    float d[1];
                    dot32<1>(&act, wv, keys, scv, d);
                    part[i] = d[0];
                }
            } else {
#pragma unroll
                for (int i = 0; i < kRowsPerLane; ++i) {
                    if (ok && 2 * i + hh < rows_valid) {
                        const uint4 wv = wst[2 * i * nvec];
                        const float scv = __uint_as_float((uint32_t)sst[2 * i * ngroups] << 16);
                        float d[1];
                        dot32<1>(&act, wv, keys, scv, d);
                        part[i] = d[0];
                    } else {
                        part[i] = 0.f;
                    }
                }
            }
            // the stage's reads before the producer's next bulk copy overwrites it
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[c]);
            const float wsum = half_reduce_scatter<kRowsPerLane>(part, lane);
            if (((lane & 15) & (kLanesPerValue - 1)) == 0) {
                const int r = 2 * ((lane & 15) / kLanesPerValue) + hh;
                red[(size_t)warp * kWindowRows + (c * kStepR + r)] = wsum;
            }
        }
        named_bar_sync(1, ncons);
        // ------------------------------------------------- y_l, and h = bf16(y_l + residual)
        const bool fail = failed_in || abort_flag != 0;
        uint32_t *hbuf = hrows + (size_t)(l & 1) * N;
        const uint32_t tag = (uint32_t)(l + 1);
        if (tid < n_cnt) {
            const int n = n_begin + tid;
            const float acc = sum_partials(red + tid, ncw, kWindowRows);
            const __nv_bfloat16 yb = __float2bfloat16_rn(acc);
            const uint16_t ybits = *reinterpret_cast<const uint16_t *>(&yb);
            static_cast<uint16_t *>(Ly.y)[n] = fail ? (uint16_t)0x7FC0 : ybits;
            if (fold) {
                // the rounded y as the next layer's add reads it
                const __nv_bfloat16 h = __float2bfloat16_rn(bf16lo(ybits) + hres);
                const uint16_t hbits = fail ? (uint16_t)0x7FC0 : *reinterpret_cast<const uint16_t *>(&h);
                st_relaxed_u32(hbuf + n, (tag << 16) | hbits);
                hres = bf16lo(hbits);
            }
        }
        if (!fold) break;
        // ------------------------------------------------- add-RMSNorm l + 1, whole row
        uint4 wv[kStepRmsMaxVpt], hv[kStepRmsMaxVpt];
        load_norm_weight(layers[l + 1].rms_weight, nvec_h, rms_vpt, rms_threads, wv);
        named_bar_sync(1, ncons);
        if (tid == 0) {
            if (!(withhold && l == 0)) atomicAdd(&count[l], 1u);
            if (!wait_counter(&count[l], (unsigned)grid, limit)) abort_flag = 1;
        }
        named_bar_sync(1, ncons);
        bool got = true;
#pragma unroll
        for (int i = 0; i < kStepRmsMaxVpt; ++i) {
            const int v = tid + i * rms_threads;
            hv[i] = make_uint4(0u, 0u, 0u, 0u);
            if (tid < rms_threads && i < rms_vpt && v < nvec_h) got &= read_tagged_vec(hbuf, v, tag, &hv[i], limit);
        }
        if (!got) {
            record_wait_timeout();
            abort_flag = 1;
        }
        norm_row(hv, wv, nvec_h, rms_vpt, rms_threads, inv_hidden, eps, warp_ss, s_normed, ncons);
        named_bar_sync(1, ncons);
        if (tid < n_cnt) {
            const int n = n_begin + tid;
            static_cast<uint16_t *>(layers[l + 1].normed)[n] =
                abort_flag != 0 ? (uint16_t)0x7FC0 : s_normed16[n];
        }
    }
    // ------------------------------------------------- the residual: h of the last layer
    // Every CTA reads the whole input residual for add-RMSNorm 0 before it publishes h_1,
    // and a CTA gets here only after reading every CTA's h_1, so no CTA still needs the
    // input rows. A single layer has no h_1: its CTAs count in here instead.
    if (n_layers == 1) {
        named_bar_sync(1, ncons);
        if (tid == 0) {
            if (!withhold) atomicAdd(&count[0], 1u);
            if (!wait_counter(&count[0], (unsigned)grid, limit)) abort_flag = 1;
        }
        named_bar_sync(1, ncons);
    }
    if (tid < n_cnt) {
        const __nv_bfloat16 h = __float2bfloat16_rn(hres);  // exact: hres is a bf16 value
        residual[n_begin + tid] = abort_flag != 0 ? (uint16_t)0x7FC0 : *reinterpret_cast<const uint16_t *>(&h);
    }
}

template <int NVEC_C, int NG_C>
cudaError_t launch_shape(const DeviceInfo &di, const fd_step_layer *layers, int n_layers,
                         const void *x0, void *residual, float eps, int K, int N, int group,
                         int rms_vpt, int rms_threads, void *scratch, cudaStream_t stream,
                         bool *launched) {
    static std::atomic<uint64_t> attr_done{0};
    static std::atomic<int> static_smem_cache{-1};
    auto kern = decode_step_kernel<NVEC_C, NG_C>;
    int static_smem = static_smem_cache.load(std::memory_order_relaxed);
    if (static_smem < 0) {
        cudaFuncAttributes fa;
        cudaError_t err = cudaFuncGetAttributes(&fa, kern);
        if (err != cudaSuccess) return err;
        static_smem = (int)fa.sharedSizeBytes;
        static_smem_cache.store(static_smem, std::memory_order_relaxed);
    }
    const size_t budget = (size_t)di.max_smem_optin - (size_t)static_smem;
    StepPlan plan{};
    if (!plan_step(di.sm_count, budget, K, N, group, &plan)) return cudaSuccess;  // not launched
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)budget);
        if (err != cudaSuccess) return err;
        attr_done.fetch_or(bit, std::memory_order_acq_rel);
    }
    // the counters and every tag start at zero
    err = cudaMemsetAsync(scratch, 0, FD_STEP_SCRATCH_BYTES(n_layers, N), stream);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid);
    cfg.blockDim = dim3((unsigned)(2 * NVEC_C + 32));
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident at once, or an error
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    *launched = true;
    err = cudaLaunchKernelEx(&cfg, kern, layers, n_layers, static_cast<const uint16_t *>(x0),
                             static_cast<uint16_t *>(residual), eps, N, plan.rows_base,
                             plan.rows_extra, plan.S, plan.w_rows, rms_vpt, rms_threads,
                             static_cast<unsigned *>(scratch),
                             reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(scratch) +
                                                          FD_STEP_SCRATCH_HROWS_OFFSET(n_layers)),
                             (launch_flags() & FD_LAUNCH_TEST_WAIT_TIMEOUT) ? 1 : 0);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_step(const fd_step_layer *layers, int n_layers, const void *x0,
                               void *residual, float eps, int hidden, int inter, int group,
                               void *scratch, cudaStream_t stream, bool *launched) {
    *launched = false;
    int vpt = 0, threads = 0;
    if (!step_shape_supported(hidden, inter, group) || !step_rms_shape(hidden, &vpt, &threads))
        return cudaSuccess;
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    return launch_shape<14336 / 32, 14336 / 128>(di, layers, n_layers, x0, residual, eps, inter,
                                                  hidden, group, vpt, threads, scratch, stream,
                                                  launched);
}

FD_DEFINE_STATUS_ACCESSOR(status_decode_step)

}  // namespace fd
