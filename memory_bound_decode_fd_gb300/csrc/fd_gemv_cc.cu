// fd_gemv_cc.cu - SwiGLU-prologue W4A16 GEMV on the CUDA cores (any M, tuned for M = 1).
//
// y[m, n] = bf16( [residual[m, n] +] sum_k silu(g[m, k]) * u[m, k] * q[n, k] * s[n, k / group] )
//
// With up == nullptr the activation is gate itself (a plain W4A16 GEMV, the horizontal
// gate/up projection), and the output rows may be split between two tensors (out_at).
//
// Sources: "09 - Operator fusion", section 5 (taxonomy item 4, GEMM prologue fusion: the
// dequantisation happens as the weights are loaded, so only int4 crosses HBM; "The fusion
// boundary problem": act = silu(gate) * up feeds out = act @ W_down). "PyTorch Community
// Proposes Fusion Fix ..." ("Reproduction and analysis": an M = 1 matmul must not
// materialise its (1, K, N) product; "Fix proposal": materialise the small input first -
// here that input, a = silu(g) * u, lives in registers).
//
// Work decomposition (one CTA per SM, persistent):
//   * Thread t of a CTA owns the weight vector positions p = t + v * T (v < VPT) of every
//     row: each position is 16 bytes = 4 words = 32 consecutive k, inside one scale group.
//     So thread t needs a[m, k] only for its own k, and computes silu(g) * u once per
//     m-chunk straight into registers. Nothing is staged through HBM.
//   * The CTA owns a contiguous range of output rows n; it walks them in chunks of R rows.
//     Each thread streams its own 16-byte slot of each row (and the 2-byte scale that
//     belongs to it) with cp.async into a private ring of S stages in shared memory, S - 1
//     chunks ahead of the math. Slots are thread-private, so the ring needs no barriers:
//     cp.async.wait_group orders each thread's own copies.
//   * Math per 32-bit word: 2 lop3 (even/odd nibble bytes, fd_w4_unpack.cuh) + 4 dp2a
//     against the block-scaled int16 activations (fd_gemv_common.cuh), exact int32 sums
//     per 32-k slice; the activation and group scales multiply the slice's sum.
//   * Reduction: each lane holds R x MB partials per chunk; a butterfly reduce-scatter
//     over the warp (V - 1 + log2(32 / V) shuffles for V values) leaves one warp sum per
//     (row, m) in shared memory; the CTA sums over warps, adds the residual if one is
//     given, and stores bf16 once per output.
//   * M > MB: the CTA repeats its rows for each chunk of MB activation rows (weights are
//     then read with an evict-last L2 policy so the repeats hit L2).
#include <atomic>

#include "fd_internal.h"
#include "fd_gemv_common.cuh"

namespace fd {
namespace {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async_16(void *dst, const void *src, int src_bytes,
                                            uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;"
                 :
                 : "r"(smem_addr(dst)), "l"(src), "r"(src_bytes), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void cp_async_4(void *dst, const void *src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;"
                 :
                 : "r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Shared memory layout (dynamic):
//   wring  uint4    [S][R][VPT][T]   weight slots
//   sring  uint32_t [S][R][VPT][T]   scale slots (the bf16 scale in the low or high half)
//   red    float    [nwarps][kWindowRows][MB]
template <int VPT, int MB, int R, int S>
__global__ void __launch_bounds__(512, 1)
    gemv_cc_kernel(const uint16_t *__restrict__ gate, const uint16_t *__restrict__ up,
                   const uint4 *__restrict__ qweight, const uint16_t *__restrict__ scales,
                   const uint16_t *residual, uint16_t *out, uint16_t *out2, int split, int ldo,
                   int M, int K, int N, int group, int rows_base,
                   int rows_extra, int weights_evict_first) {
    static_assert(R * MB <= 32 && (R * MB & (R * MB - 1)) == 0, "R*MB: power of 2, <= 32");
    static_assert(kWindowRows % R == 0, "window must hold whole chunks");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int T = blockDim.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = T >> 5;
    const int nvec = K >> 5;           // 16-byte weight vectors per row
    const int ngroups = K / group;

    uint4 *wring = reinterpret_cast<uint4 *>(smem_raw);
    uint32_t *sring = reinterpret_cast<uint32_t *>(wring + (size_t)S * R * VPT * T);
    float *red = reinterpret_cast<float *>(sring + (size_t)S * R * VPT * T);

    const int b = blockIdx.x;
    const int n_begin = b * rows_base + min(b, rows_extra);
    const int n_cnt = rows_base + (b < rows_extra ? 1 : 0);
    const int n_chunks = (n_cnt + R - 1) / R;
    const int m_chunks = (M + MB - 1) / MB;
    const int total = n_chunks * m_chunks;

    const uint64_t pol = weights_evict_first ? policy_evict_first() : policy_evict_last();

    int pos[VPT];
    bool active[VPT];
    int sidx_col[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        pos[v] = tid + v * T;
        active[v] = pos[v] < nvec;
        sidx_col[v] = active[v] ? (pos[v] * 32) / group : 0;
    }

    // Issue the copies of work item c (m-chunk major: c = mc * n_chunks + nc) into ring
    // stage c % S. Rows past the CTA's range are zero-filled (no bytes read).
    auto issue = [&](int c) {
        if (c < total) {
            const int nc = c % n_chunks;
            const int stage = c % S;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int n_local = nc * R + r;
                const bool row_ok = n_local < n_cnt;
                const int n = n_begin + (row_ok ? n_local : 0);
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    if (!active[v]) continue;
                    const size_t slot = ((size_t)(stage * R + r) * VPT + v) * T + tid;
                    const uint4 *src = qweight + (size_t)n * nvec + pos[v];
                    cp_async_16(&wring[slot], src, row_ok ? 16 : 0, pol);
                    const size_t sidx = (size_t)n * ngroups + sidx_col[v];
                    const uint16_t *ssrc = scales + (sidx & ~(size_t)1);
                    const int sbytes = row_ok ? ((sidx & 1) ? 4 : 2) : 0;
                    cp_async_4(&sring[slot], ssrc, sbytes);
                }
            }
        }
        cp_async_commit();  // always commit (possibly empty) so group counting is uniform
    };

    // gate/up may come from the previous kernel in the stream (programmatic dependent
    // launch); the weights are read only after this wait too.
    grid_dep_wait();
    grid_dep_launch();

#pragma unroll
    for (int c = 0; c < S - 1; ++c) issue(c);

    const W4Keys keys = w4_keys();
    Act16 act[VPT][MB];
    int window_base = 0;  // first local row of the current flush window

    for (int c = 0; c < total; ++c) {
        issue(c + S - 1);
        const int mc = c / n_chunks;
        const int nc = c % n_chunks;
        const int m0 = mc * MB;

        if (nc == 0) {
            // New m-chunk: build a = silu(g) * u for this thread's k and rows m0..m0+MB-1.
#pragma unroll
            for (int mb = 0; mb < MB; ++mb) {
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    const size_t off = (size_t)(m0 + mb) * K + (size_t)pos[v] * 32;
                    if (!(active[v] && m0 + mb < M)) {
                        zero_activation(act[v][mb]);
                    } else if (up) {
                        load_activation_q16(gate, up, off, act[v][mb]);
                    } else {  // a plain activation (no SwiGLU): gate holds x
                        const uint4 *x4 = reinterpret_cast<const uint4 *>(gate + off);
                        const uint4 x[4] = {x4[0], x4[1], x4[2], x4[3]};
                        encode_plain(x, act[v][mb]);
                    }
                }
            }
        }

        cp_async_wait<S - 1>();  // this thread's copies for item c have landed

        const int stage = c % S;
        float part[R * MB];
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int mb = 0; mb < MB; ++mb) part[r * MB + mb] = 0.f;
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                if (!active[v]) continue;
                const size_t slot = ((size_t)(stage * R + r) * VPT + v) * T + tid;
                const uint4 wv = wring[slot];
                const uint32_t sw = sring[slot];
                const size_t sidx = (size_t)(n_begin + nc * R + r) * ngroups + sidx_col[v];
                const float s = (sidx & 1) ? bf16hi(sw) : bf16lo(sw);
                float d[MB];
                dot32<MB>(act[v], wv, keys, s, d);
#pragma unroll
                for (int mb = 0; mb < MB; ++mb) part[r * MB + mb] += d[mb];
            }
        }

        const float wsum = warp_reduce_scatter<R * MB>(part, lane);
        constexpr int kLanesPerValue = 32 / (R * MB);
        if ((lane & (kLanesPerValue - 1)) == 0) {
            const int idx = lane / kLanesPerValue;  // = r * MB + mb
            const int r = idx / MB, mb = idx % MB;
            const int row_in_window = nc * R + r - window_base;
            red[((size_t)warp * kWindowRows + row_in_window) * MB + mb] = wsum;
        }

        const int rows_done = (nc + 1) * R;
        const bool last_chunk = (nc == n_chunks - 1);
        if (rows_done - window_base == kWindowRows || last_chunk) {
            __syncthreads();
            const int rows_in_window = min(rows_done, n_cnt) - window_base;
            for (int i = tid; i < rows_in_window * MB; i += T) {
                const int row = i / MB, mb = i % MB;
                float acc =
                    sum_partials(red + (size_t)row * MB + mb, nwarps, kWindowRows * MB);
                if (m0 + mb < M) {
                    const int n = n_begin + window_base + row;
                    if (residual) acc += bf16lo(residual[(size_t)(m0 + mb) * N + n]);
                    __nv_bfloat16 y = __float2bfloat16_rn(acc);
                    *out_at(out, out2, split, ldo, m0 + mb, n) = *reinterpret_cast<uint16_t *>(&y);
                }
            }
            __syncthreads();
            window_base = last_chunk ? 0 : rows_done;
        }
    }
    cp_async_wait<0>();
}

template <int VPT, int MB, int R, int S>
size_t gemv_smem_bytes(int T) {
    return (size_t)S * R * VPT * T * (16 + 4) + (size_t)(T / 32) * kWindowRows * MB * 4;
}

int threads_for(int K, int VPT) {
    const int nvec = K / 32;
    const int T = (nvec + VPT - 1) / VPT;
    return (T + 31) / 32 * 32;
}

// Raises the kernel's dynamic shared memory limit once per device (to the opt-in limit
// less the kernel's static shared memory).
template <typename Kern>
cudaError_t ensure_smem_attr(Kern kern, size_t smem, std::atomic<uint64_t> &done) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    int max_optin = 0;
    err = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (err != cudaSuccess) return err;
    cudaFuncAttributes fa;
    err = cudaFuncGetAttributes(&fa, kern);
    if (err != cudaSuccess) return err;
    const int limit = max_optin - (int)fa.sharedSizeBytes;
    if ((size_t)limit < smem) return cudaErrorInvalidConfiguration;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    done.fetch_or(bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

template <int VPT, int MB, int R, int S>
cudaError_t launch_cfg(const DeviceInfo &di, const void *gate, const void *up,
                       const void *qweight, const void *scales, const void *residual,
                       GemvOut o, int M, int K, int N, int group, cudaStream_t stream) {
    static std::atomic<uint64_t> attr_done{0};
    const int T = threads_for(K, VPT);
    const size_t smem = gemv_smem_bytes<VPT, MB, R, S>(T);
    auto kern = gemv_cc_kernel<VPT, MB, R, S>;
    cudaError_t err = ensure_smem_attr(kern, smem, attr_done);
    if (err != cudaSuccess) return err;
    // One CTA per SM; fewer when there are not enough rows for a chunk each.
    int grid = di.sm_count;
    if ((long long)grid * R > N) grid = (N + R - 1) / R;
    if (grid < 1) grid = 1;
    const int rows_base = N / grid;
    const int rows_extra = N % grid;
    const int evict_first = (M <= MB) ? 1 : 0;
    err = launch_kernel(kern, dim3(grid), dim3(T), smem, stream, 1,
                        static_cast<const uint16_t *>(gate), static_cast<const uint16_t *>(up),
                        static_cast<const uint4 *>(qweight),
                        static_cast<const uint16_t *>(scales),
                        static_cast<const uint16_t *>(residual), static_cast<uint16_t *>(o.out),
                        static_cast<uint16_t *>(o.out2), o.split, o.ldo, M, K, N, group,
                        rows_base, rows_extra, evict_first);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace

// Picks the deepest ring that fits the SM's shared memory, for the M = 1 kernel (MB = 1)
// or the M > 1 kernel (MB = 2), with one (K <= 16384) or two (K <= 32768) weight vector
// positions per thread.
cudaError_t launch_gemv_cc(const void *gate, const void *up, const void *qweight,
                           const void *scales, const void *residual, GemvOut o, int M, int K,
                           int N, int group, cudaStream_t stream) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const size_t limit = (size_t)di.max_smem_optin;
#define FD_TRY(VPT, MB, R, S)                                                              \
    if (gemv_smem_bytes<VPT, MB, R, S>(threads_for(K, VPT)) <= limit)                      \
        return launch_cfg<VPT, MB, R, S>(di, gate, up, qweight, scales, residual, o, M, K, N, \
                                         group, stream);
    const bool wide = K / 32 > 512;  // more than 512 vector positions: two per thread
    if (!wide && M == 1) {
        FD_TRY(1, 1, 8, 4)
        FD_TRY(1, 1, 8, 3)
        FD_TRY(1, 1, 4, 3)
        FD_TRY(1, 1, 4, 2)
    } else if (!wide) {
        FD_TRY(1, 2, 8, 3)
        FD_TRY(1, 2, 4, 3)
        FD_TRY(1, 2, 4, 2)
    } else {
        FD_TRY(2, 1, 4, 3)
        FD_TRY(2, 1, 4, 2)
        FD_TRY(2, 1, 2, 2)
    }
#undef FD_TRY
    return cudaErrorInvalidConfiguration;
}

}  // namespace fd
