// fd_tma.cuh - mbarrier and bulk-copy (TMA, non-tensor) wrappers in inline PTX, and a
// bounded wait. Every wait in this library gives up after kWaitLimitCycles SM clocks
// (about a second) or as soon as another thread of the CTA has given up, so a lost
// completion can never hang the GPU; the caller then records the failure and exits.
#pragma once

#include "fd_internal.h"

namespace fd {

constexpr long long kWaitLimitCycles = 1ll << 31;
// The limit under FD_LAUNCH_TEST_WAIT_TIMEOUT (about 0.5 ms at 2 GHz).
constexpr long long kTestWaitLimitCycles = 1ll << 20;

// Set by a kernel of this translation unit whose bounded wait gave up
// (FD_DEVICE_STATUS_WAIT_TIMEOUT); read and cleared on the host through the accessor that
// FD_DEFINE_STATUS_ACCESSOR defines in the same file (see fd_device_status in fd.h).
static __device__ unsigned int g_wait_status;

__device__ __forceinline__ void record_wait_timeout() {
    atomicOr(&g_wait_status, (unsigned)FD_DEVICE_STATUS_WAIT_TIMEOUT);
}

// Host accessor of this translation unit's status word: copies it to *out (pinned or
// pageable host memory) on `stream` and, with `clear`, zeroes it after the copy. The caller
// synchronises the stream.
#define FD_DEFINE_STATUS_ACCESSOR(name)                                                      \
    cudaError_t name(cudaStream_t stream, unsigned *out, bool clear) {                       \
        cudaError_t err = cudaMemcpyFromSymbolAsync(out, g_wait_status, sizeof(unsigned), 0, \
                                                    cudaMemcpyDeviceToHost, stream);         \
        if (err != cudaSuccess || !clear) return err;                                        \
        void *p = nullptr;                                                                   \
        err = cudaGetSymbolAddress(&p, g_wait_status);                                       \
        if (err != cudaSuccess) return err;                                                  \
        return cudaMemsetAsync(p, 0, sizeof(unsigned), stream);                              \
    }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes the initialised barriers visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// True once the phase with parity `parity` has completed.
__device__ __forceinline__ bool mbar_test_parity(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Like mbar_test_parity, but the hardware may suspend the thread for a short,
// system-defined time while the phase is incomplete (no issue slots spent spinning).
__device__ __forceinline__ bool mbar_try_parity(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Address (shared window, 32-bit) forms of mbar_try_parity and mbar_arrive.
__device__ __forceinline__ bool mbar_try_parity_at(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ void mbar_arrive_at(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Slow path of mbar_wait_bounded (kept out of line so the fast path stays small):
// several suspending polls between checks of the abort flag and the cycle budget.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t *bar, uint32_t parity,
                                                   volatile int *abort_flag, long long limit) {
    const long long t0 = clock64();
    while (true) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (mbar_try_parity(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            *abort_flag = 1;
            record_wait_timeout();
            return false;
        }
    }
}

// Waits for the phase with parity `parity`. Returns false if the wait ran past `limit`
// SM clocks or `*abort_flag` became nonzero (another thread gave up); in the first case it
// also sets `*abort_flag` and the translation unit's status word.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  volatile int *abort_flag,
                                                  long long limit = kWaitLimitCycles) {
    if (mbar_try_parity(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, abort_flag, limit);
}
__device__ __forceinline__ bool mbar_wait_bounded_at(uint32_t bar, uint32_t parity,
                                                     volatile int *abort_flag) {
    if (mbar_try_parity_at(bar, parity)) return true;
    return mbar_wait_slow(reinterpret_cast<uint64_t *>(__cvta_shared_to_generic(bar)), parity,
                          abort_flag, kWaitLimitCycles);
}

// Bulk copy global -> shared (this CTA), completion counted in bytes on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory (plain loads and
// stores) before later async-proxy accesses (bulk copies) to the same memory. Issued
// before releasing a buffer that a bulk copy will overwrite.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32-bit shared-memory (this CTA) loads and stores, volatile so that they stay ordered
// with the barrier waits around them.
__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Barrier over the first `threads` threads of the CTA (named barrier `id`, id != 0).
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace fd
