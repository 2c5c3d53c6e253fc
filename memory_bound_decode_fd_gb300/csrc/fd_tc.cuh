// fd_tc.cuh - inline-PTX wrappers for the Blackwell tensor-core path: tensor-map (tiled)
// bulk copies, fifth-generation tensor-core MMA (tcgen05) with its tensor-memory (TMEM)
// accumulator, and thread-block-cluster distributed shared memory.
//
// The mbarrier helpers and the bounded wait live in fd_tma.cuh.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; no driver call is made from device code)

#include "fd_tma.cuh"

namespace fd {

// ---------------------------------------------------------------- tensor-map copies

// 2D tiled copy global -> shared (this CTA) of the box at element coordinates (x, y);
// completion is counted in bytes (the full box, including zero-filled out-of-range
// elements) on `bar`. `map` must be a __grid_constant__ kernel parameter.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tensor memory

// Allocates `ncols` (a power of two >= 32) TMEM columns for this CTA; the warp that
// calls it (all 32 lanes) writes the base address to *dst. Must be freed by the same
// warp with tmem_dealloc.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}

// Ordering of tcgen05 operations across a thread synchronisation (barrier or mbarrier).
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T for one K = 16 step, bf16/fp16 operands, issued by
// one thread. `accumulate` = 0 overwrites D.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= (A * SFA) * (B * SFB)^T for one K = 64 step of packed FP4 (E2M1) operands
// with one E4M3 scale per 16 elements of each row (block-scaled MMA, scale vectors of 4 per
// K = 64), issued by one thread. `sfa_tmem` / `sfb_tmem` are the TMEM addresses of the
// scale factors of this step (4 columns each, see tmem_st_x4).
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem,
                                            uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
        "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// One arrival on `bar` once every tcgen05.mma this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Each lane of the warp reads 8 consecutive 32-bit columns of its own TMEM lane
// (the warp may only address lanes 32 * (warp % 4) .. + 31).
__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr)
        : "memory");
}
// The same with 16 consecutive columns.
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Each lane of the warp writes 4 consecutive 32-bit columns of its own TMEM lane (the warp
// may only address lanes 32 * (warp % 4) .. + 31); tmem_st_wait makes them complete.
__device__ __forceinline__ void tmem_st_x4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2,
                                           uint32_t v3) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
                 "r"(v0), "r"(v1), "r"(v2), "r"(v3)
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, no swizzle ("interleaved" 8 x 16-byte core
// matrices, each 128 contiguous bytes). For a K-major operand: `lbo` = byte distance
// between the two core matrices adjacent along K, `sbo` = byte distance between
// adjacent 8-row groups. Bits 46-47 hold the descriptor version (1).
__device__ __forceinline__ uint64_t smem_desc_interleaved(uint32_t saddr, uint32_t lbo,
                                                          uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzle layout
// that a tensor-map copy with CU_TENSOR_MAP_SWIZZLE_128B writes: rows of 128 bytes, 16-byte
// chunk c of row r stored at chunk c ^ (r & 7), 8-row atoms of 1024 bytes; `sbo` is the
// stride between 8-row groups (1024 when the atoms are contiguous, a multiple of 1024
// otherwise). The leading-dimension offset is unused for this layout (1).
// The atom must be 1024-byte aligned; a K step inside the 128-byte row advances the start
// address by its byte offset (the swizzle is applied to the absolute address).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t sbo = 1024u) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::mxf4nvf4: E2M1 A and B (packed FP4), UE4M3 scale
// factors (one per 16 elements), fp32 D, both K-major, M x N tile, scale-factor ids 0.
__host__ __device__ constexpr uint32_t idesc_nvf4(int m, int n) {
    return (1u << 7)                        // A format: E2M1
           | (1u << 10)                     // B format: E2M1
           | ((uint32_t)(n >> 3) << 17)     // N / 8
           | (0u << 23)                     // scale format: UE4M3
           | ((uint32_t)(m >> 4) << 24);    // M / 16
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, both K-major, M x N tile.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
    return (1u << 4)                        // D format: f32
           | (1u << 7)                      // A format: bf16
           | (1u << 10)                     // B format: bf16
           | ((uint32_t)(n >> 3) << 17)     // N / 8
           | ((uint32_t)(m >> 4) << 24);    // M / 16
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Barrier over every thread of every CTA of the cluster, with release/acquire ordering
// of shared::cluster memory. Every thread of the CTA must call it the same number of
// times.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from this CTA's
// shared memory `src` to the shared memory of a CTA of the cluster: `dst` and that CTA's
// mbarrier `bar` are map_to_rank addresses; the copy completes `bytes` on `bar`.
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst, uint32_t src, uint32_t bytes,
                                               uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(dst),
        "r"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// ---------------------------------------------------------------- packed bf16 math

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}


}  // namespace fd
