// fd_nvfp4_plan.h - launch planning of the NVFP4 block-scaled MMA kernel (fd_nvfp4.cu):
// the K split over a cluster, the padded batch, the shared-memory layout and the tensor
// memory, as a pure host function (no CUDA calls, so it is testable without a GPU).
#pragma once

#include <cuda_runtime.h>  // __host__ __device__
#include <stdint.h>

namespace fd {

constexpr int kNfRows = 128;          // weight rows per CTA (the MMA's M)
constexpr int kNfStageK = 256;        // k per copy stage: one 128-byte row of packed FP4
constexpr int kNfMmaK = 64;           // k per block-scaled MMA
constexpr uint32_t kNfWStage = kNfRows * kNfStageK / 2;  // weight bytes per stage: 16384
constexpr int kNfMaxStages = 12;      // stages per CTA (all resident; mbarrier slots)
constexpr int kNfMaxSplit = 8;        // CTAs per cluster along K (portable cluster size)
constexpr int kNfMaxK = 16384;        // checked by the C ABI (FD_NVFP4_MAX_K)
constexpr int kNfMaxBatch = 128;      // activation rows per launch (the MMA's N, padded)
constexpr uint32_t kNfSfCol0 = 128;   // TMEM column of the first scale factors (D below it)
constexpr uint32_t kNfSfColsPerStage = 32;  // 4 K = 64 steps x (4 weight + 4 activation)

struct Nvfp4Plan {
    int split;      // CTAs per cluster along K
    int s_total;    // 256-k stages in K
    int max_stages; // stages of the largest K slice (rank r: stages [r S / split, (r+1) S / split))
    int npad;       // the batch padded to the MMA's N (16, 32, 64 or 128)
    int n_tiles;    // 128-row weight tiles (clusters)
    int tmem_cols;  // 256 or 512
    int cols_own;   // output columns (activation rows) each cluster rank finishes: ceil(npad / split)
    uint32_t sf_row;                   // scale bytes per row copied (max_stages x 16)
    uint32_t off_x, off_wsf, off_xsf;  // shared-memory offsets (weights at 0)
    uint32_t recv_bytes;               // the cluster reduction's buffers (from offset 0)
    uint32_t smem;                     // dynamic shared memory per CTA, with alignment slack
};

// The padded batch of `m` activation rows (1 <= m <= 128).
inline int nvfp4_npad(int m) { return m <= 16 ? 16 : m <= 32 ? 32 : m <= 64 ? 64 : 128; }

// First stage of rank r's K slice (the slice is [first(r), first(r + 1))).
__host__ __device__ inline int nvfp4_first_stage(int r, int s_total, int split) {
    return (int)((long long)r * s_total / split);
}

// Fills `p` for one launch of `m` (1..128) activation rows with K split over `split` CTAs;
// false when the shape is outside the kernel's rules for that split or its shared memory
// exceeds `smem_budget`.
inline bool plan_nvfp4_split(int m, int K, int N, int split, int smem_budget, Nvfp4Plan *p) {
    if (m < 1 || m > kNfMaxBatch || N < 1 || K <= 0 || K % kNfStageK != 0 || K > kNfMaxK)
        return false;
    if (split < 1 || split > kNfMaxSplit || split > K / kNfStageK) return false;
    p->split = split;
    p->s_total = K / kNfStageK;
    p->max_stages = (p->s_total + split - 1) / split;
    // tensor memory: the accumulator below column 128, scale columns above it
    if (p->max_stages > kNfMaxStages ||
        kNfSfCol0 + kNfSfColsPerStage * (uint32_t)p->max_stages > 512u)
        return false;
    p->npad = nvfp4_npad(m);
    p->n_tiles = (N + kNfRows - 1) / kNfRows;
    p->tmem_cols = kNfSfCol0 + kNfSfColsPerStage * p->max_stages <= 256 ? 256 : 512;
    p->cols_own = (p->npad + split - 1) / split;
    const uint32_t x_stage = (uint32_t)p->npad * kNfStageK / 2;
    p->sf_row = (uint32_t)p->max_stages * 16;
    p->off_x = (uint32_t)p->max_stages * kNfWStage;
    p->off_wsf = p->off_x + (uint32_t)p->max_stages * x_stage;
    p->off_xsf = p->off_wsf + (uint32_t)kNfRows * p->sf_row;
    const uint32_t end = p->off_xsf + (uint32_t)p->npad * p->sf_row;
    // receive slots [src rank][cols_own][128 rows] fp32, then the CTA's own accumulator as
    // `split` chunks [cols_own][128 rows] fp32
    p->recv_bytes = 2u * (uint32_t)split * (uint32_t)p->cols_own * kNfRows * 4;
    const uint32_t used = end > p->recv_bytes ? end : p->recv_bytes;
    p->smem = used + 1024;  // the kernel aligns its base to 1024 bytes
    // Shared memory bounds the CTAs per SM so that their TMEM allocations always fit the
    // SM's 512 columns: with 256 columns at most two CTAs (each >= 80 KB: three never fit
    // in 228 KB), with 512 at most one (each >= 116 KB). A CTA over the limit would wait
    // in tcgen05.alloc while the others of its cluster wait for it at a cluster barrier.
    const uint32_t min_smem = p->tmem_cols == 256 ? 80u * 1024 : 116u * 1024;
    if (p->smem < min_smem) p->smem = min_smem;
    return smem_budget > 0 && p->smem <= (uint32_t)smem_budget;
}

// The split for one launch: the smallest split whose K slices have at most 4 stages (256
// TMEM columns and ~110 KB of shared memory per CTA, so two CTAs share an SM), else the
// smallest split whose plan fits. Measured on GB300 for M=64 K=4096 N=6144 (per-CTA
// timelines): split 4 (192 CTAs of 4 stages) finishes first; split 2 streams through only
// 96 SMs, and splits 3, 6 and 8 leave clusters for a second wave. Returns false if no
// split fits.
inline bool plan_nvfp4(int m, int K, int N, int smem_budget, Nvfp4Plan *p) {
    for (int pass = 0; pass < 2; ++pass)
        for (int s = 1; s <= kNfMaxSplit; ++s) {
            Nvfp4Plan c{};
            if (!plan_nvfp4_split(m, K, N, s, smem_budget, &c)) continue;
            if (pass == 0 && c.max_stages > 4) continue;
            *p = c;
            return true;
        }
    return false;
}

}  // namespace fd
