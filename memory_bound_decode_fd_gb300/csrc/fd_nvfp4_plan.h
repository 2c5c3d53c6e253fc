// fd_nvfp4_plan.h - launch planning of the NVFP4 block-scaled MMA kernel (fd_nvfp4.cu):
// the K split over a cluster, the padded batch and the shared-memory layout, as a pure
// host function (no CUDA calls, so it is testable without a GPU).
#pragma once

#include <stdint.h>

namespace fd {

constexpr int kNfRows = 128;          // weight rows per CTA (the MMA's M)
constexpr int kNfStageK = 256;        // k per copy stage: one 128-byte row of packed FP4
constexpr int kNfMmaK = 64;           // k per block-scaled MMA
constexpr uint32_t kNfWStage = kNfRows * kNfStageK / 2;  // weight bytes per stage: 16384
constexpr int kNfMaxKCta = 1024;      // k per CTA
constexpr int kNfMaxStages = kNfMaxKCta / kNfStageK;
constexpr int kNfMaxSplit = 8;        // CTAs per cluster along K
constexpr int kNfMaxK = kNfMaxKCta * kNfMaxSplit;
constexpr int kNfMaxBatch = 128;      // activation rows per launch (the MMA's N, padded)
constexpr uint32_t kNfTmemCols = 256; // accumulator (<= 128 columns) + scale factors (<= 128)
// Shared memory each CTA requests at least: with 80 KB a third CTA never fits on an SM
// (3 x (80 + 1) KB > 228 KB), so at most two share one and their 2 x 256 TMEM columns are
// always free. A third CTA would wait in tcgen05.alloc while the others of its cluster
// wait for it at a cluster barrier, which could hold every CTA involved.
constexpr uint32_t kNfMinSmem = 80 * 1024;

struct Nvfp4Plan {
    int split;      // CTAs per cluster along K
    int k_cta;      // k per CTA
    int stages;     // 256-k copy stages per CTA (all resident)
    int npad;       // the batch padded to the MMA's N (16, 32, 64 or 128)
    int n_tiles;    // 128-row weight tiles (clusters)
    uint32_t off_x, off_wsf, off_xsf;  // shared-memory offsets (weights at 0)
    uint32_t recv_bytes;               // the cluster reduction's buffer (from offset 0)
    uint32_t smem;                     // dynamic shared memory per CTA, with alignment slack
};

// The padded batch of `m` activation rows (1 <= m <= 128).
inline int nvfp4_npad(int m) { return m <= 16 ? 16 : m <= 32 ? 32 : m <= 64 ? 64 : 128; }

// The smallest split in {1, 2, 4, 8} whose K slice is a whole number of 256-k stages and
// at most 1024 k; 0 if there is none (K not a multiple of 256, or above 8192).
inline int nvfp4_split(int K) {
    if (K <= 0 || K % kNfStageK != 0) return 0;
    for (int s = 1; s <= kNfMaxSplit; s *= 2)
        if (K % (kNfStageK * s) == 0 && K / s <= kNfMaxKCta) return s;
    return 0;
}

// Fills `p` for one launch of `m` (1..128) activation rows; false when the shape is
// outside the kernel's rules or its shared memory exceeds `smem_budget`.
inline bool plan_nvfp4(int m, int K, int N, int smem_budget, Nvfp4Plan *p) {
    if (m < 1 || m > kNfMaxBatch || N < 1) return false;
    const int split = nvfp4_split(K);
    if (split == 0) return false;
    p->split = split;
    p->k_cta = K / split;
    p->stages = p->k_cta / kNfStageK;
    p->npad = nvfp4_npad(m);
    p->n_tiles = (N + kNfRows - 1) / kNfRows;
    const uint32_t x_stage = (uint32_t)p->npad * kNfStageK / 2;
    const uint32_t sf_row = (uint32_t)p->k_cta / 16;
    p->off_x = (uint32_t)p->stages * kNfWStage;
    p->off_wsf = p->off_x + (uint32_t)p->stages * x_stage;
    p->off_xsf = p->off_wsf + (uint32_t)kNfRows * sf_row;
    const uint32_t end = p->off_xsf + (uint32_t)p->npad * sf_row;
    // [src rank][npad][128 / split] fp32: npad * 128 * 4 bytes for any split
    p->recv_bytes = (uint32_t)p->npad * kNfRows * 4;
    const uint32_t used = end > p->recv_bytes ? end : p->recv_bytes;
    p->smem = used + 1024;  // the kernel aligns its base to 1024 bytes
    if (p->smem < kNfMinSmem) p->smem = kNfMinSmem;
    return smem_budget > 0 && p->smem <= (uint32_t)smem_budget;
}

}  // namespace fd
