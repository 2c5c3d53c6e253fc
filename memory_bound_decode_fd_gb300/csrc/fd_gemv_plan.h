// fd_gemv_plan.h - launch planning of the bulk-copy GEMV kernel (fd_gemv_tma.cu): grid,
// rows per CTA, shared-memory layout and CTAs per SM, as a pure host function of the
// device's facts and the call's shape (no CUDA calls, so it is testable without a GPU).
#pragma once

#include <stddef.h>

namespace fd {

struct TmaPlanInput {
    // device and compiled-kernel facts
    int sm_count, smem_optin, smem_per_sm, smem_reserved, static_smem, regs;
    // the call and the kernel's compile-time shape
    int M, K, N, group;
    int MB;          // activation rows per pass
    int LPS;         // consumer lanes per 32-k slice
    int R;           // weight rows per chunk
    int max_stages;  // mbarrier slots
    int plain;       // plain activation (x, K*2 bytes) instead of gate and up (K*4 bytes)
};

struct TmaPlan {
    int grid, rows_base, rows_extra;  // CTAs; rows per CTA (the first rows_extra get one more)
    int S;                            // stages (mbarrier pairs)
    int w_rows;                       // weight rows of shared memory (stage s: rows [sR, sR + R))
    int act_first_stage;              // M == 1: first stage the activation copy overlays
    int ring;                         // stages are reused (else one stage per chunk)
    int per_sm;                       // resident CTAs per SM the plan was made for
    size_t smem;                      // dynamic shared memory per CTA
};

// Fills `p`; false if the kernel cannot run this call (the ring would be too small).
bool plan_gemv_tma(const TmaPlanInput &in, TmaPlan *p);

}  // namespace fd
