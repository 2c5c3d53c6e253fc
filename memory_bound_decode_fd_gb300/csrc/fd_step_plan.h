// fd_step_plan.h - launch planning of the persistent decode-step kernel (fd_decode_step.cu):
// the shapes it runs, its row partition and shared-memory layout, and the block of the
// add-RMSNorm row arithmetic, as pure host functions (no CUDA calls, so they are testable
// without a GPU).
#pragma once

#include <stddef.h>

namespace fd {

constexpr int kStepR = 8;            // weight rows per chunk (the bulk-copy GEMV's chunk)
constexpr int kStepMaxStages = 8;    // chunks of one layer's rows per CTA (mbarrier slots)
constexpr int kStepWindowRows = 64;  // rows whose per-warp partials are held (one flush)
constexpr int kStepRmsMaxVpt = 4;    // 16-byte vectors per thread of the add-RMSNorm row

struct StepPlan {
    int grid, rows_base, rows_extra;  // CTAs; rows per CTA (the first rows_extra get one more)
    int S;                            // chunks of the largest CTA's rows, one stage each
    int w_rows;                       // weight rows of shared memory (all of a CTA's rows)
    size_t smem;                      // dynamic shared memory per CTA
};

// The decode shape: the down projection of K = 14336 (group 128), where the bulk-copy
// GEMV also runs one CTA per SM (928 threads), so the two share one row partition for any
// hidden; hidden: at most 64 rows per CTA (one flush of the cross-warp sums per layer).
inline bool step_shape_supported(int hidden, int inter, int group) {
    return inter == 14336 && group == 128 && hidden >= 8 && hidden % 8 == 0 &&
           hidden <= kStepWindowRows * 152;
}

// One CTA per SM (fewer when there are fewer than 8 rows per SM), the rows split as evenly
// as the bulk-copy GEMV splits them; every chunk of a CTA's rows resident at once, with the
// scales, the cross-warp sums of 2 K / 32 consumer warps and the whole normalised row.
// `budget`: dynamic shared memory a CTA may use.
inline bool plan_step(int sm_count, size_t budget, int K, int N, int group, StepPlan *p) {
    if (sm_count < 1 || K <= 0 || N <= 0 || group <= 0 || K % 32 != 0 || K % group != 0)
        return false;
    const int nvec = K / 32, ngroups = K / group;
    int grid = sm_count;
    if ((long long)grid * kStepR > N) grid = (N + kStepR - 1) / kStepR;
    if (grid < 1) return false;
    p->grid = grid;
    p->rows_base = N / grid;
    p->rows_extra = N % grid;
    const int n_max = p->rows_base + (p->rows_extra > 0 ? 1 : 0);
    if (n_max > kStepWindowRows) return false;
    p->S = (n_max + kStepR - 1) / kStepR;
    if (p->S > kStepMaxStages) return false;
    p->w_rows = n_max;
    const size_t w_bytes = (size_t)p->w_rows * nvec * 16;
    const size_t s_bytes = (size_t)p->S * kStepR * ngroups * 2;
    const size_t red = (size_t)(2 * nvec / 32) * kStepWindowRows * 4;
    const size_t normed = (size_t)N * 2;
    p->smem = w_bytes + s_bytes + red + normed;
    return p->smem <= budget;
}

// The add-RMSNorm row kernel's block for one row of `hidden`: the smallest vpt of 1, 2, 4
// that keeps the block at <= 256 threads (threads rounded up to whole warps).
inline bool step_rms_shape(int hidden, int *vpt, int *threads) {
    const int nvec = hidden / 8;
    for (int v = 1; v <= kStepRmsMaxVpt; v *= 2) {
        int t = (nvec + v - 1) / v;
        t = (t + 31) / 32 * 32;
        if (t <= 256) {
            *vpt = v;
            *threads = t;
            return true;
        }
    }
    return false;
}

}  // namespace fd
