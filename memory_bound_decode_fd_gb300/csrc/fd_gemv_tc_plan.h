// fd_gemv_tc_plan.h - launch planning of the tensor-core GEMV (fd_gemv_tc.cu): the k step,
// the rings and the shared-memory layout, as pure host functions (no CUDA calls, so they
// are testable without a GPU).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime.h>  // __host__ __device__

namespace fd {

constexpr int kTcRows = 128;    // weight rows per CTA (MMA M)
constexpr int kTcGuBoxK = 64;   // k per gate/up tensor-map box (128 bytes)
constexpr int kTcSplit = 4;     // CTAs per cluster (K quarters)
constexpr int kTcWTileK = 256;  // k per weight tile (128 bytes of a row)
constexpr uint32_t kWStageBytes = kTcRows * kTcWTileK / 2;  // int4 tile: 16384

// k per pipeline step: 128 for up to 64 activation rows (half the per-step handshakes per
// weight byte), 64 for 128 rows (whose larger operand stages would not fit twice).
__host__ __device__ constexpr int tc_step_k(int npad) { return npad <= 64 ? 128 : 64; }

// The activation rows of one launch padded to the MMA's N.
inline int tc_npad(int m) { return m <= 16 ? 16 : m <= 32 ? 32 : m <= 64 ? 64 : 128; }

struct TcPlan {
    int s_w, s_gu, s_op, sg;             // weight tiles, gate/up stages, operand stages; scale
                                         // columns copied per row
    uint32_t off_gu, off_op, off_sc, smem;  // offsets (weights at 0); dynamic smem per CTA
};

// Shared-memory plan: a ring of int4 weight tiles (the HBM stream; 4 tiles, fewer where the
// operand stages need the room), then as many gate/up and operand stages as fit (2..4 each;
// operand stages in pairs, the two halves the MMA thread commits), then the scales. Every
// region starts on a 1024-byte boundary (the 128-byte-swizzled tensor-map destinations).
inline bool make_plan(int npad, int stepk, int k_cta, int group, size_t budget, TcPlan *p) {
    if (npad < 16 || npad > 128 || (stepk != 64 && stepk != 128) || k_cta % stepk != 0 ||
        group <= 0)
        return false;
    const uint32_t gu_stage = 2u * (stepk / kTcGuBoxK) * npad * 128;
    const uint32_t op_stage = (uint32_t)kTcRows * stepk * 2 + (uint32_t)npad * stepk * 2;
    p->sg = ((k_cta + group - 1) / group + 7 + 7) & ~7;
    if (p->sg > 256) return false;
    const uint32_t sc_bytes = ((uint32_t)kTcRows * p->sg * 2 + 1023u) & ~1023u;
    size_t avail = 0;
    for (p->s_w = 4; p->s_w >= 2; --p->s_w) {
        const size_t fixed = 1024 + (size_t)p->s_w * kWStageBytes + sc_bytes;
        avail = budget > fixed ? budget - fixed : 0;
        if (2 * (size_t)gu_stage + 2 * (size_t)op_stage <= avail) break;
    }
    if (p->s_w < 2) return false;
    const uint32_t w_bytes = p->s_w * kWStageBytes;
    int s_gu = 2, s_op = 2;
    size_t used = 2 * (size_t)gu_stage + 2 * (size_t)op_stage;
    for (bool grew = true; grew;) {
        grew = false;
        if (s_op < 4 && used + 2 * (size_t)op_stage <= avail) { s_op += 2; used += 2 * (size_t)op_stage; grew = true; }
        if (s_gu < 4 && used + gu_stage <= avail) { ++s_gu; used += gu_stage; grew = true; }
    }
    p->s_gu = s_gu;
    p->s_op = s_op;
    p->off_gu = w_bytes;
    p->off_op = p->off_gu + s_gu * gu_stage;
    p->off_sc = p->off_op + s_op * op_stage;
    p->smem = p->off_sc + sc_bytes + 1024;  // + alignment slack of the dynamic base
    // the cluster reduction reuses the gate/up and operand rings
    return (size_t)kTcSplit * npad * 32 * 4 <= (size_t)p->off_sc - p->off_gu &&
           p->smem <= budget;
}

// The plan of one launch: 128-k steps where they fit (up to 64 activation rows), else 64-k
// steps (every batch at K = 32768 with group 64, where the 128-k stages and the scale
// window together exceed a CTA's shared memory). *stepk receives the step.
inline bool plan_tc(int npad, int k_cta, int group, size_t budget, int *stepk, TcPlan *p) {
    *stepk = tc_step_k(npad);
    if (make_plan(npad, *stepk, k_cta, group, budget, p)) return true;
    if (*stepk == 64) return false;
    *stepk = 64;
    return make_plan(npad, 64, k_cta, group, budget, p);
}

}  // namespace fd
