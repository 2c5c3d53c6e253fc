// fd_gemv_plan.cu - launch planning of the bulk-copy GEMV kernel (see fd_gemv_plan.h).
#include "fd_gemv_plan.h"

#include <algorithm>

#include "fd_gemv_common.cuh"  // kWindowRows

namespace fd {
namespace {

struct Shape {
    size_t w_row, s_row, red;
    int R, act_rows;
    size_t bytes(int wr, int st) const { return (size_t)wr * w_row + (size_t)st * R * s_row + red; }
};

// The plan for `per_sm` resident CTAs per SM, each within `cap` bytes of dynamic shared
// memory; false if the ring would be too small.
bool plan_for(const TmaPlanInput &in, const Shape &sh, int per_sm, size_t cap, TmaPlan &p) {
    const int R = in.R;
    int grid = in.sm_count * per_sm;
    if ((long long)grid * R > in.N) grid = (in.N + R - 1) / R;
    if (grid < 1) grid = 1;
    p.grid = grid;
    p.rows_base = in.N / grid;
    p.rows_extra = in.N % grid;
    p.per_sm = per_sm;
    const int n_max = p.rows_base + (p.rows_extra > 0 ? 1 : 0);
    const int n_chunks_max = (n_max + R - 1) / R;
    p.S = 0;
    p.w_rows = 0;
    if (in.M <= in.MB) {
        // One pass over the rows: when the CTA's share fits, every chunk gets a stage of
        // its own and all are issued at once. The activation (M == 1) takes the stages
        // after the chunks if there is room, else it overlays the last weight rows and the
        // chunks there are issued once the consumers have read it.
        const int own = n_chunks_max + (in.M == 1 ? (sh.act_rows + R - 1) / R : 0);
        if (own <= in.max_stages && sh.bytes(own * R, own) <= cap) {
            p.S = own;
            p.w_rows = own * R;
        } else if (in.M == 1 && n_chunks_max <= in.max_stages && n_max >= sh.act_rows &&
                   sh.bytes(n_max, n_chunks_max) <= cap) {
            p.S = n_chunks_max;
            p.w_rows = n_max;
        }
    }
    p.ring = (p.S == 0);
    if (p.ring) {
        // a ring of uniform stages, reused across chunks and activation-row passes
        const size_t stage = (size_t)R * (sh.w_row + sh.s_row);
        if (sh.red + 2 * stage > cap) return false;
        p.S = (int)std::min<size_t>((cap - sh.red) / stage, (size_t)in.max_stages);
        p.w_rows = p.S * R;
    }
    // With M == 1 the activation copy borrows the last act_rows weight rows: stages from
    // act_first_stage on are filled after it is read. A ring keeps two stages for weights
    // (three when CTAs share an SM).
    p.act_first_stage = (in.M == 1) ? (p.w_rows - sh.act_rows) / R : p.S;
    const int min_free = per_sm > 1 ? 3 : 2;
    if (p.ring && (in.M == 1 ? p.act_first_stage : p.S) < min_free) return false;
    p.smem = sh.bytes(p.w_rows, p.S);
    return true;
}

}  // namespace

bool plan_gemv_tma(const TmaPlanInput &in, TmaPlan *p) {
    const int nvec = in.K / 32;
    const int ngroups = in.K / in.group;
    Shape sh;
    sh.w_row = (size_t)in.K / 2;
    sh.s_row = (size_t)ngroups * 2;
    sh.red = (size_t)(in.LPS * nvec / 32) * kWindowRows * in.MB * 4;
    sh.R = in.R;
    sh.act_rows = in.plain ? 4 : 8;  // x: 2K bytes = 4 rows of K/2; gate + up: 4K bytes = 8
    const size_t budget = (size_t)in.smem_optin - (size_t)in.static_smem;
    // Persistent CTAs: one per SM, or several when a CTA is small (few consumer warps at
    // small K) and the registers (per warp, in units of 256), threads and shared memory
    // allow. More warps per scheduler hide the row loop's latency: at K=4096 three CTAs of
    // 288 threads share an SM.
    const int threads = in.LPS * nvec + 32;
    const int warps = (threads + 31) / 32;
    const int regs_per_warp = ((in.regs * 32 + 255) / 256) * 256;
    int max_per_sm = regs_per_warp > 0 ? 65536 / (regs_per_warp * warps) : 1;
    max_per_sm = std::min(max_per_sm, 2048 / (warps * 32));
    max_per_sm = std::min(max_per_sm, 4);
    for (int c = max_per_sm; c > 1; --c) {
        const long long share = (long long)in.smem_per_sm / c - in.smem_reserved - in.static_smem;
        if (share > 0 && plan_for(in, sh, c, std::min((size_t)share, budget), *p)) return true;
    }
    return plan_for(in, sh, 1, budget, *p);
}

}  // namespace fd
