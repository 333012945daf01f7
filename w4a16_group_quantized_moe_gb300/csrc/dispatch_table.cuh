// dispatch_table.cuh -- the per-shape choice of kernels for the step calls,
// from measurement.
//
// For a weight geometry (H, I, E, k) and a range of batch sizes T, the
// kernel family that ran the step calls (route + align, gate/up, down)
// fastest on a GB300, with every step's weights read from HBM (the weight
// stack rotated over copies larger than L2).  Shapes not listed fall back to
// the shape rule of resolve_path.
#pragma once
#include "../../include/moe_w4a16.h"

namespace moe {

struct PathRange {
    int H, I, E, k;  // weight geometry
    int t_lo, t_hi;  // batch sizes (inclusive)
    int path;        // MOE_PATH_*
};

// Step calls, mean us per layer (route, align, gate/up, down), decode kernels
// against tensor cores; the stream kernels were slower at every T measured
// (1-512), by 1.6x to 40x:
//   Qwen4Exp (2560, 640, 512, 10):  T=9 123 / 216, 12 159 / 225, 16 219 / 272,
//       17 234 / 276, 20 274 / 315, 24 343 / 359, 26 406 / 372, 28 443 / 400
//   TP4 shard (2560, 160, 512, 10): T=9 75 / 100, 12 93 / 107, 16 109 / 134,
//       17 117 / 138, 20 126 / 144, 22 142 / 144, 24 149 / 148, 26 164 / 150
constexpr PathRange kPathTable[] = {
    {2560, 640, 512, 10, 1, 24, MOE_PATH_DECODE},
    {2560, 640, 512, 10, 25, 1 << 24, MOE_PATH_TENSOR_CORE},
    {2560, 160, 512, 10, 1, 22, MOE_PATH_DECODE},
    {2560, 160, 512, 10, 23, 1 << 24, MOE_PATH_TENSOR_CORE},
};

inline int tuned_path(int T, int E, int k, int H, int I) {
    for (const PathRange &r : kPathTable)
        if (r.H == H && r.I == I && r.E == E && r.k == k && T >= r.t_lo && T <= r.t_hi) return r.path;
    return MOE_PATH_AUTO;
}

}  // namespace moe
