// decode_layer.cu -- planning and dispatch of the one-launch decode layer
// (kernel and method: decode_layer.cuh).
#include "decode_layer.cuh"

namespace moe {

// ---------------------------------------------------------------- host side
#ifndef PAIR_SEGMENTS_MAX_T
#define PAIR_SEGMENTS_MAX_T 4
#endif
constexpr int kPairSegmentsMaxT = PAIR_SEGMENTS_MAX_T;  // on the Qwen4Exp geometry

namespace {

// Lanes per gate/up row pair and per down row: about five groups per lane,
// task buffers of a few kilobytes.
int layer_l1(int G1) { return G1 >= 40 ? 16 : (G1 >= 10 ? 4 : 1); }
int layer_l2(int G2) { return G2 >= 10 ? 4 : 1; }

LayerPlan layer_plan(int T, int E, int k, int H, int I, int num_sms, size_t smem_limit) {
    LayerPlan pl{};
    const int P = T * k;
    if (T < 1 || T > kLayerMaxT || P > kLayerMaxPairs || E > 32 * kLayerRoutePer || num_sms < 1) return pl;
    const int G1 = H / 32, G2 = I / 32;
    pl.L1 = layer_l1(G1);
    pl.L2 = layer_l2(G2);
    const int RT1 = 32 / pl.L1, RT2 = 2 * (32 / pl.L2);
    const uint32_t b1 = warp_geom(RT1, 2, H).bytes, b2 = warp_geom(RT2, 1, I).bytes;
    pl.slot_bytes = b1 > b2 ? b1 : b2;
    // the router keeps E keys in a routing warp's ring before any copy
    if ((size_t)kLayerSlots * pl.slot_bytes < (size_t)E * 4) pl.slot_bytes = (uint32_t)align_up((size_t)E * 4 / kLayerSlots, 128);
    // h rows one CTA's down share can read.  Shares are contiguous runs of
    // tasks of equal weight, a task of expert a weighing (1 + rows of a), so
    // the experts wholly inside a share hold at most (A + P)/NC + 1 <=
    // 2P/NC + 1 rows; the two experts cut by its ends add at most T rows each.
    const long long hr = (2LL * P + num_sms - 1) / num_sms + 1 + 2LL * T;
    pl.hrows = (int)(hr < P ? hr : P);
    for (int nw = kLayerMaxWarps; nw >= kLayerMinWarps; --nw) {
        if (nw <= T) break;  // warps beyond the T routing warps stage x
        const size_t smem = layer_layout(T, H, I, P, pl.hrows, nw, pl.slot_bytes).total;
        if (smem <= smem_limit) {
            pl.nw = nw;
            pl.smem = smem;
            pl.ok = true;
            break;
        }
    }
    return pl;
}

}  // namespace

// One-row segment per pair (see decode_layer_kernel): with one token it is
// the grouping itself; above, it streams an expert once per token that chose
// it, traded against starting every copy as soon as its pair is ranked.
// Measured on GB300 (one-call layer, mean us, grouped / pair segments):
//   Qwen4Exp (2560, 640, 512, 10): T=1 27.3 / 25.1, T=2 34.9 / 35.0,
//       T=4 52.3 / 49.3, T=8 82.0 / 106.5
//   TP4 shard (2560, 160, 512, 10, hot experts): T=2 25.0 / 22.3,
//       T=4 32.1 / 26.0, T=8 41.6 / 41.0
// Compiled for H = 2560 with I = 640 or 160 (the instantiations with a
// compile-time group count); other shapes take the grouped path.
int pair_segments(int T, int E, int k, int H, int I) {
    (void)E; (void)k;
    if (H != 2560) return 0;
    if (I == 640) return T <= kPairSegmentsMaxT ? 1 : 0;
    if (I == 160) return T <= 8 ? 1 : 0;
    return 0;
}

bool layer_fusable(int T, int E, int k, int H, int I, int num_sms, size_t smem_limit) {
    return layer_plan(T, E, k, H, I, num_sms, smem_limit).ok;
}

// An empty kernel launched exactly as the layer kernel is for the same
// shape (one CTA per SM, the plan's warps and dynamic shared memory, a
// cooperative launch): the cost of the launch alone, the floor under the
// layer's time.
__global__ void __launch_bounds__(kLayerMaxWarps * 32, 1) layer_floor_kernel() {}

cudaError_t launch_layer_floor(int T, int E, int k, int H, int I, int num_sms, size_t smem_limit,
                               cudaStream_t stream) {
    const LayerPlan pl = layer_plan(T, E, k, H, I, num_sms, smem_limit);
    if (!pl.ok) return cudaErrorInvalidConfiguration;
    static int configured[128];
    cudaError_t e = ensure_smem(layer_floor_kernel, configured, pl.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(pl.nw * 32);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, layer_floor_kernel);
}

template <int FMT>
static cudaError_t launch_decode_layer_f(const float *logits, const __half *x, const uint32_t *q13,
                                         const __half *s13, const uint32_t *z13, const uint32_t *q2,
                                         const __half *s2, const uint32_t *z2, int T, int E, int k, int H, int I,
                                         int32_t *topk_ids, float *topk_w, __half *out, __half *h, float *y,
                                         uint32_t *blkctr, uint32_t *done, uint32_t *exitctr, uint32_t *err,
                                         int num_sms, size_t smem_limit, cudaStream_t stream) {
    const LayerPlan pl = layer_plan(T, E, k, H, I, num_sms, smem_limit);
    if (!pl.ok) return cudaErrorInvalidConfiguration;
    LayerArgs a{};
    a.logits = logits; a.x = x;
    a.q13 = q13; a.s13 = s13; a.z13 = z13; a.q2 = q2; a.s2 = s2; a.z2 = z2;
    a.T = T; a.E = E; a.k = k; a.H = H; a.I = I; a.P = T * k;
    a.topk_ids = topk_ids; a.topk_w = topk_w; a.out = out;
    a.h = h; a.y = y; a.blkctr = blkctr; a.done = done; a.exitctr = exitctr; a.err = err;
    a.nw = pl.nw; a.hrows = pl.hrows; a.slot_bytes = pl.slot_bytes;
    a.pair_mode = pair_segments(T, E, k, H, I);
    const int G1 = H / 32, G2 = I / 32;
    // the geometries the layer is specified on get compile-time group counts
    if (G1 == 80 && pl.L1 == 16 && G2 == 20 && pl.L2 == 4)
        return launch_layer_t<16, 80, 4, 20, FMT>(a, pl, num_sms, stream);
    if (G1 == 80 && pl.L1 == 16 && G2 == 5 && pl.L2 == 1)
        return launch_layer_t<16, 80, 1, 5, FMT>(a, pl, num_sms, stream);
    switch (pl.L1 * 8 + pl.L2) {
        case 16 * 8 + 4: return launch_layer_t<16, 0, 4, 0, FMT>(a, pl, num_sms, stream);
        case 16 * 8 + 1: return launch_layer_t<16, 0, 1, 0, FMT>(a, pl, num_sms, stream);
        case 4 * 8 + 4: return launch_layer_t<4, 0, 4, 0, FMT>(a, pl, num_sms, stream);
        case 4 * 8 + 1: return launch_layer_t<4, 0, 1, 0, FMT>(a, pl, num_sms, stream);
        case 1 * 8 + 4: return launch_layer_t<1, 0, 4, 0, FMT>(a, pl, num_sms, stream);
        default: return launch_layer_t<1, 0, 1, 0, FMT>(a, pl, num_sms, stream);
    }
}

cudaError_t launch_decode_layer(const float *logits, const __half *x, const uint32_t *q13, const __half *s13,
                                const uint32_t *z13, const uint32_t *q2, const __half *s2,
                                const uint32_t *z2, int T, int E, int k, int H, int I, int32_t *topk_ids,
                                float *topk_w, __half *out, __half *h, float *y, uint32_t *blkctr,
                                uint32_t *done, uint32_t *exitctr, uint32_t *err, int num_sms,
                                size_t smem_limit, cudaStream_t stream) {
    return launch_decode_layer_f<kFmtW4A16>(logits, x, q13, s13, z13, q2, s2, z2, T, E, k, H, I, topk_ids, topk_w,
                                            out, h, y, blkctr, done, exitctr, err, num_sms, smem_limit, stream);
}

// NVFP4 weights: s13 / s2 hold the E4M3 scale bytes, gs13 / gs2 the
// per-expert scales (decode_common.cuh).
cudaError_t launch_decode_layer_nvfp4(const float *logits, const __half *x, const uint32_t *q13,
                                      const uint8_t *s13, const float *gs13, const uint32_t *q2, const uint8_t *s2,
                                      const float *gs2, int T, int E, int k, int H, int I, int32_t *topk_ids,
                                      float *topk_w, __half *out, __half *h, float *y, uint32_t *blkctr,
                                      uint32_t *done, uint32_t *exitctr, uint32_t *err, int num_sms,
                                      size_t smem_limit, cudaStream_t stream) {
    return launch_decode_layer_f<kFmtNvfp4>(logits, x, q13, reinterpret_cast<const __half *>(s13),
                                            reinterpret_cast<const uint32_t *>(gs13), q2,
                                            reinterpret_cast<const __half *>(s2),
                                            reinterpret_cast<const uint32_t *>(gs2), T, E, k, H, I, topk_ids, topk_w,
                                            out, h, y, blkctr, done, exitctr, err, num_sms, smem_limit, stream);
}

}  // namespace moe
