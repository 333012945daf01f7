/*
 * moe_w4a16.h -- C ABI of libmoe_w4a16: the routed-expert MoE layer with
 * W4A16 group-32 expert weights, as hand-written CUDA kernels for GB300
 * (sm_103a).
 *
 * The layer (geometry from "[Model][SM70] Adapt Qwen3.8 Flash Next NVFP4",
 * section Implemented route: hidden 2560, expert intermediate 640, 512
 * experts, top-10; grouping and quantisation from "[Perf][SM70] Narrow
 * Qwen3.8 AWQ active grouped decode", section Purpose: AWQ W4A16 "effective
 * g32", "multi-row active-expert segments and offsets-based scheduling") is
 * four calls, issued in this order on one stream:
 *
 *   moe_topk_route          logits -> top-k expert ids and renormalised weights
 *   moe_align_offsets       ids -> per-expert segments of token-expert pairs
 *   moe_w4a16_gate_up_silu  x, W13 -> h = silu(x Wg^T) * (x Wu^T), per pair
 *   moe_w4a16_down_combine  h, W2, weights -> out = sum_j w_j * (h_j W2^T)
 *
 * Conventions for every call below.
 *   - Pointers are CUDA device pointers unless marked (host).  Every device
 *     pointer must be 16-byte aligned (PyTorch and cudaMalloc allocations
 *     are); a misaligned pointer is rejected with MOE_ERR_INVALID_ARG.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous: they validate arguments on the host,
 *     enqueue kernels and return.  They never synchronise, never allocate
 *     device or pinned memory, and never abort or trap.
 *   - The caller owns every buffer.  The library keeps no state between
 *     calls except cached device attributes (SM count, shared-memory limit).
 *   - fp16 buffers hold IEEE binary16 values (passed as uint16_t*).
 *   - T = tokens, E = experts, k = experts per token, H = hidden size,
 *     I = expert intermediate size, P = T*k token-expert pairs.  A pair is
 *     p = t*k + j: token t's j-th selected expert.
 *   - Supported sizes: 0 <= T, T*k <= 2^24, 1 <= k <= min(E, 32), E <= 1024,
 *     H and I positive multiples of 32 up to 65536, group_size == 32.  Anything else is
 *     MOE_ERR_INVALID_ARG (malformed) or MOE_ERR_UNSUPPORTED (outside the
 *     sizes above).  T == 0 is a no-op that returns MOE_OK.
 *
 * Packed weight layout (AWQ-style W4A16, groups of 32 along the reduction
 * dimension K; row-major, little-endian 32-bit words).  For one expert's
 * matrix W[N][K]:
 *   qweight u32 [N][K/8]   : code of (n, kk) = bits 4*(kk%8)..+3 of word [n][kk/8]
 *   scales  f16 [N][K/32]  : s of (n, kk) = scales[n][kk/32]
 *   qzeros  u32 [N/8][K/32]: zero of (n, kk) = bits 4*(n%8)..+3 of word [n/8][kk/32]
 *   w(n, kk) = (code - zero) * s
 * Experts are stacked on the outermost axis: W13 = [E][2I][H] (rows [0,I)
 * gate, [I,2I) up), W2 = [E][H][I].
 *
 * Workspace.  gate_up and down_combine need a caller-owned device workspace
 * of at least moe_workspace_bytes(T, E, k, H, I) bytes.  It must be zero-
 * filled before its first use (e.g. cudaMemsetAsync or torch.zeros) and is
 * left zeroed in its control words after every call that completed without
 * a device error, so it can be reused as is.  Calls that share a workspace
 * must be ordered on one stream.  It also carries the device error word read
 * by moe_get_device_error.  After a device error is reported, zero the
 * workspace again before reusing it.
 *
 * Diagnostic words of the workspace's control block (its first 256 bytes).
 * A zero-filled workspace selects the defaults; a caller may write them
 * (e.g. with cudaMemcpy) between calls to test or observe the kernels:
 *   u32 word MOE_CTRL_WAIT_POLLS  polls before an in-kernel wait on other
 *                                 CTAs gives up (0: about one second)
 *   u32 word MOE_CTRL_WAIT_EXTRA  added to the target of every such wait;
 *                                 nonzero makes them unsatisfiable, so they
 *                                 run out and report MOE_DEVERR_WAIT_TIMEOUT
 *   u64 at word MOE_CTRL_TIMELINE device address of a buffer of 8 u64 per
 *                                 CTA that the one-call decode layer fills
 *                                 with global-timer stamps of its phases
 *                                 (0: off)
 */
#define MOE_CTRL_WAIT_POLLS 1
#define MOE_CTRL_WAIT_EXTRA 2
#define MOE_CTRL_TIMELINE 4
#ifndef MOE_W4A16_H
#define MOE_W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, k > E, ... */
    MOE_ERR_UNSUPPORTED = 2,  /* well-formed but outside the supported sizes  */
    MOE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required   */
    MOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed         */
    MOE_ERR_DEVICE_FLAG = 5   /* a kernel flagged bad data (see below)        */
} moe_status_t;

/* Bits of the device error word (moe_get_device_error). */
#define MOE_DEVERR_BAD_EXPERT_ID 0x1u  /* topk_ids entry outside [0, E): pair skipped */
#define MOE_DEVERR_WAIT_TIMEOUT  0x2u  /* an in-kernel wait gave up; outputs invalid  */
#define MOE_DEVERR_BAD_METADATA  0x4u  /* offsets / sorted_pair / active list invalid */

/* Version of this ABI (incremented on incompatible change). */
int moe_abi_version(void);

/* Static English text for a status code (host; never NULL). */
const char *moe_status_string(int status);

/* Bytes of workspace gate_up and down_combine need for this shape (host,
 * pure).  Returns 0 for sizes the library rejects. */
size_t moe_workspace_bytes(int T, int E, int k, int H, int I);

/* Diagnostic: waits for `stream` to finish, copies the device error word of
 * `workspace` into *flag_out (host), clears it on the device, and returns
 * MOE_ERR_DEVICE_FLAG if it was nonzero, MOE_OK otherwise.  This is the only
 * call that synchronises; it is meant for tests and debugging. */
int moe_get_device_error(void *workspace, size_t ws_bytes, uint32_t *flag_out,
                         void *stream);

/* Which kernels the step calls (moe_w4a16_gate_up_silu and
 * moe_w4a16_down_combine) run for a shape on the current device, chosen from
 * the shape alone (host; queries the device's SM count and shared-memory
 * limit on first use): the per-shape table of measured choices where it
 * lists the shape, else a rule on the shape.  Returns MOE_PATH_NONE for
 * sizes the library rejects, for T == 0 and when no device is usable. */
#define MOE_PATH_NONE 0
#define MOE_PATH_DECODE 1       /* latency-first weight-streaming decode kernels */
#define MOE_PATH_TENSOR_CORE 2  /* tcgen05 grouped contractions */
#define MOE_PATH_STREAM 3       /* staged CUDA-core streaming kernels */
#define MOE_PATH_AUTO 0         /* as an argument: the library's choice */
int moe_step_kernel_path(int T, int E, int k, int H, int I);

/* Step 1, router.  For each token t: softmax over logits[t][0..E), the k
 * most probable experts (ties: lower expert index first), and their
 * probabilities renormalised to sum to one -- equivalently softmax over the
 * k selected logits.  Selection compares the fp32 logits themselves (softmax
 * is monotone); -0.0 ranks equal to +0.0; NaN ranks below every number.
 *   logits   f32 [T][E]   (read)
 *   topk_ids i32 [T][k]   (written) in rank order
 *   topk_w   f32 [T][k]   (written)
 * No workspace. */
int moe_topk_route(const float *logits, int T, int E, int k,
                   int32_t *topk_ids, float *topk_w, void *stream);

/* Step 2, active-expert segments.  Groups the P pairs by expert: a stable
 * counting sort of pair ids by expert id.
 *   topk_ids       i32 [T][k]  (read) expert of each pair
 *   expert_offsets i32 [E+1]   (written) segment of expert e is rows
 *                              [offsets[e], offsets[e+1]); offsets[E] = pairs kept
 *   sorted_pair    i32 [P]     (written) pair ids, segment after segment,
 *                              ascending within a segment
 *   active_experts i32 [E]     (written) experts with a non-empty segment in
 *                              ascending order, then -1 up to E
 *   num_active     i32 [1]     (written) number of active experts A
 * An id outside [0, E) is skipped (its pair is in no segment, trailing
 * sorted_pair entries are -1) and sets MOE_DEVERR_BAD_EXPERT_ID in the
 * workspace error word.  workspace may be NULL (then bad ids are skipped
 * silently); if given it must hold at least 256 bytes.  With T == 0,
 * topk_ids and sorted_pair may be NULL. */
int moe_align_offsets(const int32_t *topk_ids, int T, int E, int k,
                      int32_t *expert_offsets, int32_t *sorted_pair,
                      int32_t *active_experts, int32_t *num_active,
                      void *workspace, size_t ws_bytes, void *stream);

/* Steps 1 and 2 together: exactly the outputs of moe_topk_route followed by
 * moe_align_offsets on the same arguments (same layouts, error bits and
 * workspace rules).  For T <= 32 both steps run in one launch (one CTA),
 * which removes a kernel launch and a global-memory round trip from the
 * decode critical path; larger batches run the two kernels.  Reference: the
 * grouped-decode route of "[Perf][SM70] Narrow Qwen3.8 AWQ active grouped
 * decode" (section Purpose) prepares routing and segments for 2-8 tokens. */
int moe_topk_route_align(const float *logits, int T, int E, int k,
                         int32_t *topk_ids, float *topk_w,
                         int32_t *expert_offsets, int32_t *sorted_pair,
                         int32_t *active_experts, int32_t *num_active,
                         void *workspace, size_t ws_bytes, void *stream);

/* Step 3, gate/up projection with the int4 dequantisation fused in, and
 * SiLU(gate) * up.  For every sorted row r of every active expert's segment
 * (pair p = sorted_pair[r], token t = p / k):
 *   g_i = sum_K x[t][K] * W13[e][i][K],  u_i = sum_K x[t][K] * W13[e][I+i][K]
 *   h[r][i] = silu(g_i) * u_i,  silu(v) = v / (1 + exp(-v)),  i in [0, I)
 *   x     f16 [T][H]                         (read)
 *   w13_q u32 [E][2I][H/8], w13_s f16 [E][2I][H/32], w13_z u32 [E][2I/8][H/32]
 *   expert_offsets, sorted_pair, active_experts, num_active: step 2 outputs
 *   h     f16 [P][I]  (written) in sorted-row order; rows not in any segment
 *                      are left untouched
 * Arithmetic: codes minus zero times activation in fp16 within each group of
 * 32 (exact integer differences, one rounding per product and sum), group
 * sums scaled and accumulated in fp32, SiLU in fp32, h rounded to fp16.
 * `h` must not alias any input. */
int moe_w4a16_gate_up_silu(const uint16_t *x,
                           const uint32_t *w13_q, const uint16_t *w13_s,
                           const uint32_t *w13_z, int group_size,
                           const int32_t *expert_offsets, const int32_t *sorted_pair,
                           const int32_t *active_experts, const int32_t *num_active,
                           int T, int E, int k, int H, int I,
                           uint16_t *h, void *workspace, size_t ws_bytes,
                           void *stream);

/* Step 4, down projection with the dequantisation fused in, and the
 * weighted combine.  For every sorted row r (pair p = t*k + j):
 *   y_p[n] = sum_i h[r][i] * W2[e][n][i],  n in [0, H)
 *   out[t][n] = sum_{j<k} topk_w[t][j] * y_{t*k+j}[n]   (j in order, fp32)
 *   h      f16 [P][I]   (read) step 3 output
 *   w2_q u32 [E][H][I/8], w2_s f16 [E][H][I/32], w2_z u32 [E][H/8][I/32]
 *   topk_w f32 [T][k]   (read) step 1 weights
 *   out    f16 [T][H]   (written) rounded from fp32
 * The per-pair y lives in the workspace in fp32; the combine sums a token's
 * k terms in a fixed order, so results are deterministic.  `out` may alias
 * x of step 3 but not h or topk_w. */
int moe_w4a16_down_combine(const uint16_t *h,
                           const uint32_t *w2_q, const uint16_t *w2_s,
                           const uint32_t *w2_z, int group_size,
                           const int32_t *expert_offsets, const int32_t *sorted_pair,
                           const int32_t *active_experts, const int32_t *num_active,
                           const float *topk_w, int T, int E, int k, int H, int I,
                           uint16_t *out, void *workspace, size_t ws_bytes,
                           void *stream);

/* The whole layer in one call: steps 1-4 above, in order, with the same
 * arithmetic and results (routing ids and weights bit-identical to
 * moe_topk_route; h and out as steps 3 and 4).  The method is the layer of
 * the overview (route with renormalised top-k softmax, group the pairs into
 * active-expert segments, gate/up + SiLU, down, weighted combine); the
 * single entry point is this library's own.
 *   logits f32 [T][E], x f16 [T][H]   (read)
 *   w13_*, w2_*                        packed weights as in steps 3 and 4
 *   topk_ids i32 [T][k], topk_w f32 [T][k]  (written) step 1 outputs
 *   out    f16 [T][H]                  (written)
 *   workspace: at least moe_layer_workspace_bytes(T, E, k, H, I) bytes, with
 *   the rules of the workspace paragraph above; it holds the grouping, h
 *   and the per-pair projections.
 * For decode batches (T <= 8, T*k <= 256) whose buffers fit one SM's shared
 * memory, the layer runs as one cooperative kernel (one CTA per SM, all
 * resident): every CTA routes and groups the tokens itself, and the CTAs
 * wait on each other only where a step needs another CTA's results (h of
 * an expert before its down rows, all of a block's rows before its
 * combine), with bounded waits that report MOE_DEVERR_WAIT_TIMEOUT.  Other
 * sizes run the four steps as separate launches.  `out` must not alias any
 * input. */
size_t moe_layer_workspace_bytes(int T, int E, int k, int H, int I);

/* Diagnostic, the launch-cost floor of the call above: launches an empty
 * kernel exactly as moe_w4a16_moe_layer launches its one cooperative
 * kernel for this shape (grid = one CTA per SM, the same block size and
 * dynamic shared memory, cooperative), on `stream`, and computes nothing.
 * The layer's time minus this one is what its kernel costs beyond
 * launching.  MOE_ERR_UNSUPPORTED where the shape does not take the
 * one-launch path; MOE_OK for T == 0 (nothing launched); MOE_ERR_CUDA on a
 * launch error.  Takes no buffers. */
int moe_decode_layer_floor(int T, int E, int k, int H, int I, void *stream);

int moe_w4a16_moe_layer(const float *logits, const uint16_t *x,
                        const uint32_t *w13_q, const uint16_t *w13_s, const uint32_t *w13_z,
                        const uint32_t *w2_q, const uint16_t *w2_s, const uint32_t *w2_z,
                        int group_size, int T, int E, int k, int H, int I,
                        int32_t *topk_ids, float *topk_w, uint16_t *out,
                        void *workspace, size_t ws_bytes, void *stream);

/* ---- Second weight format: NVFP4 weights with fp16 activations.
 * "[Model][SM70] Adapt Qwen3.8 Flash Next NVFP4", section Implemented route,
 * runs the checkpoint's ModelOpt NVFP4 routed experts through the W4A16
 * kernel with fp16 activations (the "A16" route).  The format, as publicly
 * defined, for one expert's matrix W[N][K]:
 *   codes  u32 [N][K/8]  : E2M1 value of (n, kk) = nibble 4*(kk%8) of word [n][kk/8]
 *                          (bit 3 sign, bits 2-1 exponent with bias 1, bit 0 mantissa)
 *   bscale u8  [N][K/16] : FP8 E4M3 scale of (n, kk) = bscale[n][kk/16]
 *   gscale f32 per expert: scale of the whole matrix
 *   w(n, kk) = e2m1(code) * e4m3(bscale) * gscale[e]
 * Experts are stacked as for W4A16 (codes [E][N][K/8], bscale [E][N][K/16],
 * gscale [E]).  The three calls below take the place of steps 3, 4 and the
 * one-call layer; routing, grouping, workspace sizes and rules, error codes
 * and results are as for the W4A16 calls.  Arithmetic: e2m1 values times
 * activations in fp16 within each 16-element block, scaled by the block's
 * E4M3 scale and the expert's scale in fp32 (decode kernels), or the MMA
 * operand e2m1 * e4m3 in fp16 (exact) with fp32 accumulation and the
 * expert's scale applied to the accumulator (tensor-core kernels): the
 * decode kernels up to 16 tokens where their layout fits, else the tensor
 * cores (there are no stream kernels for this format).  A shape neither
 * takes returns MOE_ERR_UNSUPPORTED before any launch.
 * Scale products |e4m3 * gscale| and activations must keep each block's fp16
 * partial sum finite. */
int moe_nvfp4_gate_up_silu(const uint16_t *x, const uint32_t *w13_codes, const uint8_t *w13_bscale,
                           const float *w13_gscale, const int32_t *expert_offsets,
                           const int32_t *sorted_pair, const int32_t *active_experts,
                           const int32_t *num_active, int T, int E, int k, int H, int I, uint16_t *h,
                           void *workspace, size_t ws_bytes, void *stream);

int moe_nvfp4_down_combine(const uint16_t *h, const uint32_t *w2_codes, const uint8_t *w2_bscale,
                           const float *w2_gscale, const int32_t *expert_offsets,
                           const int32_t *sorted_pair, const int32_t *active_experts,
                           const int32_t *num_active, const float *topk_w, int T, int E, int k, int H,
                           int I, uint16_t *out, void *workspace, size_t ws_bytes, void *stream);

/* The whole layer with NVFP4 weights (workspace: moe_layer_workspace_bytes). */
int moe_nvfp4_moe_layer(const float *logits, const uint16_t *x, const uint32_t *w13_codes,
                        const uint8_t *w13_bscale, const float *w13_gscale, const uint32_t *w2_codes,
                        const uint8_t *w2_bscale, const float *w2_gscale, int T, int E, int k, int H,
                        int I, int32_t *topk_ids, float *topk_w, uint16_t *out, void *workspace,
                        size_t ws_bytes, void *stream);

/* ---- The steps on either side of the layer.
 *
 * Router logits, the step ahead of moe_topk_route.  The grouped-decode work
 * takes the router's fp32 logits as given ("[Perf][SM70] Narrow Qwen3.8 AWQ
 * active grouped decode", section Purpose: 512 experts, top-k 10, hidden
 * 2560); the model's gate is a bias-free linear map from the hidden state
 * to one score per expert:
 *     logits[t][e] = sum over h of x[t][h] * w_router[e][h]
 *   x        f16 [T][H]   hidden states (the layer's x)
 *   w_router f16 [E][H]   one row per expert (a linear layer's weight)
 *   logits   f32 [T][E]   out
 * Products of fp16 values are exact in fp32 and are summed in fp32 (order
 * unspecified).  T <= 16: a weight-streaming GEMV; larger T: tcgen05 tensor
 * cores.  Sizes as for moe_topk_route with k = 1 (H a multiple of 32).
 * `workspace` is optional (NULL, or at least 256 bytes, zero-filled): it
 * receives MOE_DEVERR_WAIT_TIMEOUT if a tensor-core wait gives up. */
int moe_router_logits(const uint16_t *x, const uint16_t *w_router, int T, int E, int H, float *logits,
                      void *workspace, size_t ws_bytes, void *stream);

/* Router logits, steps 1 and 2 in one call: the outputs of
 * moe_router_logits followed by moe_topk_route_align on those logits (so
 * the routing is exactly that of moe_topk_route applied to `logits`).  For
 * T <= 16 one launch: the last CTA of the GEMV to finish (an atomic ticket
 * in the workspace's control block; no CTA waits for another) routes and
 * groups.  `workspace` is required: at least 256 bytes, zero-filled before
 * first use, left reusable after every call that completed without a
 * device error; calls sharing it must be ordered on one stream. */
int moe_router_route_align(const uint16_t *x, const uint16_t *w_router, int T, int E, int k, int H,
                           float *logits, int32_t *topk_ids, float *topk_w, int32_t *expert_offsets,
                           int32_t *sorted_pair, int32_t *active_experts, int32_t *num_active,
                           void *workspace, size_t ws_bytes, void *stream);

/* AWQ checkpoint import.  "[Model][SM70] Support Qwen3.8 Flash Next with
 * PLE offload", section Purpose, names the AWQ g32 metadata adapter that
 * feeds the grouped decode; the checkpoint layout is the public AWQ "GEMM"
 * packing of a linear layer with input size K and output size N (experts
 * stacked on a leading E axis):
 *   awq_qweight u32 [E][K][N/8]    nibble i of word [kk][c] = code of column 8c + ORDER[i]
 *   awq_qzeros  u32 [E][K/32][N/8] nibble i of word [g][c]  = zero of column 8c + ORDER[i]
 *   awq_scales  f16 [E][K/32][N]
 *   ORDER = (0, 2, 4, 6, 1, 3, 5, 7); w = (code - zero) * scale.
 * Writes the same (code, zero, scale) of every element into rows
 * [row0, row0 + N) of a matrix stack in this library's layout with N_dst
 * rows per expert: qweight [E][N_dst][K/8], scales [E][N_dst][K/32],
 * qzeros [E][N_dst/8][K/32] (e.g. a gate layer at row0 = 0 and the up
 * layer at row0 = I of W13; a down layer at row0 = 0 of W2).  Only the
 * destination rows named are written (their zero words whole: row0 and N
 * are multiples of 8).  Requires K % 32 == 0, N % 8 == 0, N_dst % 8 == 0,
 * row0 % 8 == 0, row0 + N <= N_dst, group_size == 32; E <= 1024, K <= 65536.
 * Source and destination must not overlap.  Bit-exact (a permutation of
 * bits); asynchronous on `stream`, no workspace. */
int moe_awq_import(const uint32_t *awq_qweight, const uint32_t *awq_qzeros, const uint16_t *awq_scales,
                   int E, int K, int N, int group_size, uint32_t *qweight, uint16_t *scales,
                   uint32_t *qzeros, int N_dst, int row0, void *stream);

/* Steps 3 and 4 with the kernel family named: `path` is MOE_PATH_AUTO (the
 * choice of moe_step_kernel_path, as the calls without _ex make), or
 * MOE_PATH_DECODE, MOE_PATH_TENSOR_CORE or MOE_PATH_STREAM to force one.
 * Every family computes the same step (results within the layer's
 * tolerance of each other; h is in sorted-row order on every path), so the
 * two steps of a layer may run on different paths.  A forced path that
 * cannot take the shape returns MOE_ERR_UNSUPPORTED before any launch; any
 * other value is MOE_ERR_INVALID_ARG.  Other arguments and rules as for the
 * calls without _ex. */
int moe_w4a16_gate_up_silu_ex(const uint16_t *x, const uint32_t *w13_q, const uint16_t *w13_s,
                              const uint32_t *w13_z, int group_size, const int32_t *expert_offsets,
                              const int32_t *sorted_pair, const int32_t *active_experts,
                              const int32_t *num_active, int T, int E, int k, int H, int I, uint16_t *h,
                              void *workspace, size_t ws_bytes, int path, void *stream);

int moe_w4a16_down_combine_ex(const uint16_t *h, const uint32_t *w2_q, const uint16_t *w2_s,
                              const uint32_t *w2_z, int group_size, const int32_t *expert_offsets,
                              const int32_t *sorted_pair, const int32_t *active_experts,
                              const int32_t *num_active, const float *topk_w, int T, int E, int k, int H,
                              int I, uint16_t *out, void *workspace, size_t ws_bytes, int path,
                              void *stream);

/* Step 4 for callers that cannot allocate device memory.  The paper has no
 * counterpart: this is a convenience of this library.  Some callers are not
 * allowed to call cudaMalloc -- an engine that plans all device memory
 * before serving and forbids allocation afterwards, a plugin inside a host
 * application that owns the allocators, a latency-critical loop where an
 * allocation could synchronise the device -- so they cannot provide the
 * workspace moe_w4a16_down_combine needs.
 *
 * Same arguments, meaning and results as moe_w4a16_down_combine, without
 * the workspace.  Instead the library keeps one scratch array of
 * MOE_NOALLOC_SCRATCH_BYTES bytes in device memory, which every GPU that
 * loads the library holds until the process exits.  The call allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *   - Shapes whose moe_workspace_bytes(T, E, k, H, I) exceeds
 *     MOE_NOALLOC_SCRATCH_BYTES are rejected with MOE_ERR_UNSUPPORTED before
 *     anything is launched (at k = 10, H = 2560 that allows T <= 81).  Other
 *     size errors are those of moe_w4a16_down_combine.
 *   - Every call made outside stream capture looks up the scratch array's
 *     device address on the current device, so a device reset that reloads
 *     the library's module is harmless; a call made during capture reuses
 *     the address of the last call on that device, so make the first call on
 *     a device before any stream capture (otherwise MOE_ERR_CUDA).
 *   - Argument errors are reported before anything is enqueued: a rejected
 *     call leaves the stream and the scratch array untouched.
 *   - Every call shares the one array and it keeps the last call's contents;
 *     each call clears the parts that must start at zero (an asynchronous
 *     memset on `stream`).  Calls that overlap on the GPU, on any stream,
 *     race on the array and give wrong results: order them.
 *   - Device-detected errors are written to the scratch's error word, which
 *     moe_get_device_error cannot reach; the next call clears it. */
#define MOE_NOALLOC_SCRATCH_BYTES (8u << 20)

int moe_w4a16_down_combine_noalloc(const uint16_t *h,
                                   const uint32_t *w2_q, const uint16_t *w2_s,
                                   const uint32_t *w2_z, int group_size,
                                   const int32_t *expert_offsets, const int32_t *sorted_pair,
                                   const int32_t *active_experts, const int32_t *num_active,
                                   const float *topk_w, int T, int E, int k, int H, int I,
                                   uint16_t *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_W4A16_H */
