/*
 * moe.h -- C ABI of the GB300 (sm_103a) routed-expert hot path.
 *
 * One call runs, on one GPU, the routed-expert layer whose caller owns the
 * activations x[T,d] (bf16), the top-k expert ids[T,k] (int32, distinct per
 * row), the routing scores[T,k] (fp32) and the expert weights W13[E,2I,d] and
 * W2[E,d,I] (bf16):
 *
 *     dispatch (expert-major permutation) -> W13 grouped GEMM -> SwiGLU
 *       -> W2 grouped GEMM x score -> deterministic combine
 *
 * and its backward (input gradients, weight gradients accumulated in place,
 * score gradients).  Sources: "Dist-MoE: Meta's Blackwell SM100 MoE Kernels"
 * (section "What it is selling": caller-owned inputs, one library-owned
 * context, the pipeline, FPROP/DGRAD/WGRAD, BF16 with FP32 accumulate, MXFP8
 * E4M3 after routing with prepared weights, plain/clamped SwiGLU, in-place
 * WGRAD; section "Caveats": fixed physical token count with zero-score padding,
 * sequentially reusable, non-reentrant contexts, fatal scratch overflow) and
 * the "nvfp4moe" README (section "Grouped GEMM": expert-major rows, m_indptr of
 * length E+1, empty experts; section "MoE layer": distinct int32 ids, fp32
 * weights, workspace overwritten by the next call, one plan per stream,
 * allocation-free warmed plans; sections "Training" and "Supported kernel
 * surface": deterministic dispatch, combine and router gradients; "Limits").
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller unless the
 *     argument name ends in _host.  The library never frees them.
 *   - bf16 tensors are passed as void* holding IEEE bfloat16 values; all
 *     tensors are dense row-major (C order) with the shapes given.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Work is enqueued on it; no entry point below synchronises unless it says
 *     so.  A plan is not reentrant: use one plan per concurrent stream.
 *   - Return value: MOE_OK (0) or one of the MOE_ERR_* codes.  Argument errors
 *     are detected on the host before anything is enqueued.  Errors found by
 *     the device (bad ids, a wait that gave up) are recorded in the plan's
 *     device error word and reported by moe_plan_check().
 *   - No entry point allocates device memory after moe_plan_set_workspace();
 *     forward and backward enqueue kernels and async copies only, so they may
 *     be captured in a CUDA graph.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define MOE_OK                0
#define MOE_ERR_INVALID_ARG   1  /* bad size, null pointer, misaligned pointer   */
#define MOE_ERR_WORKSPACE     2  /* workspace missing or too small               */
#define MOE_ERR_STATE         3  /* e.g. backward without a saving forward       */
#define MOE_ERR_BAD_IDS       4  /* device found an id outside [0,E) or repeated */
#define MOE_ERR_TIMEOUT       5  /* a device-side wait gave up                   */
#define MOE_ERR_CUDA          6  /* a CUDA runtime/driver call failed            */
#define MOE_ERR_UNSUPPORTED   7  /* combination not implemented                  */

/* ---- precisions ------------------------------------------------------------ */
#define MOE_PREC_BF16   0   /* bf16 operands, fp32 accumulate                     */
#define MOE_PREC_MXFP8  1   /* E4M3 operands with E8M0 scales per 32 along K      */
#define MOE_PREC_NVFP4  2   /* E2M1 operands with E4M3 scales per 16 along K and
                               per-tensor scales; inference only                   */

/* ---- workspace flags ------------------------------------------------------- */
#define MOE_WS_TRAINING     1  /* keep forward activations and backward buffers */
#define MOE_WS_HOST_STAGING 2  /* device copies of per-step host inputs/outputs  */

typedef struct moe_plan moe_plan;

/*
 * moe_plan_create -- describe one routed-expert layer.
 *   T  physical tokens per call (a fixed shape: callers with fewer tokens pad
 *      and give the padding rows zero scores -- "Caveats", item 2)
 *   d  hidden size, I expert intermediate size, E experts, k experts per token
 *   precision  MOE_PREC_BF16 or MOE_PREC_MXFP8
 * Limits ("Limits" section of the nvfp4moe README, adapted to whole tiles):
 *   d % 128 == 0, I % 64 == 0, 1 <= k <= E <= 256, T >= 1, T*k < 2^31.
 * Returns a host-side plan object (owned by the caller, free with
 * moe_plan_destroy) or NULL on invalid arguments.  Does not touch the GPU
 * except to query the current device's properties.  A plan belongs to the
 * device current at creation (its grids are sized for that device's SMs): make
 * that device current for every later call with the plan.  Plans on different
 * devices may be used from different host threads at once.
 */
moe_plan* moe_plan_create(int T, int d, int I, int E, int k, int precision);

/* Free the plan (host memory only; the caller frees its workspace). */
void moe_plan_destroy(moe_plan* plan);

/*
 * Clamped SwiGLU ("What it is selling": plain or clamped SwiGLU).  limit = 0
 * selects plain silu(gate)*up; limit > 0 clips gate and up to [-limit, limit]
 * before the activation, and the backward passes gradient only where the
 * pre-activation lies inside the closed interval.
 */
int moe_plan_set_swiglu_clamp(moe_plan* plan, float limit);

/*
 * Bytes of device workspace the plan needs for `flags` (MOE_WS_*).  The size
 * covers the worst case of padded expert-major rows,
 *   Rpad <= T*k + E*(G-1)    (G = the plan's row granule, 128 or 256),
 * so it never depends on the routing.  Returns 0 for a NULL plan.
 */
size_t moe_plan_workspace_bytes(const moe_plan* plan, int flags);

/*
 * Hand the plan a caller-allocated device buffer (256-byte aligned) of at least
 * moe_plan_workspace_bytes(plan, flags) bytes.  The plan owns its contents from
 * now on ("MoE layer": the workspace is overwritten by the next call).  Clears
 * the device error word (a synchronous cudaMemset on the legacy stream).
 * Returns MOE_ERR_WORKSPACE if `bytes` is too small.
 */
int moe_plan_set_workspace(moe_plan* plan, void* workspace, size_t bytes, int flags);

/*
 * Forward.  Inputs (device):
 *   x       [T, d]  bf16         ids  [T, k] int32      scores [T, k] fp32
 *   w13     [E, 2I, d] bf16: rows [0,I) gate, [I,2I) up (not interleaved)
 *   w2      [E, d, I]  bf16
 *   For MOE_PREC_MXFP8, w13/w2 hold E4M3 codes (uint8, same shapes) and
 *   w13_sf / w2_sf their E8M0 scales in the tiled layout, both produced by
 *   moe_prepare_weights_mxfp8; for bf16 pass NULL.  An MXFP8 plan quantises
 *   the routed activation rows along d and h along I (32-element blocks) and
 *   runs block-scaled E4M3 GEMMs; it needs I % 128 == 0, d <= 4096, I <= 4096.
 *   With save_for_backward = 1 it also keeps a and the routed x rows
 *   quantised along the rows for moe_backward_mxfp8 (h is kept as its E4M3
 *   codes only; the backward recomputes the bf16 h from a).
 * Output: y [T, d] bf16, overwritten:
 *   y[t] = bf16( sum_{j=0..k-1} bf16( scores[t,j] * W2[e] . h ) ),
 *   h = bf16(silu(G) * U),  (G, U) = bf16(W13[e] . x[t]),  e = ids[t,j]
 * (sum in fixed j order).  save_for_backward = 1 keeps what moe_backward needs
 * in the workspace (requires a MOE_WS_TRAINING workspace).
 * Ids outside [0,E) or repeated within a row set MOE_ERR_BAD_IDS in the device
 * error word (detail = smallest offending flat index t*k+j); such elements are
 * dropped, so memory stays safe, but y is then not meaningful.
 */
int moe_forward(moe_plan* plan, const void* x, const int32_t* ids, const float* scores,
                const void* w13, const void* w2, const uint8_t* w13_sf, const uint8_t* w2_sf,
                void* y, int save_for_backward, void* stream);

/*
 * Forward over rows the caller has already laid out expert-major (nvfp4moe
 * README, "MoE layer": its run_routed entry takes such rows with m_indptr and
 * the padded offsets, for callers that route on their own).  Dispatch and gather are
 * skipped; the W13 GEMM + SwiGLU and the W2 GEMM run over the caller's layout,
 * and the combine runs when row_of and y are given.  Inputs (device):
 *   x_e      [rows, d] bf16: expert e's routed rows at [off_pad[e], off_pad[e] + m_e)
 *            with m_e = m_indptr[e+1] - m_indptr[e]; the rows up to off_pad[e+1]
 *            are padding (computed like routed rows; zero rows give zero outputs)
 *   m_indptr [E+1] int32: m_indptr[0] = 0, non-decreasing (exact row counts)
 *   off_pad  [E+1] int32: off_pad[0] = 0, every entry a multiple of
 *            moe_tile_rows() (128), off_pad[e+1] - off_pad[e] >= m_e,
 *            off_pad[E] <= rows
 *   score_of [rows] fp32 routing score of each row, or NULL (no score)
 *   w13, w2  as moe_forward (bf16 plans)
 *   row_of   [T, k] int32 row of x_e holding token t's j-th contribution (-1:
 *            none), or NULL
 * Outputs (device):
 *   ys [rows, d] bf16: ys[r] = bf16(score_of[r] * W2[e] . h),
 *      h = bf16(silu(G) * U), (G, U) = bf16(W13[e] . x_e[r]), for the m tiles
 *      that hold routed rows (rows in other tiles are not written)
 *   y  [T, d] bf16 (with row_of, else NULL): y[t] = bf16(sum_j ys[row_of[t,j]])
 *      in fixed j order
 * On the same layout, inputs and weights, ys and y equal those of moe_forward
 * bit for bit.  rows <= the plan's worst-case padded row count
 * (T*k + E*127 rounded down to a multiple of 128), else MOE_ERR_INVALID_ARG.
 * The layout is checked on the device: an inconsistent m_indptr / off_pad runs
 * no tile and records MOE_ERR_INVALID_ARG in the device error word (detail:
 * the first offending expert index e, 0..E); on a consistent layout a row_of
 * entry outside [0, off_pad[E]) is treated as -1 and records
 * MOE_ERR_INVALID_ARG with detail E + 1 + its flat index t*k + j.  bf16 plans
 * only (MOE_ERR_UNSUPPORTED otherwise).  The call uses the plan's workspace
 * (h, the tile list, a checked copy of row_of), so it overwrites the tables of
 * the previous call and cannot be followed by moe_backward.
 */
int moe_forward_routed(moe_plan* plan, const void* x_e, long long rows, const int32_t* m_indptr,
                       const int32_t* off_pad, const float* score_of, const void* w13,
                       const void* w2, void* ys, const int32_t* row_of, void* y, void* stream);

/*
 * Backward of the last saving forward on this plan ("What it is selling":
 * DGRAD and WGRAD; nvfp4moe "Training": router gradients).  Inputs: dy [T, d]
 * bf16 and the same w13/w2 as the forward.  Outputs:
 *   dx      [T, d]      bf16, overwritten
 *   dscores [T, k]      fp32, overwritten (gradient w.r.t. the given scores)
 *   dw13    [E, 2I, d]  fp32, ACCUMULATED in place (+=); experts with no rows
 *   dw2     [E, d, I]   fp32, ACCUMULATED in place      are left untouched
 * Returns MOE_ERR_STATE if no saving forward preceded it, MOE_ERR_UNSUPPORTED
 * for an MXFP8 plan (use moe_backward_mxfp8).
 */
int moe_backward(moe_plan* plan, const void* dy, const void* w13, const void* w2,
                 void* dx, float* dw13, float* dw2, float* dscores, void* stream);

/*
 * Backward of an MXFP8 plan ("What it is selling": MXFP8 E4M3 for FPROP, DGRAD
 * and WGRAD; nvfp4moe "Training").  Every block-scaled GEMM takes its operands
 * quantised in 32-element blocks along its own K (block rule of
 * moe_quantize_mxfp8):
 *   DGRAD-W2:  dY rows along d, W2[e]^T prepared along d         -> g
 *   DGRAD-W13: dA rows along 2I, W13[e]^T prepared along 2I       -> dX_e
 *   WGRAD-W2:  dY and hs along the rows of each expert            -> dW2[e]
 *   WGRAD-W13: dA and x along the rows of each expert             -> dW13[e]
 * (row blocks start at each expert's first padded row; the zero padding rows do
 * not change a block's scale).  Rounding points and outputs are those of
 * moe_backward: dx, dscores overwritten, dw13/dw2 accumulated in place.
 * w13t/w13t_sf and w2t/w2t_sf come from moe_prepare_weights_mxfp8_backward.
 * Needs a MOE_WS_TRAINING workspace and a saving forward (MOE_ERR_STATE
 * otherwise); MOE_ERR_UNSUPPORTED for a bf16 plan.
 */
int moe_backward_mxfp8(moe_plan* plan, const void* dy, const uint8_t* w13t,
                       const uint8_t* w13t_sf, const uint8_t* w2t, const uint8_t* w2t_sf,
                       void* dx, float* dw13, float* dw2, float* dscores, void* stream);

/*
 * One training (or, with dy_host == NULL, inference) step from HOST buffers:
 * copies x_host, ids_host, scores_host (and dy_host) into the plan's staging
 * area, runs moe_forward (+ moe_backward), and copies y (and dx, dscores) back
 * into the host buffers, all enqueued on `stream`; the caller synchronises the
 * stream before reading the host outputs.  The copies run on a plan-owned side
 * stream (created with the host-staging workspace) that joins `stream` at the
 * end of the step, overlapped with compute: x and dY upload during dispatch and
 * the forward, y downloads during the backward, dx and dscores during the
 * weight-gradient GEMMs.  After a training step on the plan, the next step's
 * uploads need not wait for that step to end (its last reads of the staged
 * inputs came before its dX combine), so in a loop of training steps they
 * overlap the previous step's weight-gradient GEMMs.  The host buffers are read
 * and written asynchronously: the caller keeps the inputs unchanged and leaves
 * the outputs alone until the stream has passed the step.  Host buffers should
 * be pinned (page-locked) for the copies to be asynchronous.  Weights and weight
 * gradients stay on the device.  Needs a MOE_WS_HOST_STAGING workspace (plus
 * MOE_WS_TRAINING when dy_host != NULL).
 */
int moe_step_host(moe_plan* plan, const void* x_host, const int32_t* ids_host,
                  const float* scores_host, const void* dy_host,
                  const void* w13, const void* w2, float* dw13, float* dw2,
                  void* y_host, void* dx_host, float* dscores_host, void* stream);

/*
 * MXFP8 block quantiser ("What it is selling": MXFP8 E4M3 with prepared
 * weights).  in [rows, K] bf16 -> codes [rows, K] E4M3, scales [rows, K/32]
 * E8M0, per 32-element block along K: X = floor(log2(amax)) - 8 clamped to
 * [-127,127], scale code X+127 (0 for an all-zero block), code =
 * E4M3(v * 2^-X) rounded to nearest even and saturated to +-448.
 * K % 32 == 0.  Used to prepare weights and exported for bit-exact tests.
 */
int moe_quantize_mxfp8(const void* in, long rows, int K, uint8_t* codes, uint8_t* scales,
                       void* stream);

/*
 * Prepared MXFP8 weights ("What it is selling": MXFP8 E4M3 accepts prepared
 * weights; nvfp4moe "Training": re-prepare after each optimizer step).
 * Quantises w13 [E,2I,d] along d and w2 [E,d,I] along I with the block rule of
 * moe_quantize_mxfp8 into
 *   w13_codes [E,2I,d], w2_codes [E,d,I]  (E4M3 bytes, same layout as the input)
 *   w13_scales, w2_scales                 (E8M0 bytes in the tiled layout the
 *                                           block-scaled GEMMs read; sizes from
 *                                           moe_mxfp8_weight_scale_bytes)
 * Tiled scale layout: rows are grouped in blocks of 128 and K in groups of 128
 * elements (four 32-element blocks); each (row block, K group) is a 512-byte
 * chunk, chunk index block*(K/128) + kb/4, in which row r = row%128 and block
 * j = kb%4 sit at byte 16*(r%32) + 4*(r/32) + j.  For W13 the row
 * blocks are, per expert, the 64 gate rows and 64 up rows of each 64-column
 * n-tile (block e*(I/64)+t holds gate rows [64t,64t+64) then up rows
 * [I+64t, I+64t+64)); for W2 they are consecutive 128-row blocks of [E*d].
 * d % 128 == 0, I % 128 == 0.
 */
size_t moe_mxfp8_weight_scale_bytes(int d, int I, int E,
                                    int which /* 0: W13, 1: W2, 2: W13^T, 3: W2^T */);
int moe_prepare_weights_mxfp8(const void* w13, const void* w2, int d, int I, int E,
                              uint8_t* w13_codes, uint8_t* w13_scales, uint8_t* w2_codes,
                              uint8_t* w2_scales, void* stream);

/*
 * Weights prepared for the MXFP8 backward (moe_backward_mxfp8): each expert's
 * matrix transposed so that the DGRAD GEMMs read it K-major, and quantised
 * along that K:
 *   w13t_codes [E, d, 2I]  W13[e]^T quantised along 2I
 *   w2t_codes  [E, I, d]   W2[e]^T  quantised along d
 * Scales in the tiled layout above with plain 128-row blocks of the transposed
 * matrices ([E*d] and [E*I] rows); sizes from moe_mxfp8_weight_scale_bytes
 * (which = 2, 3).  d % 128 == 0, I % 128 == 0.
 */
int moe_prepare_weights_mxfp8_backward(const void* w13, const void* w2, int d, int I, int E,
                                       uint8_t* w13t_codes, uint8_t* w13t_scales,
                                       uint8_t* w2t_codes, uint8_t* w2t_scales, void* stream);

/*
 * NVFP4 inference ("Dist-MoE" note, "What it is selling": the FP4 mode serves
 * inference only, with weights prepared ahead of the call; nvfp4moe README,
 * "Dense GEMM" / "Grouped GEMM": E2M1 codes two to a byte, one E4M3 scale per
 * block, one dequantisation scale per tensor, the GEMM scaled by the product of
 * its operands' tensor scales; "MoE layer": fixed activation scales from a
 * calibration pass or a checkpoint).  Block rule: a tensor with per-tensor dequantisation
 * scale s has encode scale g = 1/s; each 16-element block along K with amax A
 * gets the E4M3 scale code E4M3((A / 6) * g) and its elements
 * E2M1(v * (g / S)), S the scale's value (fp32 arithmetic, round to nearest
 * even, saturating; S = 0 gives zero codes).  Codes are packed two per byte,
 * element 2i in the low nibble.
 *
 * An NVFP4 plan (precision MOE_PREC_NVFP4; d % 256 == 0, I % 256 == 0) takes
 * only an inference workspace (flags 0; MOE_ERR_UNSUPPORTED for
 * MOE_WS_TRAINING or MOE_WS_HOST_STAGING) and runs moe_forward_nvfp4 only
 * (moe_forward returns MOE_ERR_UNSUPPORTED).
 */

/*
 * Static activation scales of an NVFP4 plan: the per-tensor dequantisation
 * scales of the routed activation rows (x_scale) and of h (h_scale), e.g.
 * amax / (6 * 448) of calibration data (moe_amax_bf16).  Values beyond the
 * calibrated range saturate.  Both > 0 and finite (MOE_ERR_INVALID_ARG).
 */
int moe_plan_set_activation_scales(moe_plan* plan, float x_scale, float h_scale);

/*
 * Prepared NVFP4 weights: W13 [E,2I,d] quantised along d and W2 [E,d,I] along I,
 * each expert with its own dequantisation scale amax(W[e]) / (6 * 448) (1 for
 * an all-zero expert):
 *   w13_codes [E, 2I, d/2], w2_codes [E, d, I/2]   packed E2M1
 *   w13_sf, w2_sf                                  E4M3 scales, tiled: rows in
 *       blocks of 128, K in groups of 64 elements (four 16-element blocks); each
 *       (row block, K group) a 512-byte chunk, chunk index block*(K/64) + k/64,
 *       row r = row%128 and block j = (k/16)%4 at byte 16*(r%32) + 4*(r/32) + j;
 *       W13 row blocks per expert and 64-column n-tile (64 gate rows, then the
 *       same 64 up rows), W2 plain 128-row blocks of [E*d]
 *   w13_scale, w2_scale [E] fp32 (device)
 * Buffer sizes from moe_nvfp4_weight_bytes (which: 0 W13 codes, 1 W13 scales,
 * 2 W2 codes, 3 W2 scales).  d % 256 == 0, I % 256 == 0.
 */
size_t moe_nvfp4_weight_bytes(int d, int I, int E, int which);
int moe_prepare_weights_nvfp4(const void* w13, const void* w2, int d, int I, int E,
                              uint8_t* w13_codes, uint8_t* w13_sf, float* w13_scale,
                              uint8_t* w2_codes, uint8_t* w2_sf, float* w2_scale, void* stream);

/*
 * NVFP4 inference forward: x [T,d] bf16, ids, scores as moe_forward; weights
 * from moe_prepare_weights_nvfp4.  The routed x rows are quantised along d with
 * the static x scale; gate/up = bf16(alpha13 * sum) with alpha13 = x_scale *
 * w13_scale[e] (R1); h = bf16(silu(G) * U) (R2) quantised along I with the
 * static h scale; ys = bf16(s * (alpha2 * sum)), alpha2 = h_scale * w2_scale[e]
 * (R3); y = the fixed-order combine (R6).  MOE_ERR_STATE if the activation
 * scales were not set.
 */
int moe_forward_nvfp4(moe_plan* plan, const void* x, const int32_t* ids, const float* scores,
                      const uint8_t* w13_codes, const uint8_t* w13_sf, const float* w13_scale,
                      const uint8_t* w2_codes, const uint8_t* w2_sf, const float* w2_scale,
                      void* y, void* stream);

/*
 * amax = max |in[i]| over n bf16 values (device pointers; amax is one fp32 on
 * the device), for calibrating static NVFP4 scales.
 */
int moe_amax_bf16(const void* in, long long n, float* amax, void* stream);

/*
 * Synchronise the device, read and clear the plan's device error word.
 * Returns MOE_OK or the first recorded device error; *detail (may be NULL)
 * receives its detail (for MOE_ERR_BAD_IDS the smallest offending flat index).
 */
int moe_plan_check(moe_plan* plan, long long* detail);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(int status);

/*
 * Inspection of the plan's workspace (for tests and tools).  Returns the device
 * address and byte size of one internal tensor of the last call:
 *   MOE_BUF_M_INDPTR  int32 [E+1]    expert-major row offsets (exact counts)
 *   MOE_BUF_OFF_PAD   int32 [E+1]    row offsets with segments padded to BM
 *   MOE_BUF_ROW_OF    int32 [T*k]    padded row of element t*k+j (-1: dropped)
 *   MOE_BUF_TOKEN_OF  int32 [Rpad]   token of each padded row (-1: padding)
 *   MOE_BUF_SCORE_OF  fp32  [Rpad]   score of each padded row (0: padding)
 *   (NVFP4 plans: MOE_BUF_XQ / XSF / HQ / HSF hold packed E2M1 codes [Rpad, d/2],
 *   [Rpad, I/2] and their tiled E4M3 scales)
 *   MOE_BUF_XE        bf16  [Rpad,d] gathered activations
 *   MOE_BUF_A         bf16  [Rpad,2I] gate/up pre-activations (training)
 *   MOE_BUF_H         bf16  [Rpad,I] SwiGLU output (bf16 plans; MXFP8 plans keep
 *                                    only its E4M3 codes, MOE_BUF_HQ)
 *   MOE_BUF_YS        bf16  [Rpad,d] score-weighted expert outputs
 *   MOE_BUF_DYE       bf16  [Rpad,d] gathered upstream gradient
 *   MOE_BUF_DA        bf16  [Rpad,2I] gradient at gate/up (bf16 plans; MXFP8 plans
 *                                    keep only its E4M3 codes, MOE_BUF_DAQ / DAQT)
 *   MOE_BUF_HS        bf16  [Rpad,I] score * h, the WGRAD-W2 operand (bf16 plans;
 *                                    MXFP8 plans keep only MOE_BUF_HSQT)
 *   MOE_BUF_DXE       bf16  [Rpad,d] per-row input gradients
 * Rows are valid up to off_pad[E].  Sizes are the worst-case capacities.  A
 * tensor the plan does not hold returns MOE_ERR_WORKSPACE.
 * off_pad rounds each expert's segment up to moe_plan_row_granule(plan) rows.
 */
#define MOE_BUF_M_INDPTR 0
#define MOE_BUF_OFF_PAD  1
#define MOE_BUF_ROW_OF   2
#define MOE_BUF_TOKEN_OF 3
#define MOE_BUF_SCORE_OF 4
#define MOE_BUF_XE       5
#define MOE_BUF_A        6
#define MOE_BUF_H        7
#define MOE_BUF_YS       8
#define MOE_BUF_DYE      9
#define MOE_BUF_DA       10
#define MOE_BUF_HS       11
#define MOE_BUF_DXE      12
#define MOE_BUF_XQ       13   /* u8   [Rpad,d] E4M3 activations (MXFP8 plans) */
#define MOE_BUF_XSF      14   /* u8   tiled E8M0 scales of XQ                   */
#define MOE_BUF_HQ       15   /* u8   [Rpad,I] E4M3 h (MXFP8 plans)             */
#define MOE_BUF_HSF      16   /* u8   tiled E8M0 scales of HQ                   */
#define MOE_BUF_XQT      17   /* MXFP8 training: E4M3 [d, Rpad], routed x quantised along the rows */
#define MOE_BUF_XQTSF    18   /* its tiled scales (row blocks over d, K groups over Rpad)      */
#define MOE_BUF_DAQ      19   /* MXFP8 training: E4M3 [Rpad, 2I], dA quantised along 2I        */
#define MOE_BUF_DASF     20   /* its tiled scales (row blocks over Rpad, K groups over 2I)     */
#define MOE_BUF_DAQT     21   /* MXFP8 training: E4M3 [2I, Rpad], dA quantised along the rows  */
#define MOE_BUF_DAQTSF   22   /* its tiled scales (row blocks over 2I, K groups over Rpad)     */
#define MOE_BUF_HSQT     23   /* MXFP8 training: E4M3 [I, Rpad], hs quantised along the rows   */
#define MOE_BUF_HSQTSF   24   /* its tiled scales (row blocks over I, K groups over Rpad)      */
int moe_plan_buffer(const moe_plan* plan, int which, void** dev_ptr, size_t* bytes);

/*
 * Stage timing (for benchmarks and tools).  `events` holds caller-created
 * cudaEvent_t handles (as void*); while set, each call records them on its
 * stream at its stage boundaries:
 *   which = 0 (moe_forward, n >= 6):  [0] start, [1] after dispatch (3 launches),
 *     [2] after gather, [3] after W13+SwiGLU, [4] after W2 x score, [5] after combine
 *   which = 1 (moe_backward, n >= 7): [0] start, [1] after dY gather,
 *     [2] after DGRAD-W2 + SwiGLU backward, [3] after DGRAD-W13,
 *     [4] after dX/dscores combine, [5] after WGRAD-W2, [6] after WGRAD-W13
 * n = 0 (or events = NULL) stops recording.  The plan keeps the pointer: the
 * array must stay valid while set.  The records are "external" ones
 * (cudaEventRecordExternal), so events captured in a CUDA graph still time
 * each replay.
 */
int moe_plan_set_timing_events(moe_plan* plan, int which, void* const* events, int n);

/*
 * Failure-path testing (the pages' kernels trap on fatal conditions, see
 * "Caveats"; this library records errors instead).  wait_limit_ns > 0 makes
 * every bounded device wait of this plan's GEMM kernels give up after that many
 * nanoseconds (0 restores the default of 2 s); stall_w13 = 1 makes the MMA role
 * of the W13 GEMM wait on a barrier that nothing arrives at, so that wait runs
 * out: the kernel then records MOE_ERR_TIMEOUT (detail = the wait's site), stops
 * every role, drains its outstanding copies and MMAs with bounded waits, frees
 * its tensor memory and exits, leaving the CUDA context usable.  The outputs of
 * such a call are not meaningful.  stall_w13 = 0 restores normal operation.
 */
int moe_plan_set_debug(moe_plan* plan, long long wait_limit_ns, int stall_w13);

/*
 * Concurrent backward.  wgrad_sms > 0 makes moe_backward run the two
 * weight-gradient GEMMs (bound by the fp32 gradient traffic) on a plan-owned
 * stream, with persistent grids of wgrad_sms CTAs, while DGRAD-W13 (bound by
 * the tensor pipe and its operand loads) and the dX combine run on the
 * caller's stream on the other SMs; the caller's stream then waits for the
 * weight gradients, so the call's semantics are unchanged and the results are
 * bit-identical (every tile is computed the same way).  0 (the default)
 * launches every GEMM on every SM, one after the other.  With stage timing
 * events set, the events of the weight-gradient stages are recorded on the
 * plan's stream.  The first call with wgrad_sms > 0 creates the stream and two
 * events (no device memory).  0 <= wgrad_sms < the number of SMs, else
 * MOE_ERR_INVALID_ARG.  Applies to moe_backward and moe_backward_mxfp8.
 */
int moe_plan_set_backward_split(moe_plan* plan, int wgrad_sms);

/*
 * Weight-gradient tile order.  Each SM walks its weight-gradient tiles
 * longest expert first; a tile of a heavy expert is bound by its K loop over
 * the expert's rows and leaves DRAM idle, a tile of a light expert by the
 * read-modify-write of its fp32 gradient.  With min_rows > 0, the tiles of
 * experts with more than min_rows routed rows (padded) run in pieces on one
 * accumulator, each piece followed by a whole tile of a lighter expert on the
 * other, so that the light tiles' gradient traffic overlaps the heavy tiles'
 * K loops.  Every tile still sums its K range in the same order, so the
 * gradients are bit-identical to those of the plain order (min_rows = 0).
 * Default 2560.  min_rows < 0 or > 2^30: MOE_ERR_INVALID_ARG.  Applies to
 * moe_backward and moe_backward_mxfp8.
 */
int moe_plan_set_wgrad_interleave(moe_plan* plan, long long min_rows);

/* Number of SMs of the plan's device (the persistent kernels' grid size). */
int moe_plan_num_sms(const moe_plan* plan);

/* Number of kernels this plan has launched so far (all entry points). */
long long moe_plan_launch_count(const moe_plan* plan);

/*
 * moe_dispatch_static -- the expert-major dispatch of moe_forward (per-expert
 * histogram, prefix scan, stable scatter) for callers that cannot allocate
 * device memory: code that runs inside another framework's allocator or
 * memory-pool callbacks, hosts whose device memory is already carved into
 * fixed pools, or processes that may only touch memory they are handed.  It
 * calls no cudaMalloc, cudaFree or other allocating routine; the kernels'
 * scratch (chunk histograms, counts, tile table, error word) lives in one
 * static __device__ array of about 280 KB that every GPU loading this library
 * keeps until the process exits.  The source pages have no counterpart of this
 * entry point.
 *   ids [T,k] int32, scores [T,k] fp32                       (inputs, device)
 *   m_indptr [E+1], off_pad [E+1], row_of [T*k] int32,
 *   token_of [rows_capacity] int32, score_of [rows_capacity] fp32,
 *   status [2] int32: {MOE_OK or MOE_ERR_BAD_IDS, smallest bad flat index or -1}
 *                                                            (outputs, device)
 * Same contents as the tables moe_forward builds (see moe_plan_buffer) for a
 * plan whose row granule is 128.
 * Limits: T*k <= MOE_STATIC_MAX_ROUTED (else MOE_ERR_WORKSPACE: the static
 * scratch is too small), k <= E <= 256, rows_capacity >=
 * floor((T*k + E*(BM-1)) / BM) * BM (else MOE_ERR_INVALID_ARG).
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current.  The address is kept per
 * device and CUDA context: the first call from another context on the device
 * (a non-primary context, or the primary context re-created after
 * cudaDeviceReset) looks it up again and is a first call in the same sense.  All calls on a device share the one array,
 * which keeps the last call's contents (the error word is cleared at the start
 * of each call): calls whose work overlaps on the GPU (for example on two
 * streams) race and must not be issued.
 */
#define MOE_STATIC_MAX_ROUTED 262144
int moe_dispatch_static(const int32_t* ids, const float* scores, int T, int k, int E,
                        int32_t* m_indptr, int32_t* off_pad, int32_t* row_of, int32_t* token_of,
                        float* score_of, long long rows_capacity, int32_t* status, void* stream);

/* Rows per GEMM m tile (128). */
int moe_tile_rows(void);

/*
 * Row GEMMs on CTA pairs.  on = 1 runs W13, W2 and DGRAD-W13 of a bf16 plan on
 * pairs of CTAs of a thread-block cluster with 256 x 256 tiles (tcgen05
 * cta_group::2), each CTA reading a third less operand data per product: the
 * 128-row m tiles of each expert go to the pair kernel two at a time, and an
 * expert's odd last m tile to the one-CTA kernel (dispatch builds both lists),
 * so expert segments stay padded to 128 rows.  DGRAD-W2 stays on one CTA.
 * Must be called before moe_plan_workspace_bytes / moe_plan_set_workspace
 * (MOE_ERR_STATE afterwards); needs d % 256 == 0 and I % 256 == 0 (else
 * MOE_ERR_UNSUPPORTED).
 */
int moe_plan_set_cta_pairs(moe_plan* plan, int on);

/* Padding granule of this plan's expert segments (off_pad): 128. */
int moe_plan_row_granule(const moe_plan* plan);

/*
 * Dense bf16 GEMM through the same tcgen05 kernels (for tests):
 *   mode 0: C[M,N] bf16  = A[M,K] . B[N,K]^T      (both operands K-major)
 *   mode 1: C[M,N] bf16  = A[M,K] . B[K,N]        (B MN-major)
 *   mode 2: C[M,N] fp32 += A[K,M]^T . B[K,N]      (both operands MN-major)
 *   mode 3: as mode 0 on CTA pairs (256 x 256 tiles, M % 256 == N % 256 == 0)
 *   mode 4: as mode 1 on CTA pairs
 * M % 128 == 0, N % 64 == 0, K % 64 == 0 (mode 2: K % 128 == 0).  `scratch`
 * is a device buffer of moe_gemm_scratch_bytes(M, K) bytes for the tile tables.
 */
size_t moe_gemm_scratch_bytes(int M, int K);
int moe_gemm_bf16(int mode, const void* A, const void* B, void* C, int M, int N, int K,
                  void* scratch, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
