/*
 * pgg.h -- C ABI of the GB300 (sm_103a) MoE expert grouped GEMM library.
 *
 * The operation (from "Enabling DeepSeek-V4-Flash Training on AMD Instinct
 * MI355X GPUs with Primus", section "Expert parallelism: DeepEP and the grouped
 * GEMM"): tokens are already sorted by expert; each local expert multiplies its
 * own, different number of tokens by its own weights, and one kernel runs all
 * of the experts' GEMMs over the ragged batch instead of a per-expert loop.
 * The per-expert token counts ("m_splits" in "[Megatron-LM] feat: add grouped
 * gemm fp4 support ... Pull Request #891", review comments) are produced by
 * routing and bounded by the token count; here they are `group_lens`.
 *
 * Notation: G groups (experts), M = sum(group_lens) rows; group g owns rows
 * [off_g, off_g + len_g) with off_0 = 0 and off_{g+1} = off_g + len_g.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers, row-major, densely packed, and
 *    16-byte aligned; "bf16" means IEEE bfloat16 (2 bytes).
 *  - group_lens is a device int32[G]; it is scanned on the device (no host
 *    synchronisation).  1 <= G <= 1024.
 *  - The caller owns and allocates every buffer; the library allocates
 *    nothing and keeps no state beyond pgg_init's device properties.
 *  - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).
 *  - Host-detectable problems (null pointer, bad size, misalignment, an
 *    unsupported format or device) return a non-zero pgg_status and launch
 *    nothing.
 *  - Device-detectable problems (a negative group length, sum(group_lens) !=
 *    M, a bounded wait that expired) write a code to *err (a device int32,
 *    first error wins; may be NULL) and the kernel still terminates, writing
 *    no output for bad group_lens.  Clear *err to 0 before the call.
 *  - Results are deterministic: no floating-point atomics in any reduction.
 */
#ifndef PGG_H_
#define PGG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PGG_OK = 0,
  PGG_ERR_INVALID_ARG = 1,   /* null pointer, non-positive or too large size, bad enum */
  PGG_ERR_UNSUPPORTED = 2,   /* device is not sm_103, or a shape the kernels do not cover */
  PGG_ERR_ALIGNMENT = 3,     /* pointer not 16-byte aligned, or a dimension off its multiple */
  PGG_ERR_NOT_INITIALIZED = 4,
  PGG_ERR_CUDA = 5,          /* a CUDA runtime call failed */
  PGG_ERR_TOO_LARGE = 6,     /* the problem does not fit a no-alloc entry point's fixed scratch */
  /* codes written to the device error word */
  PGG_ERR_BAD_GROUP_LENS = 16, /* some len < 0, or sum(len) != M */
  PGG_ERR_TIMEOUT = 17,        /* a bounded pipeline wait expired; output incomplete */
  PGG_ERR_PAD_OVERFLOW = 18,   /* column-wise MX: sum(round_up(len, 128)) > M_pad */
  PGG_ERR_BAD_EXPERT = 19      /* MoE permute: an expert id outside [0, E) */
} pgg_status;

typedef enum { PGG_FMT_E4M3 = 1, PGG_FMT_E2M1 = 2 } pgg_mx_fmt;
typedef enum { PGG_MODE_FWD = 0, PGG_MODE_DGRAD = 1, PGG_MODE_WGRAD = 2 } pgg_mode;
typedef enum { PGG_EPI_NONE = 0, PGG_EPI_SWIGLU = 1 } pgg_epilogue;

/* Padding granule of the column-wise MX layout (rows per group are rounded up to it). */
#define PGG_MX_PAD 128

/* Library ABI version (major*100 + minor). */
int pgg_version(void);

/* Select `device` and check that it is an sm_103 GPU (compute capability
 * 10.3), caching its SM count.  Called implicitly by every entry point on the
 * current device; calling it first surfaces PGG_ERR_UNSUPPORTED early.  The
 * pages' counterpart is the hardware capability check made when the MXFP4
 * recipe is entered (Pull Request #891, review comments). */
int pgg_init(int device);

/* Static string for a status code. */
const char* pgg_status_string(int status);

/* Copy the device error word to *host_out, synchronising `stream` first. */
int pgg_read_error(const int32_t* err_dev, int32_t* host_out, void* stream);

/* ---------------------------------------------------------------- BF16 */

/* Forward: Y_g = X_g . W_g^T for every group.
 *   X [M, K] bf16, W [G, N, K] bf16 (K contiguous), Y [M, N] bf16 (out).
 *   fp32 accumulation in tensor memory, bf16 round-to-nearest-even output.
 *   K >= 8, K % 8 == 0, N % 8 == 0.  M == 0 is a no-op. */
int pgg_grouped_gemm_fwd(const void* X, const void* W, const int32_t* group_lens, void* Y,
                         int64_t M, int64_t N, int64_t K, int G, int32_t* err, void* stream);

/* Dgrad: dX_g = dY_g . W_g (same grouping, weight used transposed; W is read
 * in place, no transposed copy -- cf. the transposed-weight cache that Pull
 * Request #891, "Changes", stops reusing).
 *   dY [M, N] bf16, W [G, N, K] bf16, dX [M, K] bf16 (out).
 *   N >= 8, N % 8 == 0, K % 8 == 0. */
int pgg_grouped_gemm_dgrad(const void* dY, const void* W, const int32_t* group_lens, void* dX,
                           int64_t M, int64_t N, int64_t K, int G, int32_t* err, void* stream);

/* Variable-K wgrad: dW_g = dY_g^T . X_g, reduced over group g's own len_g
 * rows; a group with len_g == 0 gets dW_g = 0 (the backward emits dW1/dW2:
 * "Enabling DeepSeek-V4-Flash ...", section "MegaMoE", backward order).
 *   X [M, K] bf16, dY [M, N] bf16, dW [G, N, K] bf16 (out, fully written).
 *   N % 8 == 0, K % 8 == 0. */
int pgg_grouped_gemm_wgrad(const void* X, const void* dY, const int32_t* group_lens, void* dW,
                           int64_t M, int64_t N, int64_t K, int G, int32_t* err, void* stream);

/* Variable-K wgrad accumulated into an fp32 gradient buffer ("main_grad"):
 *   dW_f32[g] += dY_g^T . X_g  for every group (an empty group adds nothing).
 * The weight-gradient bridge of "[Megatron-LM] feat: add grouped gemm fp4
 * support ... Pull Request #891", "Changes": the weight gradient is always
 * accumulated into weight.main_grad.  fp32 accumulation in tensor memory; the
 * add into dW_f32 is done by bulk tensor reduce-adds, one add per element per
 * call, so repeated calls (gradient accumulation over micro-batches) are
 * deterministic.
 *   X [M, K] bf16, dY [M, N] bf16, dW_f32 [G, N, K] fp32 (in/out).
 *   N % 8 == 0, K % 8 == 0.  Calls that overlap on the same dW_f32 race. */
int pgg_grouped_gemm_wgrad_accumulate(const void* X, const void* dY, const int32_t* group_lens,
                                      float* dW_f32, int64_t M, int64_t N, int64_t K, int G,
                                      int32_t* err, void* stream);

/* FC1 with SwiGLU folded into the epilogue ("Primus-Turbo" README, "What's
 * New": fused GroupedMLP with SwiGLU folded into the grouped GEMM; weight
 * layout w1 [g, 2I, H] "gate + up" from the MegaMoE section).
 *   H_g = X_g . W1_g^T  [len_g, 2I];  A = silu(H[:, :I]) * H[:, I:]
 *   X [M, K] bf16, W1 [G, 2I, K] bf16 (rows 0..I-1 gate, I..2I-1 up),
 *   A [M, I] bf16 (out), H [M, 2I] bf16 (out, optional: NULL skips it; it is
 *   the pre-activation the backward needs).  silu(x) = x / (1 + exp(-x)),
 *   evaluated in fp32 from the fp32 accumulators.  I % 8 == 0, K % 8 == 0. */
int pgg_grouped_fc1_swiglu(const void* X, const void* W1, const int32_t* group_lens, void* A,
                           void* H, int64_t M, int64_t I, int64_t K, int G, int32_t* err,
                           void* stream);

/* FC2 dgrad with the SwiGLU backward in the epilogue:
 *   dA_g = dY_g . W2_g  [len_g, I];  with g = H[:, :I], u = H[:, I:], s = sigmoid(g):
 *   dH[:, :I] = dA * u * s * (1 + g * (1 - s)),  dH[:, I:] = dA * g * s
 *   dY [M, Hd] bf16, W2 [G, Hd, I] bf16, H [M, 2I] bf16 (saved by FC1),
 *   dH [M, 2I] bf16 (out).  Hd % 8 == 0, I % 8 == 0. */
int pgg_grouped_fc2_dgrad_swiglu_bwd(const void* dY, const void* W2, const void* H,
                                     const int32_t* group_lens, void* dH, int64_t M, int64_t Hd,
                                     int64_t I, int G, int32_t* err, void* stream);

/* Clamped SwiGLU (the `swiglu_limit` knob of "Enabling DeepSeek-V4-Flash ...",
 * model-config table; the pages give no formula -- read here as): with L =
 * swiglu_limit > 0, gate <- min(gate, L) and up <- clamp(up, -L, L) before
 * A = silu(gate) * up.  H keeps the values before the clamp; the backward
 * applies the clamp to them again and passes no gradient where a clamp is
 * active (gate > L, |up| > L).  swiglu_limit == 0 is the plain SwiGLU (the two
 * calls above); a negative or non-finite limit returns PGG_ERR_INVALID_ARG.
 * Arguments otherwise as pgg_grouped_fc1_swiglu / pgg_grouped_fc2_dgrad_swiglu_bwd. */
int pgg_grouped_fc1_swiglu_clamped(const void* X, const void* W1, const int32_t* group_lens, void* A,
                                   void* H, int64_t M, int64_t I, int64_t K, int G, float swiglu_limit,
                                   int32_t* err, void* stream);
int pgg_grouped_fc2_dgrad_swiglu_bwd_clamped(const void* dY, const void* W2, const void* H,
                                             const int32_t* group_lens, void* dH, int64_t M, int64_t Hd,
                                             int64_t I, int G, float swiglu_limit, int32_t* err,
                                             void* stream);

/* ---------------------------------------------------------------- MX (microscaling) */

/* Row-wise MX quantization: one E8M0 scale per block of 32 consecutive
 * elements along C ("Primus-Turbo" README: MXFP8 / MXFP4 grouped GEMM; Pull
 * Request #891, "Changes": MXFP4 weights built as float4_e2m1fn_x2 buffers).
 * Rule (OCP Microscaling v1.0): E = clamp(floor(log2(amax)) - emax, -127, 127)
 * with emax 8 (e4m3) or 2 (e2m1), scale code E + 127, element code =
 * round-to-nearest-even(v * 2^-E) saturated to +-448 / +-6, sign of zero kept;
 * a block with a NaN or Inf gets scale 0xFF and zero codes.
 *   in [R, C] bf16; C % 32 == 0.
 *   codes [R, C] u8 (e4m3) or [R, C/2] u8 (e2m1: element 2j in the low
 *   nibble of byte j); scales [R, C/32] u8. */
int pgg_mx_quantize_rowwise(const void* in, int64_t R, int64_t C, int fmt, uint8_t* codes,
                            uint8_t* scales, void* stream);

/* Row-wise MX quantization with the scales in the blocked atom layout of the
 * block-scaled MMA -- the weight operand of the forward GEMM, quantized once
 * into the caller's weight cache.  Codes and the quantization rule are those of
 * pgg_mx_quantize_rowwise.
 *   in [R, C] bf16; C % 128 == 0.  codes as pgg_mx_quantize_rowwise.
 *   scales: round_up(R, 128) * C / 32 bytes; block j of row r sits at byte
 *   ((r / 128) * (C / 128) + j / 4) * 512 + 16 (r % 32) + 4 ((r % 128) / 32) + j % 4;
 *   rows past R hold scale 0. */
int pgg_mx_quantize_rowwise_blocked(const void* in, int64_t R, int64_t C, int fmt, uint8_t* codes,
                                    uint8_t* scales, void* stream);

/* Group-aware column-wise MX quantization (the wgrad operands, quantized
 * along the token axis).  Blocks of 32 rows run inside one group, starting at
 * the group's first row; group g is stored transposed in columns
 * [P_g, P_g + round_up(len_g, 32)) of the output, where P_g is the exclusive
 * prefix sum of round_up(len_h, PGG_MX_PAD).  Tail positions and everything
 * past the last group up to M_pad hold code 0 and scale 0.
 *   in [M, C] bf16; group_lens may be NULL for one group of M rows.
 *   codes_t [C, M_pad] u8 (e4m3) or [C, M_pad/2] (e2m1).
 *   scales_t: round_up(C, 128) * M_pad / 32 bytes in the blocked layout the
 *   block-scaled MMA reads: one 512-byte atom per 128-row block rb of C and
 *   per 128-column k-block p of [0, M_pad), at byte (rb * M_pad / 128 + p) * 512;
 *   inside it the scale of row 128 rb + m, 32-block 4 p + q sits at byte
 *   16 (m % 32) + 4 (m / 32) + q.  Rows past C hold scale 0.
 *   M_pad % PGG_MX_PAD == 0 and M_pad >= sum(round_up(len_g, PGG_MX_PAD))
 *   (else *err = PGG_ERR_PAD_OVERFLOW and nothing is written);
 *   M + G * (PGG_MX_PAD - 1) rounded up to PGG_MX_PAD always suffices. */
int pgg_mx_quantize_colwise(const void* in, int64_t M, int64_t C, const int32_t* group_lens,
                            int G, int fmt, uint8_t* codes_t, uint8_t* scales_t, int64_t M_pad,
                            int32_t* err, void* stream);

/* Block-scaled grouped GEMM on MX operands (both operands in `fmt`, scales
 * applied per 32-element block of the reduction axis, fp32 accumulation,
 * bf16 output):
 *   PGG_MODE_FWD:   out[M, N] = deq(A)_g . deq(B)_g^T
 *                   A [M, K] row-wise codes, SA [M, K/32];
 *                   B [G*N, K] row-wise codes (W) with SB in the blocked layout
 *                   of pgg_mx_quantize_rowwise_blocked.
 *                   epilogue PGG_EPI_SWIGLU: N = 2I, out = A_act [M, I],
 *                   out2 = H [M, 2I] or NULL (as pgg_grouped_fc1_swiglu).
 *   PGG_MODE_DGRAD: out[M, K] = deq(A)_g . W_g with A = dY [M, N] row-wise
 *                   codes (blocks along N), SA [M, N/32]; B = W quantized
 *                   along N and stored transposed, [K, G*N] codes, SB in the
 *                   blocked layout of pgg_mx_quantize_colwise (that call on W
 *                   viewed as [G*N, K] with G groups of N rows and M_pad =
 *                   G*N produces exactly this).
 *                   epilogue PGG_EPI_SWIGLU: the SwiGLU backward with the
 *                   saved bf16 H [M, 2K]; out = dH [M, 2K].
 *   PGG_MODE_WGRAD: out[G, N, K] = sum over group g's padded columns of
 *                   deq(A)[:, r] deq(B)[:, r]^T with A = dY column-wise
 *                   codes [N, M_pad], B = X column-wise codes [K, M_pad],
 *                   SA / SB their blocked scales (pgg_mx_quantize_colwise);
 *                   empty groups give 0.
 * Fused MX output (SwiGLU epilogues only; both NULL to skip): out_codes /
 * out_scales receive the row-wise MX quantization, in `fmt`, of the bf16 tensor
 * written to `out` (A of the forward, dH of the dgrad) -- bit-identical to
 * pgg_mx_quantize_rowwise(out) -- so the next GEMM's operand needs no separate
 * quantize pass ("Primus-Turbo" README, "What's New": fused GroupedMLP in
 * FP8 / MXFP8).  The width of `out` (I) must be a multiple of 32.
 * Row-major scales (fwd SA, dgrad SA) need 4-byte alignment, blocked ones
 * (fwd SB, dgrad SB, wgrad SA / SB) 16-byte alignment.
 * Sizes: the reduction axis is a multiple of 128 (fwd K, dgrad N); the other
 * dimensions are multiples of 8 (N of a SwiGLU forward a multiple of 16); e2m1
 * codes are packed two per byte.  fp32 accumulation, bf16 output. */
int pgg_mx_grouped_gemm(int mode, int fmt, int epilogue, const uint8_t* A, const uint8_t* SA,
                        const uint8_t* B, const uint8_t* SB, const void* H,
                        const int32_t* group_lens, void* out, void* out2, uint8_t* out_codes,
                        uint8_t* out_scales, int64_t M, int64_t N, int64_t K, int G,
                        int64_t M_pad, int32_t* err, void* stream);

/* ---------------------------------------------------------------- FP8 tensor-wise */

/* FP8 (e4m3) with one fp32 scale per tensor, computed from the tensor itself
 * ("current scaling": "[Megatron-LM] feat: add grouped gemm fp4 support ...
 * Pull Request #891", description and "Changes": the grouped linear layer's
 * FP8 path is the plain grouped_gemm_fp8 call, and under current scaling a
 * cached transposed weight must not be reused; "Primus-Turbo" README: FP8
 * GroupedGEMM).  The pages give no formula; the library takes the usual
 * per-tensor recipe:
 *   amax = max |x| over the tensor's finite elements;
 *   s = 448 / amax in fp32 (1 when amax is 0; clamped to the largest finite
 *       fp32 if the quotient overflows), so the largest element maps to +-448;
 *   code = e4m3 round-to-nearest-even of the fp32 product x * s, saturating
 *       at +-448 (+-Inf saturates too);
 *   deq(code) = decode(code) / s.
 * amax_scale is a device float[2] = {s, amax}, 16-byte aligned.  Every tensor
 * that the GEMM below reads takes its own amax_scale. */

/* amax and s of a bf16 tensor of n elements (n % 8 == 0; n == 0 gives s = 1,
 * amax = 0).  Writes amax_scale[0..1]; two small kernels and a 4-byte memset. */
int pgg_fp8_tensor_scale(const void* in, int64_t n, float* amax_scale, void* stream);

/* Row-major e4m3 codes [R, C] of bf16 in [R, C] with the scale amax_scale[0]
 * (from pgg_fp8_tensor_scale on the same tensor).  C % 8 == 0. */
int pgg_fp8_quantize_rowwise(const void* in, int64_t R, int64_t C, const float* amax_scale, uint8_t* codes,
                             void* stream);

/* Column-wise e4m3 codes for the wgrad GEMM: codes_t [C, M_pad], where group
 * g's row i of in [M, C] lands in column poff_g + i, poff the prefix sum of
 * round_up(len_g, PGG_MX_PAD), and every other column holds code 0 (the same
 * layout as pgg_mx_quantize_colwise's codes, with no scales).  group_lens NULL
 * means one group of M rows (G 0 or 1).  C % 8 == 0; M_pad a multiple of
 * PGG_MX_PAD; a layout past M_pad sets *err = PGG_ERR_PAD_OVERFLOW and writes
 * nothing.  W [G, N, K] for the dgrad GEMM is the same call on W viewed as
 * [G*N, K] with G groups of N rows and M_pad = G*N: codes_t = W^T [K, G*N]. */
int pgg_fp8_quantize_colwise(const void* in, int64_t M, int64_t C, const int32_t* group_lens, int G,
                             const float* amax_scale, uint8_t* codes_t, int64_t M_pad, int32_t* err,
                             void* stream);

/* Bytes of the workspace pgg_fp8_grouped_gemm needs: 0 (the FP8 MMAs read no
 * scale factors).  Kept so that callers sizing a workspace keep working. */
size_t pgg_fp8_workspace_size(int64_t N, int64_t K, int G, int64_t M_pad);

/* FP8 tensor-wise grouped GEMM (grouped_gemm_fp8): the operands, shapes and
 * epilogues of pgg_mx_grouped_gemm with fmt e4m3, each operand carrying one
 * scale instead of per-block scales:
 *   FWD    out[M, N]    = deq(A)_g . deq(B)_g^T   A = X codes [M, K], B = W codes [G*N, K]
 *   DGRAD  out[M, K]    = deq(A)_g . W_g          A = dY codes [M, N], B = W^T codes [K, G*N]
 *   WGRAD  out[G, N, K] = sum over group g's padded columns of deq(A)[:, r] deq(B)[:, r]^T
 *                         A = dY^T codes [N, M_pad], B = X^T codes [K, M_pad] (column-wise)
 * i.e. the sum of code products divided by s_A s_B, fp32 accumulation, bf16 out.
 * epilogue PGG_EPI_SWIGLU (fwd / dgrad, as pgg_mx_grouped_gemm): the fused
 * GroupedMLP in FP8 ("Primus-Turbo" README, "What's New": FP8 / MXFP8 expert
 * MLP with SwiGLU folded into the grouped GEMM).  FWD: N = 2I, out = A_act
 * [M, I], out2 = H [M, 2I] or NULL; DGRAD: the SwiGLU backward with the saved
 * bf16 H [M, 2K], out = dH [M, 2K].  swiglu_limit > 0 clamps as in
 * pgg_grouped_fc1_swiglu_clamped (0: none; SwiGLU epilogue only).  There is no
 * fused quantized output: a current-scaled operand needs the amax of the whole
 * tensor before any of its codes.
 * scale_a / scale_b point at each operand's s (its amax_scale).  The tensor
 * cores run the plain FP8 MMA (tcgen05 kind::f8f6f4, e4m3 x e4m3, fp32
 * accumulation); 1 / (s_A s_B) is applied in the epilogue.  ws / ws_bytes:
 * reserved, ignored (may be NULL / 0).  The size rules, errors and group
 * semantics are pgg_mx_grouped_gemm's (fwd K and dgrad N multiples of 128). */
int pgg_fp8_grouped_gemm(int mode, int epilogue, const uint8_t* A, const float* scale_a, const uint8_t* B,
                         const float* scale_b, const void* H, const int32_t* group_lens, void* out, void* out2,
                         int64_t M, int64_t N, int64_t K, int G, int64_t M_pad, float swiglu_limit, void* ws,
                         size_t ws_bytes, int32_t* err, void* stream);

/* ---------------------------------------------------------------- MoE glue (one GPU) */

/* Bytes of the scratch table pgg_moe_permute needs: ceil(T / 32) * E * 4. */
size_t pgg_moe_permute_workspace_size(int64_t T, int E);

/* Token permute into the expert-sorted layout the grouped GEMM consumes
 * ("Enabling DeepSeek-V4-Flash ...", section "Expert parallelism: DeepEP and
 * the grouped GEMM": the dispatch lays tokens out for the grouped GEMM; on one
 * GPU it has no communication).  Entry (t, j) -- token t's j-th routed expert
 * e = topk_ids[t, j] -- becomes row pos[t, j] of Xs; rows are ordered by expert,
 * then token, then choice (a stable sort of the flattened entries by expert),
 * so group g's rows are [sum_{h<g} len_h, sum_{h<=g} len_h).
 *   topk_ids [T, k] int32 in [0, E); X [T, H] bf16 (may be NULL: routing only);
 *   Xs [T * k, H] bf16 (out; rows past sum(group_lens) untouched);
 *   group_lens [E] int32 (out); pos [T, k] int32 (out);
 *   ws: device scratch of at least pgg_moe_permute_workspace_size(T, E) bytes,
 *   owned by the caller, 4-byte aligned, clobbered.
 *   1 <= k <= 32, 1 <= E <= 1024, T * k < 2^31, H % 8 == 0.
 * An id outside [0, E) sets *err = PGG_ERR_BAD_EXPERT; that entry gets
 * pos = -1, is not counted and not copied.  The result is deterministic. */
int pgg_moe_permute(const int32_t* topk_ids, const void* X, int64_t T, int k, int64_t H, int E,
                    void* Xs, int32_t* group_lens, int32_t* pos, void* ws, size_t ws_bytes,
                    int32_t* err, void* stream);

/* Combine ("Enabling DeepSeek-V4-Flash ...", section "MegaMoE": the second
 * grouped GEMM is followed by the combine and the weighted reduce):
 *   out[t] = sum_j w[t, j] * Ys[pos[t, j]], fp32 accumulation in choice order,
 *   bf16 output.  w NULL means weight 1, which makes this also the permute's
 *   backward: dX[t] = sum_j dXs[pos[t, j]].  Entries with pos < 0 are skipped.
 *   Ys [R, H] bf16 (R >= max pos + 1); pos [T, k] int32; w [T, k] fp32 or NULL;
 *   out [T, H] bf16.  1 <= k <= 32, H % 8 == 0. */
int pgg_moe_combine(const void* Ys, const int32_t* pos, const float* w, void* out, int64_t T, int k,
                    int64_t H, void* stream);

/* Backward of the weighted combine:
 *   dYs[pos[t, j]] = bf16(w[t, j] * dOut[t]);  dw[t, j] = <dOut[t], Ys[pos[t, j]]>
 *   (fp32 dot product in a fixed order: deterministic).  Entries with pos < 0
 *   get dw = 0 and leave dYs untouched.
 *   dOut [T, H] bf16, Ys [R, H] bf16, pos [T, k] int32, w [T, k] fp32,
 *   dYs [R, H] bf16 (out), dw [T, k] fp32 (out).  1 <= k <= 32, H % 8 == 0. */
int pgg_moe_combine_bwd(const void* dOut, const void* Ys, const int32_t* pos, const float* w,
                        void* dYs, float* dw, int64_t T, int k, int64_t H, void* stream);

/* Capacity of pgg_moe_permute_noalloc's fixed scratch, in int32 entries
 * (4 MiB of device memory in the library's module): ceil(T / 32) * E must not
 * exceed it, e.g. 131072 tokens over 256 experts or 32768 over 1024. */
#define PGG_MOE_NOALLOC_MAX_WS_INTS (1 << 20)

/* pgg_moe_permute without a caller workspace.  The pages have no counterpart:
 * it exists for callers that cannot provide device scratch -- a C or real-time
 * component without access to the framework's allocator and with a fixed
 * memory budget, or code that must not call cudaMalloc because it
 * synchronises the device.  The count table lives instead in a statically
 * sized array of the library's own module (PGG_MOE_NOALLOC_MAX_WS_INTS int32
 * entries per device), and the call allocates nothing.
 *   Arguments, layouts and results are those of pgg_moe_permute without ws /
 *   ws_bytes.  ceil(T / 32) * E > PGG_MOE_NOALLOC_MAX_WS_INTS returns
 *   PGG_ERR_TOO_LARGE and launches nothing.
 *   The first call on each device looks up the array's device address (with
 *   that device current) and caches it; make that first call before any
 *   stream capture.  The cache is keyed on the context: after a device reset
 *   (cudaDeviceReset) the next call looks the address up again, in the new
 *   context, so that call too should come before any stream capture.
 *   All calls on one device share the one array: calls that may overlap on
 *   the GPU (different streams without ordering between them) race and give
 *   wrong results.  Calls ordered on one stream are safe. */
int pgg_moe_permute_noalloc(const int32_t* topk_ids, const void* X, int64_t T, int k, int64_t H,
                            int E, void* Xs, int32_t* group_lens, int32_t* pos, int32_t* err,
                            void* stream);

/* The block-scaled grouped GEMM with the clamped SwiGLU epilogue (see
 * pgg_grouped_fc1_swiglu_clamped): mode PGG_MODE_FWD (FC1) or PGG_MODE_DGRAD
 * (FC2 dgrad + SwiGLU backward); the other arguments as pgg_mx_grouped_gemm
 * with epilogue PGG_EPI_SWIGLU. */
int pgg_mx_grouped_gemm_clamped(int mode, int fmt, const uint8_t* A, const uint8_t* SA, const uint8_t* B,
                                const uint8_t* SB, const void* H, const int32_t* group_lens, void* out,
                                void* out2, uint8_t* out_codes, uint8_t* out_scales, int64_t M, int64_t N,
                                int64_t K, int G, float swiglu_limit, int32_t* err, void* stream);

/* Test hook; the pages have no counterpart.  Runs the forward grouped GEMM --
 * BF16 when fmt == 0 (A = X, B = W, SA and SB unused), else the block-scaled
 * forward in `fmt` (arguments as pgg_mx_grouped_gemm with PGG_MODE_FWD and
 * PGG_EPI_NONE) -- with every pipeline wait limited to `wait_ns` and the load
 * producer of each CTA told to stop before its `stall_at`-th k-block.  The MMA
 * and epilogue waits behind that k-block then run out, and the kernel must take
 * its failure path: raise the CTA's abort flag, drain what it issued, free its
 * tensor memory, exit, and write PGG_ERR_TIMEOUT to *err, leaving the device
 * usable for the next call.  It exists so that tests can run that path without
 * faulting or hanging the GPU.  stall_at >= 0; 100 us <= wait_ns <= 1 s.  The
 * output is incomplete. */
int pgg_test_stalled_fwd(int fmt, const void* A, const uint8_t* SA, const void* B, const uint8_t* SB,
                         const int32_t* group_lens, void* out, int64_t M, int64_t N, int64_t K, int G,
                         int64_t stall_at, uint64_t wait_ns, int32_t* err, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PGG_H_ */
