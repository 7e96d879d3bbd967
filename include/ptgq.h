/*
 * ptgq.h -- C ABI of the GB300 (sm_103a) per-token-group 8-bit quantization library.
 *
 * The operation (sglang PR #30924, "unify per_token_group_quant into one trait-driven
 * JIT kernel", sections "Implementation breakdown" and "Key source snippets"
 * (ref_fp8_ue8m0); sglang PR #27449, "JIT port of per_token_group_quant_8bit_v2",
 * sections "Summary" and "Implementation notes"; vLLM PR #41326, "Blackwell
 * register-resident packed group quantization kernel", sections "Implementation
 * breakdown" and "Key source snippets"):
 *
 *   For every live token row and every contiguous group of G elements of that row
 *     v_i   = x_i                          (or silu(gate_i) * up_i, fused prologue)
 *     amax  = max(max_i |v_i|, eps)
 *     s     = amax / FMAX                  FMAX = 448 (e4m3) or 127 (int8)
 *     UE8M0 formats: e = biased_exponent(s) + (mantissa(s) != 0), scale = 2^(e-127)
 *     FP32  format : scale = s
 *     q_i   = saturate(round_to_nearest_even(v_i / scale))   to e4m3fn or int8
 *   All arithmetic is IEEE binary32 with round-to-nearest-even; silu uses the
 *   correctly rounded binary32 exponential.  Codes and scales are bit-identical to
 *   that definition (the library is tested against an independent CPU oracle), except
 *   under PTGQ_FLAG_FAST_DIVIDE, which trades the exact quotient for compatibility.
 *
 * Conventions for every entry point:
 *   - Buffer pointers (x, out_q, out_s, masked_m, ...) are addresses the current device
 *     can access: device memory (cudaMalloc, a torch CUDA tensor), or page-locked host
 *     memory under unified addressing, which the kernel then reads and writes in place
 *     over the host link.  The caller owns every buffer; the library allocates nothing,
 *     never synchronises, never dereferences a buffer on the host, and launches at most
 *     one kernel per call on `stream`, so a call can be captured in a CUDA graph.
 *   - Errors are returned as negative status codes (below) before anything is
 *     launched; nothing is written in that case.  No exception crosses the ABI.
 *     PTGQ_ERR_CUDA reports a failed launch (the launch call's own status; that error
 *     is then cleared from the CUDA runtime's state).
 *   - The kernel is launched with programmatic stream serialization (PDL): it may
 *     start while the previous kernel on `stream` finishes, and waits for it
 *     (griddepcontrol.wait) before touching memory.
 */
#ifndef PTGQ_H_
#define PTGQ_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ptgq_stream_t; /* the same type as cudaStream_t */

/* Element type of x.  PTGQ_FP32 is accepted by ptgq_per_token_quant only. */
typedef enum { PTGQ_BF16 = 0, PTGQ_FP16 = 1, PTGQ_FP32 = 2 } ptgq_in_dtype;
/* Element type of out_q: FP8 E4M3 ("fn", max 448) or int8. */
typedef enum { PTGQ_E4M3 = 0, PTGQ_INT8 = 1 } ptgq_out_dtype;
/* Scale format:
 *   PTGQ_SCALE_FP32          float s per group.
 *   PTGQ_SCALE_UE8M0_PACKED  exponent byte e per group, four groups per int32 word, group
 *                            g in byte g % 4 (bits 8*(g%4)); unused bytes of the last word
 *                            are zero (vLLM PR #41326, test ..._packed_all_zero).
 *   PTGQ_SCALE_UE8M0_FP32    the power-of-two scale 2^(e-127) stored as a float. */
typedef enum {
  PTGQ_SCALE_FP32 = 0,
  PTGQ_SCALE_UE8M0_PACKED = 1,
  PTGQ_SCALE_UE8M0_FP32 = 2
} ptgq_scale_fmt;
/* Scale layout, with ncol = ng (float formats) or ceil(ng/4) (packed), rows = the out_q row
 * extent of one block and mn_pad = round_up(rows, 4):
 *   PTGQ_ROW_MAJOR      element (row, col) at row * ncol + col           ([rows, ncol])
 *   PTGQ_COL_MAJOR_TMA  element (row, col) at col * mn_pad + row         ([ncol, mn_pad]),
 *                       the TMA-aligned column-major layout (vLLM PR #41326, test
 *                       ..._packed_all_zero; sglang PR #35593, "Implementation breakdown"
 *                       item 3). */
typedef enum { PTGQ_ROW_MAJOR = 0, PTGQ_COL_MAJOR_TMA = 1 } ptgq_scale_layout;

/* Status codes. */
enum {
  PTGQ_OK = 0,
  PTGQ_ERR_NULL = -1,       /* a required pointer is NULL */
  PTGQ_ERR_DTYPE = -2,      /* unknown input dtype */
  PTGQ_ERR_OUT_DTYPE = -3,  /* unknown output dtype */
  PTGQ_ERR_GROUP = -4,      /* group_size not in {16, 32, 64, 128} (sglang PR #27449, "Notes") */
  PTGQ_ERR_HIDDEN = -5,     /* hidden <= 0 or hidden % group_size != 0 */
  PTGQ_ERR_SHAPE = -6,      /* negative count or expected_m, flat tokens_pad in
                             * (0, num_tokens), or more than 4096 experts (masked) */
  PTGQ_ERR_ALIGN = -7,      /* x not 32-byte, out_q not 16-byte or out_s not 4-byte aligned */
  PTGQ_ERR_SCALE_FMT = -8,  /* unknown scale format */
  PTGQ_ERR_LAYOUT = -9,     /* unknown scale layout */
  PTGQ_ERR_EPS = -10,       /* eps not finite or below PTGQ_EPS_MIN (2^-140) */
  PTGQ_ERR_FLAG = -11,      /* fuse_silu not 0 or 1, or an unknown flag bit */
  PTGQ_ERR_TOO_LARGE = -12, /* more than 2^31 - 1 work units (live rows times groups, or
                             * times packed words, per row), or an index beyond 2^62 */
  PTGQ_ERR_CUDA = -13       /* the kernel launch failed */
};

/* Smallest accepted eps, 2^-140.  It keeps the scale of an all-zero group positive:
 * RN(eps / FMAX) is at least the smallest binary32 subnormal for every eps >= 2^-140, while
 * a smaller eps could round it to zero and leave the group without a scale. */
#define PTGQ_EPS_MIN 0x1p-140f

/*
 * ptgq_quant -- per-token-group quantization, flat or masked (EP-MoE) scheduler.
 *
 *   x               input, row-major, element type `dtype`.
 *                     flat   (masked_m == NULL): [num_tokens, H_in]
 *                     masked (masked_m != NULL): [E, tokens_pad, H_in]
 *                   H_in = hidden, or 2*hidden with fuse_silu (gate columns [0, hidden),
 *                   up columns [hidden, 2*hidden); sglang PR #27449, "Validation").
 *                   32-byte aligned.
 *   num_tokens_or_E flat: number of token rows T.  masked: number of experts E.
 *   tokens_pad      flat: row extent of out_q (>= T, or 0 meaning T); rows [T, tokens_pad)
 *                   of out_q and the padded scale rows are zero-filled (vLLM PR #41326,
 *                   "Implementation breakdown" item 4).
 *                   masked: rows per expert in x, out_q and the scales.
 *   hidden          output width H; a multiple of group_size.
 *   group_size      G in {16, 32, 64, 128}.
 *   out_q           codes, row-major [rows, hidden] (flat) or [E, tokens_pad, hidden]
 *                   (masked), element type `out_dtype`.  16-byte aligned.
 *   out_s           scales: format `scale_fmt`, layout `scale_layout`; in masked mode one
 *                   block per expert, blocks back to back.  ptgq_scale_elems() gives the
 *                   number of elements (floats or int32 words).  4-byte aligned.
 *   fuse_silu       1: v = silu(gate) * up computed in binary32 before quantization.
 *   masked_m        NULL (flat) or device int32[E]: live rows of expert e are
 *                   [0, masked_m[e]) (values outside [0, tokens_pad] are clamped).  In
 *                   masked mode nothing outside the live rows is written or loaded:
 *                   padding rows keep the caller's contents (sglang PR #35593, "Key source
 *                   snippets", test_masked_rows_and_k_tail).  A call may prefetch guessed
 *                   rows into L2 (row 0 of each expert, or with expected_m the rows below
 *                   min(expected_m, tokens_pad)); their contents never reach the outputs.
 *   eps             floor of amax; finite and >= PTGQ_EPS_MIN.
 *   stream          CUDA stream of the launch.
 * Returns PTGQ_OK or a negative status.
 *
 * Non-finite amax.  x is finite in normal use, but a silu product can overflow binary32
 * to +-inf (and x may hold an infinity).  Such a group follows the same definition:
 * amax = +inf, s = +inf (fp32 format), e = 255 (UE8M0: byte 0xFF; float scale +inf).  Each
 * quotient v / +inf is a signed zero for finite v (codes 0x00 / 0x80, int8 0) and NaN for
 * an infinite v, encoded 0x7F (the e4m3 NaN) or 0 (int8).  Other groups are unaffected.
 */
int ptgq_quant(const void* x, int dtype, int64_t num_tokens_or_E, int64_t tokens_pad,
               int64_t hidden, int group_size, void* out_q, int out_dtype, void* out_s,
               int scale_fmt, int scale_layout, int fuse_silu, const int32_t* masked_m,
               float eps, ptgq_stream_t stream);

/* Flags of ptgq_quant_ex. */
enum {
  /* Launch without programmatic stream serialization (plain stream order). */
  PTGQ_FLAG_NO_PDL = 1,
  /* vLLM semantics for UE8M0 scales: s = max(s, 1e-10) before rounding up to a power of
   * two (vLLM PR #41326, test ..._packed_all_zero docstring: an all-zero group then gets
   * exponent byte 0x5E).  No effect on PTGQ_SCALE_FP32. */
  PTGQ_FLAG_UE8M0_SCALE_FLOOR = 2,
  /* Compatibility with builds compiled with fast math (SGLang PR #34257, "Implementation
   * notes": with --use_fast_math the division by the scale rounds differently, and SGLang
   * PR #30924, "Risks": about 0.2% of int8 codes differ by one from such a build).  Each
   * element quotient x / s is taken with CUDA's approximate division __fdividef (at most
   * 2 ulp from the IEEE quotient for the scales that occur here) instead of IEEE division.
   * Scales are unchanged.  Affects only PTGQ_SCALE_FP32: the UE8M0 quotient is an exact
   * multiply by a power of two, so the flag has no effect there. */
  PTGQ_FLAG_FAST_DIVIDE = 4
};

/* ptgq_quant with option flags (a bitwise OR of PTGQ_FLAG_*), a hint and an error counter;
 * flags == 0, expected_m == 0 and masked_m_errors == NULL is ptgq_quant.
 *   expected_m  masked mode: the caller's estimate of the live rows per expert (sglang PR
 *               #30924, "Implementation breakdown" item 2: the custom op takes masked_m
 *               and expected_m).  The live counts sit in device memory, so without a hint
 *               the grid is sized for every row of tokens_pad being live; with one it is
 *               sized for E * min(expected_m, tokens_pad) rows.  Results are the same for
 *               any value: the grid strides over whatever rows are live, so a low hint
 *               costs time, never correctness.  Rows below min(expected_m, tokens_pad)
 *               of x (row 0 of each expert without a hint) may be prefetched into L2
 *               before the live counts are known (a cache hint: their contents never reach
 *               the outputs), so x must span its whole [E, tokens_pad, H_in] extent, as
 *               ptgq_quant requires.  0: no hint.  Ignored in flat mode.
 *               Negative: PTGQ_ERR_SHAPE.
 *   masked_m_errors  masked mode: NULL, or a 4-byte aligned device int32 to which the call
 *               adds the number of experts e < E whose masked_m[e] lies outside
 *               [0, tokens_pad] (such counts are clamped, never a fault).  A second kernel
 *               of one CTA, launched after the quantizer on the same stream, adds it with
 *               atomic adds, so calls on several streams may share the counter.  The caller
 *               zeroes it and reads it after the stream's work.  Ignored in flat mode. */
int ptgq_quant_ex(const void* x, int dtype, int64_t num_tokens_or_E, int64_t tokens_pad,
                  int64_t hidden, int group_size, void* out_q, int out_dtype, void* out_s,
                  int scale_fmt, int scale_layout, int fuse_silu, const int32_t* masked_m,
                  float eps, ptgq_stream_t stream, unsigned flags, int64_t expected_m,
                  int32_t* masked_m_errors);

/* Size helper: the number of scale elements (floats, or int32 words for the packed format)
 * that out_s must hold for these arguments (masked != 0 selects the masked layout, where
 * num_tokens_or_E is E).  Host-only; touches no device.  Returns a status code. */
int ptgq_scale_elems(int64_t num_tokens_or_E, int64_t tokens_pad, int64_t hidden,
                     int group_size, int scale_fmt, int scale_layout, int masked,
                     int64_t* n_out);

/*
 * ptgq_per_token_quant -- per-token (whole-row) FP8 e4m3 quantization (sglang PR #34257,
 * "Key source snippets": the per-token kernels and their host contract).
 *
 * For each row r < num_tokens of x [num_tokens, hidden]:
 *   s   = max_i |x_i| / 448          (binary32 division; no eps floor)
 *   inv = s == 0 ? 0 : 1 / s         (an all-zero row gets scale 0 and codes 0)
 *   q_i = e4m3(clamp(x_i * inv, -448, 448)),   out_s[r] = s
 * The multiplication by the reciprocal (not a division) is the page's definition.
 *
 *   x         device, row-major [num_tokens, hidden], dtype PTGQ_BF16, PTGQ_FP16 or
 *             PTGQ_FP32; 16-byte aligned (8-byte suffices for 16-bit rows with
 *             hidden % 8 != 0).
 *   hidden    a positive multiple of 4.
 *   out_q     device e4m3 codes, row-major with row length `hidden`; it may have more rows
 *             than num_tokens (a padded output): rows past num_tokens are not touched.
 *             8-byte aligned for 16-bit input with hidden % 8 == 0, else 4-byte.
 *   out_s     device float scales, one per row; entries past num_tokens are not touched.
 * Returns PTGQ_OK or a negative status (checked before launching).
 */
int ptgq_per_token_quant(const void* x, int dtype, int64_t num_tokens, int64_t hidden,
                         void* out_q, float* out_s, ptgq_stream_t stream);

/*
 * ptgq_requant_per_tensor -- per-token-group FP8 to per-tensor FP8 requantization over the
 * masked EP-MoE layout (sglang PR #35593, "Key source snippets": the requant kernel and
 * test_masked_rows_and_k_tail).
 *
 * For every expert e < num_experts and row r < clamp(masked_m[e], 0, m) (all m rows when
 * masked_m is NULL), and every column c < k:
 *   out[e, r, c] = e4m3_satfinite((decode(x[e, r, c]) * x_scale[e, r, c / group_size])
 *                                 * (1 / *output_scale))
 * with binary32 products in that order and a saturating round-to-nearest-even conversion.
 * Rows at or past masked_m[e] are not written and do not affect the result; the kernel may
 * read or prefetch some of them (every e < num_experts, r < m lies inside x and x_scale).
 *
 *   x             device e4m3 codes [num_experts, m, k], row-major, 16-byte aligned.
 *   x_scale       device float per-token-group scales; element (e, r, g) at
 *                 e * scale_stride_e + r * scale_stride_m + g * scale_stride_g (strides in
 *                 elements, e.g. the column-major [E, m, k/group] layout of the page:
 *                 (m * k/group, 1, m)).  The caller guarantees that every element with
 *                 e < num_experts, r < m and g < k/group lies inside it, dead rows included
 *                 (the kernel may prefetch their scales into L2).
 *   masked_m      device int32[num_experts] live rows per expert, or NULL.
 *   output_scale  device pointer to the one binary32 per-tensor output scale.
 *   out           device e4m3 codes [num_experts, m, k], 16-byte aligned.
 *   k             a multiple of group_size; group_size in {16, 32, 64, 128}.
 * Returns PTGQ_OK or a negative status (checked before launching).
 */
int ptgq_requant_per_tensor(const void* x, const float* x_scale, int64_t scale_stride_e,
                            int64_t scale_stride_m, int64_t scale_stride_g,
                            const int32_t* masked_m, const float* output_scale, void* out,
                            int64_t num_experts, int64_t m, int64_t k, int group_size,
                            ptgq_stream_t stream);

/* A static, human-readable description of a status code. */
const char* ptgq_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* PTGQ_H_ */
