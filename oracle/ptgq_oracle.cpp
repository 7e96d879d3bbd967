// ptgq_oracle.cpp -- CPU oracle for per-token-group 8-bit activation quantization.
//
// TEST INFRASTRUCTURE, NOT PRODUCT CODE.  This file is the slow, single-threaded,
// obviously correct statement of what the quantizer computes.  Only the test
// suite, the smoke check and the CPU-baseline leg of the benchmark load it.  It
// shares no code, header, table or constant with the CUDA library: neither side
// includes, links or calls the other.
//
// Sources (web pages, cited by page and section):
//   [sglang#30924]  sglang PR #30924, "unify per_token_group_quant into one
//                   trait-driven JIT kernel" (prhub summary): "Implementation
//                   breakdown"; "Key source snippets" (test reference ref_fp8_ue8m0).
//   [sglang#34257]  sglang PR #34257, "per-token FP8 quantization moved to JIT"
//                   (prhub summary): "Key source snippets" (per-token kernels).
//   [sglang#35593]  sglang PR #35593, "W4AFP8 requant for 128-aligned hidden"
//                   (prhub summary): "Implementation breakdown"; "Key source snippets".
//   [sglang#27449]  sglang PR #27449, "JIT port of per_token_group_quant_8bit_v2"
//                   (GitHub PR body): "Summary"; "Implementation notes"; "Validation".
//   [vllm#41326]    vLLM PR #41326, "Blackwell register-resident packed group
//                   quantization kernel" (prhub summary): "Implementation
//                   breakdown"; "Key source snippets" (test ..._packed_all_zero).
//
// Floating point: every step is binary32 with IEEE round-to-nearest-even, in the
// order written here.  Build with -ffp-contract=off and without fast-math so the
// compiler neither fuses a multiply into an add nor reassociates.
//
// One addition is not from the pages: oracle_quant_quotient_bound gives, per element,
// the codes of the quotient moved k binary32 ulps down or up.  It checks the library's
// fast-math compatibility mode, whose division is only known to lie within 2 ulps of
// the exact quotient ([sglang#34257] "Implementation notes" and [sglang#30924] "Risks"
// report that such a division changes codes).
//
// Parity pins: every function below is checked in tests/test_oracle_pins.py,
// tests/test_oracle_pins_next.py and tests/test_oracle_pins_bounds.py against
// something other than itself (closed forms, library routines, the worked example
// of [vllm#41326], exhaustive enumeration, exact rational arithmetic), and
// tests/test_oracle_mutants.py checks that planted mistakes fail those pins.  No
// function here is "parity unpinned".

#include <cmath>
#include <cstdint>
#include <cstring>

namespace {

float bits_to_float(uint32_t b) { float f; std::memcpy(&f, &b, 4); return f; }
uint32_t float_to_bits(float f) { uint32_t b; std::memcpy(&b, &f, 4); return b; }

// ---- element decoding --------------------------------------------------------

// bfloat16 is the upper half of a binary32 word.
float bf16_to_float(uint16_t h) { return bits_to_float(static_cast<uint32_t>(h) << 16); }

// IEEE binary16 from its fields: 1 sign, 5 exponent bits (bias 15), 10 fraction bits.
float fp16_to_float(uint16_t h) {
  const int sign = h >> 15;
  const int e = (h >> 10) & 0x1F;
  const int m = h & 0x3FF;
  double v;
  if (e == 0) v = std::ldexp(static_cast<double>(m), -24);                 // subnormal: m * 2^-24
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = std::ldexp(static_cast<double>(1024 + m), e - 25);             // (1 + m/1024) * 2^(e-15)
  return static_cast<float>(sign ? -v : v);  // exact: binary16 values are binary32 values
}

float load_elem(const uint16_t* p, int in_dtype) {
  return in_dtype == 0 ? bf16_to_float(*p) : fp16_to_float(*p);
}

// ---- the fused silu(gate) * up prologue ---------------------------------------
// [sglang#30924, "Implementation breakdown" item 1: fused silu_and_mul as a trait;
//  sglang#27449, "Summary": fused silu+mul].  silu(g) = g / (1 + exp(-g)), all in
// binary32.  exp is the correctly rounded binary32 exponential: libm's binary64
// exp rounded once to binary32.

float exp_f32(float x) { return static_cast<float>(std::exp(static_cast<double>(x))); }

float silu_mul(float g, float u) {
  const float e = exp_f32(-g);
  const float d = 1.0f + e;
  const float s = g / d;
  return s * u;
}

// ---- scale -------------------------------------------------------------------
// [sglang#30924, "Key source snippets", ref_fp8_ue8m0]: amax is floored at eps,
// the raw scale is amax / FMAX, and the UE8M0 scale is the raw scale rounded up
// to a power of two by taking its biased exponent and adding one when any
// mantissa bit is set.  The result byte is that biased exponent e; the scale
// value is 2^(e - 127).

int ue8m0_exponent(float s) {
  const uint32_t b = float_to_bits(s);
  const int biased = static_cast<int>((b >> 23) & 0xFF);
  const int round_up = (b & 0x7FFFFF) != 0 ? 1 : 0;
  return biased + round_up;
}

float pow2_from_biased(int e) { return bits_to_float(static_cast<uint32_t>(e) << 23); }

// ---- 8-bit encodings ---------------------------------------------------------

// FP8 E4M3 "fn": 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
// infinities.  Finite magnitudes are the subnormals m * 2^-9 (m = 1..7) and the
// normals (1 + m/8) * 2^(E-7) for E = 1..15, except E = 15, m = 7 (NaN); the
// largest is 448.  The value is first clamped to [-448, 448] ([sglang#30924,
// "Key source snippets": quantize with bounds -FMAX, FMAX]; [sglang#35593, "Key
// source snippets": the satfinite conversion saturates instead of producing NaN]),
// then rounded to the nearest representable value, ties to the even mantissa.
// The sign is kept, so -0 and negative values that round to zero give 0x80.
// A NaN quotient (inf / inf: an element that is itself infinite in a group whose amax
// is infinite) is not clamped: [sglang#30924, "Key source snippets"] clamps with torch,
// which passes NaN through, and the cast to e4m3fn then gives the format's NaN.  It is
// encoded 0x7F, with the sign bit clear: IEEE arithmetic leaves the sign of such a NaN
// open (x86 and NVIDIA GPUs produce opposite default NaNs), so it is not carried.
uint8_t e4m3_encode(float y) {
  if (std::isnan(y)) return 0x7F;
  const uint8_t sign = std::signbit(y) ? 0x80 : 0x00;
  double a = std::fabs(static_cast<double>(y));
  if (a > 448.0) a = 448.0;
  if (a < 0x1p-6) {
    // Subnormal range, grid step 2^-9.  m == 8 lands on 2^-6, whose code 0x08
    // is the smallest normal, so the same formula covers it.
    const double m = std::nearbyint(a * 512.0);
    return static_cast<uint8_t>(sign | static_cast<int>(m));
  }
  int E;
  const double f = std::frexp(a, &E);            // a = f * 2^E, f in [0.5, 1)
  int exp2 = E - 1;                               // a = (1 + m/8) * 2^exp2
  double m = std::nearbyint((2.0 * f - 1.0) * 8.0);
  if (m == 8.0) { m = 0.0; exp2 += 1; }
  return static_cast<uint8_t>(sign | ((exp2 + 7) << 3) | static_cast<int>(m));
}

// int8: round to nearest, ties to even, then clamp to the int8 range
// [vllm#41326, "Key source snippets": min_8bit / max_8bit kernel bounds].  A NaN
// quotient (see e4m3_encode) has no integer value; it is encoded 0, the result of a
// float-to-integer conversion of NaN on NVIDIA GPUs and of torch's cast to int8.
int8_t int8_encode(float y) {
  if (std::isnan(y)) return 0;
  double r = std::nearbyint(static_cast<double>(y));
  if (r > 127.0) r = 127.0;
  if (r < -128.0) r = -128.0;
  return static_cast<int8_t>(r);
}

// Value of an e4m3fn code, from the format definition (NaN for 0x7F / 0xFF).
float e4m3_decode(uint8_t c) {
  const int sign = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  const double v = e == 0 ? std::ldexp(static_cast<double>(m), -9)
                          : std::ldexp(1.0 + m / 8.0, e - 7);
  return static_cast<float>(sign ? -v : v);
}

// ---- layouts -----------------------------------------------------------------

enum { IN_BF16 = 0, IN_FP16 = 1 };
enum { OUT_E4M3 = 0, OUT_INT8 = 1 };
enum { FMT_FP32 = 0, FMT_UE8M0_PACKED = 1, FMT_UE8M0_FP32 = 2 };
enum { LAYOUT_ROW = 0, LAYOUT_COL = 1 };
enum { FLAG_UE8M0_SCALE_FLOOR = 1 };

int64_t round_up4(int64_t v) { return (v + 3) / 4 * 4; }

struct ScaleGeom {
  int64_t ncol;     // scale columns: ng for float formats, ceil(ng/4) int32 words for packed
  int64_t rows;     // logical scale rows per block (the out_q row extent)
  int64_t mn_pad;   // column pitch of the column-major layout: rows rounded up to 4
  int64_t per_block;// scale elements per block (per expert in masked mode)
};

ScaleGeom scale_geom(int64_t rows, int64_t ng, int scale_fmt, int scale_layout) {
  ScaleGeom g;
  g.ncol = scale_fmt == FMT_UE8M0_PACKED ? (ng + 3) / 4 : ng;
  g.rows = rows;
  g.mn_pad = round_up4(rows);
  g.per_block = scale_layout == LAYOUT_ROW ? rows * g.ncol : g.ncol * g.mn_pad;
  return g;
}

int64_t scale_index(const ScaleGeom& g, int scale_layout, int64_t row, int64_t col) {
  // Row-major: [rows, ncol].  Column-major (TMA-aligned, [vllm#41326, test
  // ..._packed_all_zero]): element (row, col) at col * mn_pad + row.
  return scale_layout == LAYOUT_ROW ? row * g.ncol + col : col * g.mn_pad + row;
}

bool valid_args(int in_dtype, int64_t n, int64_t tokens_pad, int64_t hidden, int group_size,
                int out_dtype, int scale_fmt, int scale_layout, int fuse_silu) {
  if (in_dtype != IN_BF16 && in_dtype != IN_FP16) return false;
  if (out_dtype != OUT_E4M3 && out_dtype != OUT_INT8) return false;
  if (scale_fmt < 0 || scale_fmt > 2 || scale_layout < 0 || scale_layout > 1) return false;
  if (group_size != 16 && group_size != 32 && group_size != 64 && group_size != 128) return false;
  if (hidden <= 0 || hidden % group_size != 0) return false;
  if (n < 0 || tokens_pad < 0) return false;
  if (fuse_silu != 0 && fuse_silu != 1) return false;
  return true;
}

// A binary32 bound on a quotient known only to within k ulps of the exact x / s:
// with e = x / s evaluated in binary64 (exact to 2^-53 relative for binary32
// operands, far below one binary32 ulp) and u the binary32 ulp at |e| (2^-149 at
// zero and for subnormals), the bound is e + k*u rounded outward to binary32 (up
// for k > 0, down for k < 0).  The encoders are monotone, so a code between the
// encodings of the two bounds is consistent with such a division.  Used to check
// the fast-math compatibility mode, whose division has a documented error of at
// most 2 ulps (CUDA Math API, single-precision intrinsics, __fdividef).
float quotient_bound(float x, float s, int k) {
  const double e = static_cast<double>(x) / static_cast<double>(s);
  int ex = e == 0.0 ? -149 : std::ilogb(e);
  if (ex < -126) ex = -126;
  const double u = std::ldexp(1.0, ex - 23);
  const double b = e + k * u;
  float f = static_cast<float>(b);
  if (k > 0 && static_cast<double>(f) < b) f = std::nextafter(f, INFINITY);
  if (k < 0 && static_cast<double>(f) > b) f = std::nextafter(f, -INFINITY);
  return f;
}

}  // namespace

extern "C" {

float oracle_bf16_to_float(uint16_t h) { return bf16_to_float(h); }
float oracle_e4m3_decode(uint8_t c) { return e4m3_decode(c); }
float oracle_fp16_to_float(uint16_t h) { return fp16_to_float(h); }
float oracle_exp_f32(float x) { return exp_f32(x); }
float oracle_silu_mul(float g, float u) { return silu_mul(g, u); }
int oracle_ue8m0_exponent(float s) { return ue8m0_exponent(s); }
float oracle_pow2_from_biased(int e) { return pow2_from_biased(e); }
uint8_t oracle_e4m3_encode(float y) { return e4m3_encode(y); }
int8_t oracle_int8_encode(float y) { return int8_encode(y); }

// Scale elements (floats, or int32 words for the packed format) the scale buffer
// holds.  Flat: rows = tokens_pad (or num_tokens when tokens_pad is 0).  Masked:
// num_experts blocks of tokens_pad rows.
int64_t oracle_scale_elems(int64_t n, int64_t tokens_pad, int64_t hidden, int group_size,
                           int scale_fmt, int scale_layout, int masked) {
  const int64_t rows = masked ? tokens_pad : (tokens_pad ? tokens_pad : n);
  const ScaleGeom g = scale_geom(rows, hidden / group_size, scale_fmt, scale_layout);
  return masked ? n * g.per_block : g.per_block;
}

// The whole operation on host buffers, same argument meaning as the library's
// ptgq_quant:
//   x        : input bit patterns (bf16 or fp16).  Flat: [n, H_in].  Masked:
//              [n = E, tokens_pad, H_in].  H_in = hidden, or 2*hidden with
//              fuse_silu (gate columns [0, hidden), up columns [hidden, 2*hidden)).
//   out_q    : 8-bit codes.  Flat: [rows, hidden] with rows = tokens_pad or n.
//              Masked: [E, tokens_pad, hidden].
//   out_s    : scales in the requested format and layout (see scale_geom).
//   masked_m : NULL for the flat scheduler, else int32[E] live rows per expert.
//   flags    : FLAG_UE8M0_SCALE_FLOOR applies the extra max(s, 1e-10) of the
//              vLLM kernel before UE8M0 rounding ([vllm#41326], test
//              ..._packed_all_zero docstring).  0 otherwise.
//   quot_ulps: 0 for the operation itself.  Non-zero: each code is the encoding of a
//              bound on the quotient instead of the quotient, for checking a
//              division that is only known to lie within |quot_ulps| binary32 ulps
//              of the exact x / s (see quotient_bound).  Scales are unchanged.
// Returns 0, or -1 for invalid arguments.
static int quant_impl(const uint16_t* x, int in_dtype, int64_t n, int64_t tokens_pad,
                      int64_t hidden, int group_size, uint8_t* out_q, int out_dtype, void* out_s,
                      int scale_fmt, int scale_layout, int fuse_silu, const int32_t* masked_m,
                      float eps, int flags, int quot_ulps) {
  if (!valid_args(in_dtype, n, tokens_pad, hidden, group_size, out_dtype, scale_fmt, scale_layout,
                  fuse_silu))
    return -1;
  const bool masked = masked_m != nullptr;
  if (!masked && tokens_pad != 0 && tokens_pad < n) return -1;

  const int64_t H = hidden;
  const int64_t H_in = fuse_silu ? 2 * H : H;
  const int64_t G = group_size;
  const int64_t ng = H / G;
  const float fmax = out_dtype == OUT_E4M3 ? 448.0f : 127.0f;
  const int64_t blocks = masked ? n : 1;
  const int64_t rows = masked ? tokens_pad : (tokens_pad ? tokens_pad : n);
  const ScaleGeom sg = scale_geom(rows, ng, scale_fmt, scale_layout);

  float v[128];
  int exps[4];
  for (int64_t b = 0; b < blocks; ++b) {
    int64_t live = n;
    if (masked) {
      // [sglang#35593, "Key source snippets" test: rows past masked_m keep the
      // caller's values]; out-of-range counts are clamped to [0, tokens_pad].
      live = masked_m[b];
      if (live < 0) live = 0;
      if (live > tokens_pad) live = tokens_pad;
    }
    const uint16_t* xb = x + b * rows * H_in;
    uint8_t* qb = out_q + b * rows * H;
    float* sf = static_cast<float*>(out_s) + b * sg.per_block;
    uint32_t* sp = static_cast<uint32_t*>(out_s) + b * sg.per_block;

    for (int64_t r = 0; r < live; ++r) {
      const uint16_t* xr = xb + r * H_in;
      for (int64_t g = 0; g < ng; ++g) {
        // 1. the group's values, widened to binary32 (and the silu prologue)
        for (int64_t i = 0; i < G; ++i) {
          const int64_t c = g * G + i;
          if (fuse_silu)
            v[i] = silu_mul(load_elem(xr + c, in_dtype), load_elem(xr + H + c, in_dtype));
          else
            v[i] = load_elem(xr + c, in_dtype);
        }
        // 2. amax, floored at eps
        float amax = 0.0f;
        for (int64_t i = 0; i < G; ++i) amax = std::fmax(amax, std::fabs(v[i]));
        amax = std::fmax(amax, eps);
        // 3. scale.  An infinite amax (a silu product that overflows binary32, or an
        // infinite input) gives s = +inf, and for the UE8M0 formats e = 255 (byte 0xFF),
        // whose power of two 2^128 is +inf in binary32: every finite element's quotient
        // is then a signed zero, and an infinite element's is NaN (see e4m3_encode).
        float s = amax / fmax;
        float scale = s;
        int e = 0;
        if (scale_fmt != FMT_FP32) {
          if (flags & FLAG_UE8M0_SCALE_FLOOR) s = std::fmax(s, 1e-10f);
          e = ue8m0_exponent(s);
          scale = pow2_from_biased(e);
        }
        // 4. quantize: divide by the scale, round, saturate
        uint8_t* qg = qb + r * H + g * G;
        for (int64_t i = 0; i < G; ++i) {
          const float y = v[i] / scale;
          const float yb = quot_ulps == 0 ? y : quotient_bound(v[i], scale, quot_ulps);
          qg[i] = out_dtype == OUT_E4M3 ? e4m3_encode(yb) : static_cast<uint8_t>(int8_encode(yb));
        }
        // 5. scale store
        if (scale_fmt == FMT_UE8M0_PACKED) {
          exps[g % 4] = e;
          if (g % 4 == 3 || g == ng - 1) {
            uint32_t word = 0;
            for (int64_t j = 0; j <= g % 4; ++j) word |= static_cast<uint32_t>(exps[j]) << (8 * j);
            sp[scale_index(sg, scale_layout, r, g / 4)] = word;
          }
        } else {
          sf[scale_index(sg, scale_layout, r, g)] = scale;
        }
      }
    }

    if (!masked) {
      // Flat scheduler: rows past the live tokens are zero-filled in out_q
      // ([vllm#41326, "Implementation breakdown" item 4]) and in the scales, up
      // to the layout's padded row extent.
      for (int64_t r = live; r < rows; ++r)
        for (int64_t c = 0; c < H; ++c) qb[r * H + c] = 0;
      const int64_t srows = scale_layout == LAYOUT_ROW ? sg.rows : sg.mn_pad;
      for (int64_t r = live; r < srows; ++r)
        for (int64_t c = 0; c < sg.ncol; ++c) {
          if (scale_fmt == FMT_UE8M0_PACKED) sp[scale_index(sg, scale_layout, r, c)] = 0;
          else sf[scale_index(sg, scale_layout, r, c)] = 0.0f;
        }
    }
  }
  return 0;
}

int oracle_quant(const uint16_t* x, int in_dtype, int64_t n, int64_t tokens_pad, int64_t hidden,
                 int group_size, uint8_t* out_q, int out_dtype, void* out_s, int scale_fmt,
                 int scale_layout, int fuse_silu, const int32_t* masked_m, float eps, int flags) {
  return quant_impl(x, in_dtype, n, tokens_pad, hidden, group_size, out_q, out_dtype, out_s,
                    scale_fmt, scale_layout, fuse_silu, masked_m, eps, flags, 0);
}

// oracle_quant with each code taken from a quotient bound (quot_ulps != 0).
int oracle_quant_quotient_bound(const uint16_t* x, int in_dtype, int64_t n, int64_t tokens_pad,
                                int64_t hidden, int group_size, uint8_t* out_q, int out_dtype,
                                void* out_s, int scale_fmt, int scale_layout, int fuse_silu,
                                const int32_t* masked_m, float eps, int flags, int quot_ulps) {
  return quant_impl(x, in_dtype, n, tokens_pad, hidden, group_size, out_q, out_dtype, out_s,
                    scale_fmt, scale_layout, fuse_silu, masked_m, eps, flags, quot_ulps);
}

// Per-token (whole-row) FP8 quantization ([sglang#34257], "Key source snippets": the
// warp kernel).  For each of the first num_tokens rows:
//   s   = max_i |x_i| / 448                  (no eps floor)
//   inv = s == 0 ? 0 : 1 / s                 (an all-zero row gets scale 0, codes 0)
//   q_i = e4m3(max(min(x_i * inv, 448), -448))  (multiplication by the reciprocal; the
//                                               page's clamp, min first, then max)
// out_s[r] = s.  min and max are IEEE minNum / maxNum (std::fmin / std::fmax, which
// CUDA's fminf / fmaxf also are): a NaN operand yields the other one.  So when 1/s
// overflows to +inf (a row whose largest magnitude is below about 1.3e-36), a zero
// element's product 0 * inf = NaN clamps to +448, and every other element to +-448.  Rows of out_q / out_s past num_tokens are not touched (the padded
// output contract of the same page).  in_dtype: 0 bf16, 1 fp16, 2 fp32.
int oracle_per_token_quant(const void* x, int in_dtype, int64_t num_tokens, int64_t hidden,
                           uint8_t* out_q, float* out_s) {
  if (in_dtype < 0 || in_dtype > 2 || num_tokens < 0 || hidden <= 0) return -1;
  for (int64_t r = 0; r < num_tokens; ++r) {
    auto val = [&](int64_t i) -> float {
      const int64_t k = r * hidden + i;
      if (in_dtype == 2) return static_cast<const float*>(x)[k];
      return load_elem(static_cast<const uint16_t*>(x) + k, in_dtype);
    };
    float m = 0.0f;
    for (int64_t i = 0; i < hidden; ++i) m = std::fmax(m, std::fabs(val(i)));
    const float s = m / 448.0f;
    const float inv = s == 0.0f ? 0.0f : 1.0f / s;
    for (int64_t i = 0; i < hidden; ++i) {
      float y = val(i) * inv;
      y = std::fmax(std::fmin(y, 448.0f), -448.0f);
      out_q[r * hidden + i] = e4m3_encode(y);
    }
    out_s[r] = s;
  }
  return 0;
}

// Per-token-group FP8 -> per-tensor FP8 requantization over the masked EP-MoE layout
// ([sglang#35593], "Key source snippets": the requant kernel).  x holds e4m3 codes
// [E, M, K]; x_scale[e, m, k / group] (strides in elements) is the per-token-group scale;
// for rows m < clamp(masked_m[e], 0, M):
//   out = e4m3_satfinite((decode(x) * x_scale) * (1 / output_scale))
// Rows past masked_m are not touched.
int oracle_requant_per_tensor(const uint8_t* x, const float* x_scale, int64_t stride_e,
                              int64_t stride_m, int64_t stride_g, const int32_t* masked_m,
                              float output_scale, uint8_t* out, int64_t E, int64_t M, int64_t K,
                              int group_size) {
  if (E < 0 || M < 0 || K <= 0 || group_size <= 0 || K % group_size != 0) return -1;
  const float inv = 1.0f / output_scale;
  for (int64_t e = 0; e < E; ++e) {
    int64_t live = masked_m[e];
    if (live < 0) live = 0;
    if (live > M) live = M;
    for (int64_t m = 0; m < live; ++m)
      for (int64_t k = 0; k < K; ++k) {
        const int64_t i = (e * M + m) * K + k;
        const float sc = x_scale[e * stride_e + m * stride_m + (k / group_size) * stride_g];
        const float y = (e4m3_decode(x[i]) * sc) * inv;
        out[i] = e4m3_encode(y);
      }
  }
  return 0;
}

}  // extern "C"
