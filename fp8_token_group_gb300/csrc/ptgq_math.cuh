// ptgq_math.cuh -- binary32 element math of the quantizer (device code).
//
// Everything here is plain IEEE binary32 arithmetic with explicit fused
// multiply-adds; the file is compiled with -fmad=false so that no other product
// is fused into a sum.  References:
//   sglang PR #30924 "unify per_token_group_quant into one trait-driven JIT kernel"
//     (prhub summary), "Key source snippets": ref_fp8_ue8m0 (scale, UE8M0 rounding).
//   sglang PR #27449 "JIT port of per_token_group_quant_8bit_v2" (GitHub PR body),
//     "Implementation notes": the division by the scale must be exact (IEEE), a fast
//     approximate division changes scattered codes by one step.
#pragma once

#include <cstdint>
#include <cmath>

#ifdef __CUDACC__
#define PTGQ_HD __host__ __device__ __forceinline__
#else
#define PTGQ_HD inline
#endif

namespace ptgq {

PTGQ_HD float u2f(uint32_t u) {
#ifdef __CUDA_ARCH__
  return __uint_as_float(u);
#else
  float f; __builtin_memcpy(&f, &u, 4); return f;
#endif
}
PTGQ_HD uint32_t f2u(float f) {
#ifdef __CUDA_ARCH__
  return __float_as_uint(f);
#else
  uint32_t u; __builtin_memcpy(&u, &f, 4); return u;
#endif
}

// ---------------------------------------------------------------------------
// exp for 16-bit inputs.
//
// Returns RN(e^x) (correctly rounded binary32) for x a bf16 or fp16 value in
// [-20, 88.72).  Below -20 it returns 0 and from 88.72 it returns +inf; the
// caller only feeds the result into D = RN(1 + E), which is 1 for every E below
// 2^-24 (x < -16.6) and +inf for every E that overflows, so those limits do not
// change D.
//
// Method (Tang-style table reduction, evaluated in double-float):
//   i = rint(x) capped at 88, f = x - i        (exact; |f| <= 0.72)
//   j = rint(128 f),           r = f - j/128   (exact; |r| <= 1/256, <= 11 bits)
//   e^x = e^i * e^(j/128) * (1 + r + r^2/2 + c),  c = r^3/6 + r^4/24 + r^5/120
// e^i and e^(j/128) come from (hi, lo) tables accurate to ~2^-48; r^2 is exact
// because r has at most 11 significant bits; products with the large terms are
// split exactly with fma, and the last partial sum is rounded to odd, so the final
// addition rounds a value within ~2^-45 of e^x once, on the correct side of every
// rounding midpoint.  Checked against 100-bit values for every bf16 and fp16 input.
// ---------------------------------------------------------------------------
PTGQ_HD float exp_from_tables(float x, const float2* exp_int, const float2* exp_frac,
                              int int_min, int frac_jmin) {
  // Clamp into the tables' range; results outside [-20, 88.72) are replaced below.
  const float xc = fminf(fmaxf(x, -20.0f), 88.75f);
  float fi = rintf(xc);
  fi = fminf(fi, 88.0f);
  const float f = xc - fi;
  const float fj = rintf(f * 128.0f);
  const float r = fmaf(fj, -0.0078125f, f);
  const float2 A = exp_int[static_cast<int>(fi) - int_min];
  const float2 B = exp_frac[static_cast<int>(fj) - frac_jmin];
  // T = A * B as an unevaluated sum th + tl
  const float th = A.x * B.x;
  float tl = fmaf(A.x, B.x, -th);
  tl = fmaf(A.x, B.y, tl);
  tl = fmaf(A.y, B.x, tl);
  // series of e^r - 1 = r + h2 + c
  const float h2 = 0.5f * (r * r);
  float c = fmaf(r, 1.0f / 60.0f, 1.0f / 12.0f);
  c = fmaf(r, c, 1.0f / 3.0f);
  c = (h2 * r) * c;
  // th * r and th * h2, each split exactly into a rounded part and its error
  const float m1 = th * r;
  const float m1l = fmaf(th, r, -m1);
  const float m2 = th * h2;
  const float m2l = fmaf(th, h2, -m2);
  // th + m1 + m2 with the rounding errors of both additions kept
  const float s1 = th + m1;
  const float e1 = (th - s1) + m1;
  const float s2 = s1 + m2;
  const float e2 = (s1 - s2) + m2;
  // Everything below e1 (each term < 2^-24 th), then e1 added with round-to-odd:
  // the sticky last bit tells the final rounding on which side of a midpoint the
  // value lies (x = 2^-24 is such a case: e^x = 1 + 2^-24 + 2^-49 + ...).
  float rest = fmaf(th, c, tl);
  rest = fmaf(tl, r, rest);
  rest = rest + (m1l + m2l);
  const float inner = e2 + rest;
  const float w = e1 + inner;
  const float wz = w - e1;
  const float werr = (e1 - (w - wz)) + (inner - wz);
  uint32_t wb = f2u(w);
  if (werr != 0.0f && (wb & 1u) == 0u) wb += ((werr > 0.0f) == (w > 0.0f)) ? 1u : 0xFFFFFFFFu;
  float res = s2 + u2f(wb);
  res = x < -20.0f ? 0.0f : res;
  res = x >= 88.72f ? INFINITY : res;
  return res;
}

// silu(g) = g / (1 + exp(-g)) with the binary32 step sequence E, D = RN(1 + E),
// S = RN(g / D) (sglang PR #30924, "Implementation breakdown" item 1: the fused
// silu_and_mul trait).
PTGQ_HD float silu_generic(float g, const float2* exp_int, const float2* exp_frac, int int_min,
                           int frac_jmin) {
  const float e = exp_from_tables(-g, exp_int, exp_frac, int_min, frac_jmin);
  const float d = 1.0f + e;
  return g / d;
}

// The same sequence for a bf16 gate, read from the precomputed table of binary32
// results for 2^-25 <= |g| < 128; outside that range the sequence has closed
// forms: S = g/2 for |g| < 2^-25 (E = 1, D = 2), S = g for g >= 128 (E = 0) and
// S = -0 for g <= -128 (E = +inf).
PTGQ_HD float silu_bf16(uint32_t h, const float* table, uint32_t field_lo, uint32_t span) {
  const float g = u2f(h << 16);
  const uint32_t mag = h & 0x7FFFu;
  const uint32_t t = mag - (field_lo << 7);     // wraps for small magnitudes
  const bool in_table = t < span;
  const uint32_t idx = ((h >> 15) * span) + (in_table ? t : 0u);
  const float tv = table[idx];
  const float outside = mag < (field_lo << 7) ? g * 0.5f : ((h & 0x8000u) ? -0.0f : g);
  return in_table ? tv : outside;
}

// ---------------------------------------------------------------------------
// Group scale.
// ---------------------------------------------------------------------------

// UE8M0 exponent byte: biased exponent of s, plus one if any mantissa bit is set
// (rounds s up to a power of two; sglang PR #30924, "Key source snippets").
PTGQ_HD uint32_t ue8m0_exponent(float s) {
  const uint32_t b = f2u(s);
  return ((b >> 23) & 0xFFu) + ((b & 0x7FFFFFu) != 0u ? 1u : 0u);
}

// 2^(127 - e), the exact reciprocal of the UE8M0 scale 2^(e - 127) (e <= 253).
PTGQ_HD float ue8m0_inverse(uint32_t e) { return u2f((254u - e) << 23); }

}  // namespace ptgq
