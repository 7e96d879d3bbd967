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
#include <cuda_fp16.h>
#endif

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

// silu(g) = g / (1 + exp(-g)) with the binary32 step sequence E = RN(exp(-g)),
// D = RN(1 + E), S = RN(g / D) (sglang PR #30924, "Implementation breakdown" item 1: the
// fused silu_and_mul trait), for an fp16 gate g given by its bits h, read from the
// precomputed table of binary32 results: entry |h| for a positive gate, pos + |h| for a
// negative one.  The table holds every non-trivial result.  Positive gates from |h| = pos
// on (g >= 16.64) have S = g, since E is below half an ulp of 1.  Negative gates end at
// entry entries - 1 (g = -88.75, from which on exp(-g) overflows binary32), whose value is
// the -0 of every gate beyond, so the clamp of the index returns it.  Every index lies
// inside the table for any 16-bit h.  (silu_f16_index2 and silu_f16_pick below.)
// Both gates of a 32-bit word at once: the table index of each 16-bit half (|h|, plus pos
// for a negative gate) clamped to entries - 1 with one min.u16x2.  No carry crosses the
// halves, since |h| + pos < 2^16.
__device__ __forceinline__ uint32_t silu_f16_index2(uint32_t w, uint32_t pos, uint32_t entries) {
  uint32_t idx = (w & 0x7FFF7FFFu) + ((w >> 15) & 0x00010001u) * pos;
  asm("min.u16x2 %0, %0, %1;" : "+r"(idx) : "r"((entries - 1u) * 0x00010001u));
  return idx;
}
// The result for gate bits h from its table entry tv: g itself for 0 <= g with |h| >= pos.
__device__ __forceinline__ float silu_f16_pick(uint32_t h, float tv, uint32_t pos) {
  const float g = __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
  return h - pos < 0x8000u - pos ? g : tv;
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

// 2^(127 - e), the exact reciprocal of the UE8M0 scale 2^(e - 127), for 1 <= e <= 254.
// (e = 255 comes only from an infinite amax, whose scale 2^128 is +inf in binary32; the
// kernel multiplies such groups by 0 instead, which equals v / +inf for every v, or takes
// IEEE division.)
PTGQ_HD float ue8m0_inverse(uint32_t e) { return u2f((254u - e) << 23); }

}  // namespace ptgq
