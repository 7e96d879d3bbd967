// ptgq_device.cuh -- device helpers shared by the quantization kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "ptgq_internal.h"
#include "ptgq_math.cuh"

namespace ptgq {

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 16 elements of 16 bits (32 bytes), as eight 32-bit words.
struct Raw16 { uint32_t w[8]; };

__device__ __forceinline__ void ld_stream_256(Raw16& v, const void* p) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]),
                 "=r"(v.w[5]), "=r"(v.w[6]), "=r"(v.w[7])
               : "l"(p));
}

// Brings the line holding p into L2 (no register result; the address must be valid).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void st_128(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// Predicated stores: the predicate guards the instruction itself, so no branch (and no
// reconvergence) is generated around them.
__device__ __forceinline__ void st_128_if(bool pred, void* p, uint32_t a, uint32_t b, uint32_t c,
                                          uint32_t d) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t"
      "@q st.global.v4.b32 [%0], {%1,%2,%3,%4};\n\t}" ::"l"(p),
      "r"(a), "r"(b), "r"(c), "r"(d), "r"(static_cast<uint32_t>(pred))
      : "memory");
}
__device__ __forceinline__ void st_32_if(bool pred, void* p, uint32_t v) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q st.global.b32 [%0], %1;\n\t}" ::"l"(p),
      "r"(v), "r"(static_cast<uint32_t>(pred))
      : "memory");
}

// Warp-wide unsigned max (callers pass the full mask).
__device__ __forceinline__ uint32_t redux_max(uint32_t v, uint32_t mask) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(mask));
  return r;
}

template <bool kFp16>
__device__ __forceinline__ float widen_lo(uint32_t w) {
  if constexpr (kFp16) return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
  else return u2f(w << 16);
}
template <bool kFp16>
__device__ __forceinline__ float widen_hi(uint32_t w) {
  if constexpr (kFp16) return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
  else return u2f(w & 0xFFFF0000u);
}

// Four e4m3 codes, memory order a, b, c, d (cvt puts its first source in the high byte).
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// Four int8 codes.  Adding 1.5 * 2^23 rounds |y| < 2^22 to the nearest integer,
// ties to even, and leaves it in the low bits; |y| <= 127 here, so the low byte is
// the two's-complement code and no clamp is needed.
__device__ __forceinline__ uint32_t s8x4(float a, float b, float c, float d) {
  const float kMagic = 12582912.0f;
  const uint32_t ia = f2u(__fadd_rn(a, kMagic)), ib = f2u(__fadd_rn(b, kMagic));
  const uint32_t ic = f2u(__fadd_rn(c, kMagic)), id = f2u(__fadd_rn(d, kMagic));
  const uint32_t lo = __byte_perm(ia, ib, 0x0040u);
  const uint32_t hi = __byte_perm(ic, id, 0x0040u);
  return __byte_perm(lo, hi, 0x5410u);
}

// n / d for n < 2^32 with magic = floor(2^32 / d): the estimate is at most one low.
__device__ __forceinline__ uint32_t udiv(uint32_t n, uint32_t d, uint32_t magic) {
  uint32_t q = __umulhi(n, magic);
  if (n - q * d >= d) ++q;
  return q;
}

// Exclusive prefix sum over clamp(masked_m[e], 0, rows), e < n, into prefix[0..n], by a
// CTA of kT threads.
template <int kT = kThreads>
__device__ __forceinline__ void masked_prefix(const int32_t* __restrict__ masked_m, int64_t n,
                                              int64_t rows, int32_t* prefix) {
  __shared__ int32_t warp_tot[kT / 32];
  const int tid = threadIdx.x;
  const int chunk = static_cast<int>((n + kT - 1) / kT);
  const int lo = tid * chunk;
  const int hi = min(lo + chunk, static_cast<int>(n));
  int32_t local = 0;
  for (int e = lo; e < hi; ++e) {
    const int32_t m = masked_m[e];
    local += m < 0 ? 0 : (m > rows ? static_cast<int32_t>(rows) : m);
  }
  const int lane = tid & 31, warp = tid >> 5;
  int32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int32_t base = 0;
  for (int w = 0; w < warp; ++w) base += warp_tot[w];
  int32_t run = base + incl - local;
  for (int e = lo; e < hi; ++e) {
    prefix[e] = run;
    const int32_t m = masked_m[e];
    run += m < 0 ? 0 : (m > rows ? static_cast<int32_t>(rows) : m);
  }
  if (tid == kT - 1) prefix[n] = base + incl;
}

// Rows-to-expert buckets for the masked scheduler: bucket[b] is the expert of live row
// min(b << shift, live - 1) for b = 0..kBuckets, with shift the smallest value that maps
// every live row to a bucket below kBuckets.  A lookup then searches only between two
// neighbouring buckets' experts (usually zero or one step) instead of over all experts.
__device__ __forceinline__ int expert_in(const int32_t* prefix, int lo, int hi, uint32_t R) {
  // largest e in [lo, hi] with prefix[e] <= R
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<uint32_t>(prefix[mid]) <= R) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ uint32_t bucket_shift(uint32_t live) {
  const uint32_t top = live > 0u ? live - 1u : 0u;
  const int bits = 32 - __clz(top);                 // bits needed for the largest row
  return bits > 8 ? static_cast<uint32_t>(bits - 8) : 0u;
}

template <int kT = kThreads>
__device__ __forceinline__ void build_buckets(const int32_t* prefix, int n, uint32_t live,
                                              uint32_t shift, int32_t* bucket) {
  for (int b = threadIdx.x; b <= kBuckets; b += kT) {
    const uint32_t r0 = min(static_cast<uint32_t>(b) << shift, live > 0u ? live - 1u : 0u);
    bucket[b] = expert_in(prefix, 0, n - 1, r0);
  }
}

// Largest e in [0, n) with prefix[e] <= R (an expert that owns live row R).
__device__ __forceinline__ int expert_of(const int32_t* prefix, int n, uint32_t R) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<uint32_t>(prefix[mid]) <= R) lo = mid;
    else hi = mid;
  }
  return lo;
}

// ---- packed helpers -------------------------------------------------------------

// max(|a|, |b|) per 16-bit half (the xorsign variant; callers clear the sign bits).
template <bool kFp16>
__device__ __forceinline__ uint32_t maxabs2(uint32_t a, uint32_t b) {
  uint32_t r;
  if constexpr (kFp16) asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  else asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Two binary32 values in one 64-bit register pair, for the sm_100+ f32x2 instructions.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0,%1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// Rounded toward -inf: an exact zero result is -0 (see div2_by_scale).
__device__ __forceinline__ uint64_t fma2_rm(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rm.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// A pair of 16-bit elements widened to binary32 (exact), as an f32x2 pair.
template <bool kFp16>
__device__ __forceinline__ uint64_t widen2(uint32_t w) {
  return pk2(widen_lo<kFp16>(w), widen_hi<kFp16>(w));
}

// Two e4m3 codes (low byte = lo) from an f32x2 pair.
__device__ __forceinline__ uint32_t e4m3x2_pair(uint64_t v) {
  float lo, hi;
  upk2(v, lo, hi);
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(hi), "f"(lo));
  return c;
}

// The pair x / s from r = RN(1/s), ns = -s: q0 = RN(x r), e = RM(x - q0 s) (exact when the
// residual does not underflow; rounding toward -inf only fixes the sign of an exact zero,
// so x = -0 gives -0), q = RN(q0 + e r).  Same 8-bit codes as the IEEE quotient for every
// input with amax >= 1e-24 (checked for every pair of 16-bit values and 1.3e9 sampled
// binary32 pairs); the binary32 quotient itself can differ only below 2^-10, where every
// code is zero.
__device__ __forceinline__ uint64_t div2_by_scale(uint64_t x, uint64_t r, uint64_t ns) {
  const uint64_t q0 = mul2(x, r);
  const uint64_t e = fma2_rm(q0, ns, x);
  return fma2(e, r, q0);
}

// RN(a / d) for the constants d = 448 or 127 with rd = RN(1/d): one exact-residual
// correction gives the IEEE quotient for every positive normal binary32 a >= 2^-103
// (checked exhaustively for both constants).
__device__ __forceinline__ float div_by_const(float a, float d, float rd) {
  const float q0 = __fmul_rn(a, rd);
  const float e = __fmaf_rn(-q0, d, a);
  return __fmaf_rn(e, rd, q0);
}

// Copy `n16` 16-byte chunks of module constants into shared memory with cp.async, by a
// CTA of kT threads: every thread issues all its chunks before waiting, so the copy costs
// one L2 round trip.  The caller synchronizes the block afterwards.
template <int kT = kThreads>
__device__ __forceinline__ void copy_to_smem_async(void* dst, const void* src, int n16) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  const char* s = static_cast<const char*>(src);
  for (int i = threadIdx.x; i < n16; i += kT)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d + 16u * i), "l"(s + 16 * i)
                 : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void copy_to_smem_wait() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Max over the `lg` lanes of a group (lg a power of two <= 8, groups aligned to lg lanes);
// every lane of the group receives it.  Fixed-width butterfly with full-warp shuffles and
// predicated selects, so it compiles to straight-line code for any lg.
__device__ __forceinline__ uint32_t group_max(uint32_t v, uint32_t lg) {
#pragma unroll
  for (uint32_t o = 1; o < 8; o <<= 1) {
    const uint32_t w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = o < lg ? max(v, w) : v;
  }
  return v;
}

// OR of the four groups of a unit (4*lg lanes, aligned): lanes exchange with the lanes of
// the same rank in groups j^1 and j^2, so every lane receives the OR of all four.
__device__ __forceinline__ uint32_t unit_or(uint32_t v, uint32_t lg) {
  v |= __shfl_xor_sync(0xFFFFFFFFu, v, lg);
  v |= __shfl_xor_sync(0xFFFFFFFFu, v, 2u * lg);
  return v;
}

}  // namespace ptgq
