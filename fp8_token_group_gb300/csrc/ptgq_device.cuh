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

__device__ __forceinline__ void st_128(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ uint32_t redux_max(uint32_t v, uint32_t mask) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(mask));
  return r;
}
__device__ __forceinline__ uint32_t redux_or(uint32_t v, uint32_t mask) {
  uint32_t r;
  asm volatile("redux.sync.or.b32 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(mask));
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

// Exclusive prefix sum over clamp(masked_m[e], 0, rows), e < n, into prefix[0..n].
__device__ __forceinline__ void masked_prefix(const int32_t* __restrict__ masked_m, int64_t n,
                                              int64_t rows, int32_t* prefix) {
  __shared__ int32_t warp_tot[kWarps];
  const int tid = threadIdx.x;
  const int chunk = static_cast<int>((n + kThreads - 1) / kThreads);
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
  if (tid == kThreads - 1) prefix[n] = base + incl;
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

}  // namespace ptgq
