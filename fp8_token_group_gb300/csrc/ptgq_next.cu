// ptgq_next.cu -- the two neighbouring operations of the quantizer (sm_103a):
//
//  * per-token (whole-row) FP8 quantization (sglang PR #34257, "Key source
//    snippets": the per-token warp kernel): s = max|x| / 448 per row, inv = 1/s
//    (0 for an all-zero row), q = e4m3(clamp(x * inv)); rows past num_tokens of a
//    padded output are not touched.
//  * per-token-group FP8 -> per-tensor FP8 requantization over the masked EP-MoE
//    layout (sglang PR #35593, "Key source snippets": the requant kernel):
//    out = e4m3_satfinite((decode(x) * x_scale[group]) * (1 / output_scale)) for rows
//    below masked_m[e]; other rows are not touched.
//
// Both are streaming kernels bound by HBM bandwidth: persistent grids, full-width
// vector loads and stores, PDL.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <map>
#include <tuple>

#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "../../include/ptgq.h"
#include "ptgq_device.cuh"
#include "ptgq_internal.h"

namespace ptgq {

// ---------------------------------------------------------------- per-token quant

struct PerTokenParams {
  const void* x;
  uint8_t* q;
  float* s;
  int64_t tokens;
  int64_t hidden;
};

// Running max |x| of a row.  binary32: the magnitude bit patterns.  16-bit inputs: both
// halves of a word at once (max.xorsign.abs; the sign bits it leaves are cleared by
// abs_bits), which gives the same magnitudes as comparing the patterns.
template <int kIn>
__device__ __forceinline__ uint32_t absmax_words(uint32_t m, const uint32_t* w, int n) {
  for (int k = 0; k < n; ++k) {
    if constexpr (kIn == 2) m = max(m, w[k] & 0x7FFFFFFFu);
    else m = maxabs2<kIn == 1>(m, w[k]);
  }
  return m;
}

// The row's max |x| as binary32 bits, from the running value of absmax_words.
template <int kIn>
__device__ __forceinline__ uint32_t abs_bits(uint32_t m) {
  if constexpr (kIn == 2) {
    return m;
  } else {
    m &= 0x7FFF7FFFu;
    const uint32_t h = max(m & 0xFFFFu, m >> 16);
    return f2u(kIn == 1 ? widen_lo<true>(h) : widen_lo<false>(h));
  }
}

// 16 bytes of input (8 16-bit or 4 binary32 elements) -> codes, stored at dst.
// Products x * inv are formed two at a time (mul.rn.f32x2: each rounded like __fmul_rn).
template <int kIn>
__device__ __forceinline__ void quantize16(const uint32_t (&w)[4], float inv, uint8_t* dst) {
  const uint64_t inv2 = pk2(inv, inv);
  if constexpr (kIn == 2) {
    const uint32_t o = e4m3x2_pair(mul2(pk2(u2f(w[0]), u2f(w[1])), inv2)) |
                       (e4m3x2_pair(mul2(pk2(u2f(w[2]), u2f(w[3])), inv2)) << 16);
    asm volatile("st.global.b32 [%0], %1;" ::"l"(dst), "r"(o) : "memory");
  } else {
    constexpr bool h = kIn == 1;
    const uint32_t o0 = e4m3x2_pair(mul2(widen2<h>(w[0]), inv2)) |
                        (e4m3x2_pair(mul2(widen2<h>(w[1]), inv2)) << 16);
    const uint32_t o1 = e4m3x2_pair(mul2(widen2<h>(w[2]), inv2)) |
                        (e4m3x2_pair(mul2(widen2<h>(w[3]), inv2)) << 16);
    asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(dst), "r"(o0), "r"(o1) : "memory");
  }
}

// The same for a row whose reciprocal scale or scale is infinite (a row maximum below about
// 1.3e-36, where 1/s overflows, or an infinite element): the products, which can be NaN
// (0 * inf) or infinite there, go through the page's clamp, max(min(y, 448), -448) with
// IEEE minNum / maxNum (NaN yields the other operand), before the conversion.
template <int kIn>
__device__ __forceinline__ void quantize16_clamped(const uint32_t (&w)[4], float inv, uint8_t* dst) {
  auto q = [&](float xv) { return fmaxf(fminf(__fmul_rn(xv, inv), 448.0f), -448.0f); };
  if constexpr (kIn == 2) {
    const uint32_t o = e4m3x4(q(u2f(w[0])), q(u2f(w[1])), q(u2f(w[2])), q(u2f(w[3])));
    asm volatile("st.global.b32 [%0], %1;" ::"l"(dst), "r"(o) : "memory");
  } else {
    constexpr bool h = kIn == 1;
    const uint32_t o0 = e4m3x4(q(widen_lo<h>(w[0])), q(widen_hi<h>(w[0])), q(widen_lo<h>(w[1])),
                               q(widen_hi<h>(w[1])));
    const uint32_t o1 = e4m3x4(q(widen_lo<h>(w[2])), q(widen_hi<h>(w[2])), q(widen_lo<h>(w[3])),
                               q(widen_hi<h>(w[3])));
    asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(dst), "r"(o0), "r"(o1) : "memory");
  }
}

// Whether a row takes quantize16_clamped (uniform over the warp that owns the row).
__device__ __forceinline__ bool row_needs_clamp(float s, float inv) {
  return fabsf(inv) == INFINITY || fabsf(s) == INFINITY;
}

// The warp's first row goes to L2 before the dependency wait, one 128-byte line per lane
// at a time.  A prefetch reads no value and L2 is the point of coherence for device memory,
// so whatever the previous kernel writes to x, the copies after the wait see it; when x was
// not written by that kernel, the first DRAM round trip of this call overlaps its tail
// (bf16 [4096, 4096], back to back: 9.35 -> 7.90 us).
__device__ __forceinline__ void prefetch_first_row(const PerTokenParams& p, int64_t row,
                                                   int esize, int lane) {
  if (row >= p.tokens) return;
  const int64_t rb = p.hidden * esize;
  const char* r = static_cast<const char*>(p.x) + row * rb;
  for (int64_t o = static_cast<int64_t>(lane) * 128; o < rb; o += 32 * 128) prefetch_l2(r + o);
}

// Rows staged in shared memory.  A warp owns one row at a time and kPtBufs row buffers:
// 2 when it takes several rows (the copy of its next row, cp.async with 16 bytes per lane
// per instruction, is in flight while it reduces and quantizes the current one), 1 when
// every warp takes at most one row.  Each row is read from HBM once.  A lane copies and
// later reads only its own 16-byte chunks, so the only cross-lane step is the max
// reduction.  Rows must be a multiple of 16 bytes; the launcher picks the CTA size (1 to 8
// warps) and the buffer count (per_token_shape).
template <int kIn, int kPtBufs>
__global__ void __launch_bounds__(kThreads) per_token_smem_kernel(const PerTokenParams p) {
  extern __shared__ __align__(16) unsigned char rowbuf[];
  constexpr int kEsize = kIn == 2 ? 4 : 2;
  constexpr int kPer16 = 16 / kEsize;                       // elements per 16-byte chunk
  const int warps = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  prefetch_first_row(p, static_cast<int64_t>(blockIdx.x) * warps + warp, kEsize, lane);
  griddep_wait();
  griddep_launch_dependents();
  const int64_t chunks = p.hidden / kPer16;
  const int64_t row_bytes = chunks * 16;
  const uint32_t buf0 = static_cast<uint32_t>(__cvta_generic_to_shared(rowbuf)) +
                        static_cast<uint32_t>(warp * kPtBufs * row_bytes);
  const int64_t W = static_cast<int64_t>(gridDim.x) * warps;
  const char* xb = static_cast<const char*>(p.x);

  auto issue = [&](int64_t row, int slot) {
    if (row < p.tokens) {
      const char* src = xb + row * row_bytes;
      const uint32_t dst = buf0 + static_cast<uint32_t>(slot * row_bytes);
      for (int64_t c = lane; c < chunks; c += 32)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + 16u * static_cast<uint32_t>(c)),
                     "l"(src + 16 * c) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  auto chunk = [&](int slot, int64_t c, uint32_t (&w)[4]) {
    const uint32_t a = buf0 + static_cast<uint32_t>(slot * row_bytes + 16 * c);
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(a) : "memory");
  };

  int64_t row = static_cast<int64_t>(blockIdx.x) * warps + warp;
#pragma unroll
  for (int b = 0; b < kPtBufs; ++b) issue(row + b * W, b);
  for (int slot = 0; row < p.tokens; row += W, slot = slot + 1 == kPtBufs ? 0 : slot + 1) {
    // all but the kPtBufs-1 most recent groups are complete: this row's copies are done
    asm volatile("cp.async.wait_group %0;" ::"n"(kPtBufs - 1) : "memory");
    uint32_t m = 0u;
    for (int64_t c = lane; c < chunks; c += 32) {
      uint32_t w[4];
      chunk(slot, c, w);
      m = absmax_words<kIn>(m, w, 4);
    }
    m = redux_max(abs_bits<kIn>(m), 0xFFFFFFFFu);
    const float s = __fdiv_rn(u2f(m), 448.0f);
    const float inv = s == 0.0f ? 0.0f : __frcp_rn(s);
    uint8_t* qrow = p.q + row * p.hidden;
    if (!row_needs_clamp(s, inv)) {
      for (int64_t c = lane; c < chunks; c += 32) {
        uint32_t w[4];
        chunk(slot, c, w);
        quantize16<kIn>(w, inv, qrow + c * kPer16);
      }
    } else {
      for (int64_t c = lane; c < chunks; c += 32) {
        uint32_t w[4];
        chunk(slot, c, w);
        quantize16_clamped<kIn>(w, inv, qrow + c * kPer16);
      }
    }
    if (lane == 0) p.s[row] = s;
    issue(row + kPtBufs * W, slot);                        // refill this buffer
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// One CTA per row, for calls with few rows (the pages' per-token CTA variant, sglang PR
// #34257, "Key source snippets": chosen below 16 x SMs rows).  With one warp per row, a call
// of a few hundred rows leaves most of the GPU idle and each warp moves its whole row by
// itself; here the CTA's kT / 32 warps (8, or 4 for calls of a little more rows) split the
// row, the row max is combined through shared
// memory, and the first kCache 16-byte chunks of each thread stay in registers between the
// max pass and the quantize pass (the rest are read again, from L2).  Rows must be a
// multiple of 16 bytes and 16-byte aligned.  The CTA's first row goes to L2 before the
// dependency wait.  The arithmetic is that of the other per-token kernels.
template <int kIn, int kT>
__global__ void __launch_bounds__(kT) per_token_cta_kernel(const PerTokenParams p) {
  constexpr int kEsize = kIn == 2 ? 4 : 2;
  constexpr int kPer16 = 16 / kEsize;
  constexpr int kCache = 4;
  constexpr int kW = kT / 32;
  __shared__ uint32_t wmax[2][kW];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t chunks = p.hidden / kPer16;
  const int64_t row_bytes = chunks * 16;
  const char* xb = static_cast<const char*>(p.x);
  if (blockIdx.x < p.tokens) {
    const char* r = xb + static_cast<int64_t>(blockIdx.x) * row_bytes;
    for (int64_t o = static_cast<int64_t>(tid) * 128; o < row_bytes; o += kT * 128)
      prefetch_l2(r + o);
  }
  griddep_wait();
  griddep_launch_dependents();
  auto load = [&](const char* src, int64_t c, uint32_t (&w)[4]) {
    asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "l"(src + 16 * c));
  };
  int par = 0;
  for (int64_t row = blockIdx.x; row < p.tokens; row += gridDim.x, par ^= 1) {
    const char* src = xb + row * row_bytes;
    uint32_t cache[kCache][4];
    uint32_t m = 0u;
#pragma unroll
    for (int j = 0; j < kCache; ++j) {
      const int64_t c = tid + static_cast<int64_t>(j) * kT;
      if (c < chunks) {
        load(src, c, cache[j]);
        m = absmax_words<kIn>(m, cache[j], 4);
      }
    }
    for (int64_t c = tid + static_cast<int64_t>(kCache) * kT; c < chunks; c += kT) {
      uint32_t w[4];
      load(src, c, w);
      m = absmax_words<kIn>(m, w, 4);
    }
    m = redux_max(abs_bits<kIn>(m), 0xFFFFFFFFu);
    // Two slots, alternating by row: a warp writes the next row's slot only after the next
    // barrier, which every warp reaches only after reading this row's slot.
    if (lane == 0) wmax[par][warp] = m;
    __syncthreads();
    uint32_t mm = 0u;
#pragma unroll
    for (int w = 0; w < kW; ++w) mm = max(mm, wmax[par][w]);
    const float s = __fdiv_rn(u2f(mm), 448.0f);
    const float inv = s == 0.0f ? 0.0f : __frcp_rn(s);
    const bool clamp = row_needs_clamp(s, inv);
    uint8_t* qrow = p.q + row * p.hidden;
#pragma unroll
    for (int j = 0; j < kCache; ++j) {
      const int64_t c = tid + static_cast<int64_t>(j) * kT;
      if (c < chunks) {
        if (clamp) quantize16_clamped<kIn>(cache[j], inv, qrow + c * kPer16);
        else quantize16<kIn>(cache[j], inv, qrow + c * kPer16);
      }
    }
    for (int64_t c = tid + static_cast<int64_t>(kCache) * kT; c < chunks; c += kT) {
      uint32_t w[4];
      load(src, c, w);
      if (clamp) quantize16_clamped<kIn>(w, inv, qrow + c * kPer16);
      else quantize16<kIn>(w, inv, qrow + c * kPer16);
    }
    if (tid == 0) p.s[row] = s;
  }
}

// Rows in registers (for rows the staged kernel does not take: lengths that are not a
// multiple of 16 bytes, or too long for two shared buffers per warp).  One warp per row;
// the first kCache vectors of each lane stay in registers between the max pass and the
// quantize pass, the rest are read again (from L2).  kVecBytes: 16, or 8 for 16-bit rows
// whose length is only a multiple of 4.
template <int kIn, int kVecBytes>
__global__ void __launch_bounds__(kThreads) per_token_reg_kernel(const PerTokenParams p) {
  constexpr int kElems = kIn == 2 ? kVecBytes / 4 : kVecBytes / 2;
  constexpr int kWords = kVecBytes / 4;
  constexpr int kCache = 8;
  const int lane = threadIdx.x & 31;
  prefetch_first_row(p, static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5),
                     kIn == 2 ? 4 : 2, lane);
  griddep_wait();
  griddep_launch_dependents();
  const int64_t warps = static_cast<int64_t>(gridDim.x) * kWarps;
  const int64_t nvec = p.hidden / kElems;
  const char* xb = static_cast<const char*>(p.x);

  auto load = [&](int64_t row, int64_t i, uint32_t (&w)[kWords]) {
    const char* ptr = xb + (row * p.hidden + i * kElems) * (kIn == 2 ? 4 : 2);
    if constexpr (kVecBytes == 16) {
      asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "l"(ptr));
    } else {
      asm volatile("ld.global.nc.v2.b32 {%0,%1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "l"(ptr));
    }
  };
  // clamp: the row takes the page's clamp before the conversion (row_needs_clamp)
  auto quantize_store = [&](int64_t row, int64_t i, const uint32_t (&w)[kWords], float inv,
                            bool clamp) {
    uint8_t* dst = p.q + row * p.hidden + i * kElems;
    if constexpr (kVecBytes == 16) {
      if (clamp) quantize16_clamped<kIn>(w, inv, dst);
      else quantize16<kIn>(w, inv, dst);
    } else {       // 16-bit, 4 elements
      constexpr bool h = kIn == 1;
      auto q = [&](float xv) {
        const float y = __fmul_rn(xv, inv);
        return clamp ? fmaxf(fminf(y, 448.0f), -448.0f) : y;
      };
      const uint32_t o = e4m3x4(q(widen_lo<h>(w[0])), q(widen_hi<h>(w[0])), q(widen_lo<h>(w[1])),
                                q(widen_hi<h>(w[1])));
      asm volatile("st.global.b32 [%0], %1;" ::"l"(dst), "r"(o) : "memory");
    }
  };

  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
       row < p.tokens; row += warps) {
    uint32_t cache[kCache][kWords];
    uint32_t m = 0u;
#pragma unroll
    for (int j = 0; j < kCache; ++j) {
      const int64_t i = lane + 32 * j;
      if (i < nvec) {
        load(row, i, cache[j]);
        m = absmax_words<kIn>(m, cache[j], kWords);
      }
    }
    for (int64_t i = lane + 32 * kCache; i < nvec; i += 32) {
      uint32_t w[kWords];
      load(row, i, w);
      m = absmax_words<kIn>(m, w, kWords);
    }
    m = redux_max(abs_bits<kIn>(m), 0xFFFFFFFFu);
    const float s = __fdiv_rn(u2f(m), 448.0f);
    const float inv = s == 0.0f ? 0.0f : __frcp_rn(s);
    const bool clamp = row_needs_clamp(s, inv);
#pragma unroll
    for (int j = 0; j < kCache; ++j) {
      const int64_t i = lane + 32 * j;
      if (i < nvec) quantize_store(row, i, cache[j], inv, clamp);
    }
    for (int64_t i = lane + 32 * kCache; i < nvec; i += 32) {
      uint32_t w[kWords];
      load(row, i, w);
      quantize_store(row, i, w, inv, clamp);
    }
    if (lane == 0) p.s[row] = s;
  }
}

// ---------------------------------------------------------------- requant

struct RequantParams {
  const uint8_t* x;
  const float* x_scale;
  const int32_t* masked_m;       // nullptr: every row is live
  const float* output_scale;     // device scalar
  uint8_t* out;
  uint32_t experts;              // E
  uint32_t m;                    // rows per expert
  int64_t k;                     // row length (codes)
  int64_t se, sm, sg;            // x_scale strides (elements)
  uint32_t cpr;                  // lane chunks per row: k / kV
  uint32_t cpr_magic;            // floor(2^32 / cpr), or 0xFFFFFFFF when cpr == 1
  uint32_t e_magic;              // floor(2^32 / E), or 0xFFFFFFFF when E == 1
  uint32_t g_log2;               // log2(group size)
};

// CTAs of 8 warps per SM (the grid is at most this many per SM): with the speculative
// prefetch below, a wave of three reaches only rows that are live in the page's shape (8
// experts, 128 of 1024 rows live: 2.77 us, against 3.03 us with four CTAs per SM, whose
// first wave also prefetches dead rows, and 3.29 us with four and no prefetch).
constexpr int kRequantBlocksPerSm = 3;

// Requantizes kV codes (kV = 32, or 16 when k is not a multiple of 32) of one row per lane.
//
// Row slots are numbered row-major over (row, expert): slot S = r * E + e, so the rows most
// likely to be live -- the first rows of every expert -- come first, and every live row lies
// below max_e masked_m[e] * E slots.  A warp task is 32 consecutive lane chunks of that
// numbering (a row of expert e is contiguous in x, so a task is at most a few contiguous
// runs).  Each warp reads masked_m itself (one word per lane for E <= 32) and takes the
// maximum with redux.sync, which bounds its task loop; a lane then knows whether its chunk
// is live from masked_m[e] (a shuffle for E <= 32, else an L1-cached load).  Dead chunks
// are not written, and past the first task not read either: a warp's first task is loaded
// speculatively, in flight with the read of masked_m, so no dependent round trip stands
// before it (no prefix sum, no block barrier, no search for the expert).  Batches of two
// tasks are loaded, then computed, when a warp has more than one task.
template <int kV>
__global__ void __launch_bounds__(kThreads, kRequantBlocksPerSm) requant_kernel(const RequantParams p) {
  constexpr int kWords = kV / 4;
  const uint32_t lane = threadIdx.x & 31u;
  // Speculative prefetch, before the dependency wait: this lane's chunk of the warp's first
  // task, as if every row were live, goes to L2 while the previous kernel finishes and
  // masked_m and the output scale are read, so the row loads that follow mostly hit L2
  // instead of waiting for a second DRAM round trip; the chunk's group scale goes with it
  // (2.55 -> 2.46 us).  A prefetch reads no value and L2 is the point of coherence, so it
  // is correct whatever the previous kernel writes (2.81 -> 2.53 us with the prefetch ahead
  // of the wait rather than after it).  Slots are
  // numbered rows first, so the first wave covers the first rows of every expert, which
  // are the live ones unless an expert has fewer live rows than the wave reaches; a
  // prefetch of a dead row only costs a wasted read (at most 32 bytes per lane of the
  // first wave: 2.5 MB on 152 SMs).  Every prefetched address lies inside x and x_scale
  // (e < E, r < m, g < k / group).
  {
    const uint32_t c0 = ((blockIdx.x * kWarps + (threadIdx.x >> 5)) << 5) + lane;
    const uint32_t S0 = udiv(c0, p.cpr, p.cpr_magic);
    const uint32_t r0 = udiv(S0, p.experts, p.e_magic);
    if (r0 < p.m) {
      const uint32_t e0 = S0 - r0 * p.experts;
      const uint32_t col0 = c0 - S0 * p.cpr;
      prefetch_l2(p.x + (static_cast<int64_t>(e0) * p.m + r0) * p.k +
                  static_cast<int64_t>(col0) * kV);
      const uint32_t g0 = static_cast<uint32_t>((static_cast<uint64_t>(col0) * kV) >> p.g_log2);
      prefetch_l2(p.x_scale + static_cast<int64_t>(e0) * p.se + static_cast<int64_t>(r0) * p.sm +
                  static_cast<int64_t>(g0) * p.sg);
    }
  }
  griddep_wait();
  griddep_launch_dependents();
  const bool masked = p.masked_m != nullptr;
  const uint32_t warp_id = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const uint32_t stride = gridDim.x * kWarps;

  struct Chunk {
    int64_t off;           // byte offset of the chunk in x and out
    float sc0, sc1;        // group scale(s): two when a chunk spans two groups (G = 16, kV = 32)
    bool live;
    uint32_t w[kWords];
  };

  auto load = [&](Chunk& ch, uint32_t e, uint32_t r, uint32_t col) {
    const uint8_t* src = p.x + ch.off;
    if constexpr (kV == 32) {
      asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                   : "=r"(ch.w[0]), "=r"(ch.w[1]), "=r"(ch.w[2]), "=r"(ch.w[3]), "=r"(ch.w[4]),
                     "=r"(ch.w[5]), "=r"(ch.w[6]), "=r"(ch.w[7])
                   : "l"(src));
    } else {
      asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(ch.w[0]), "=r"(ch.w[1]), "=r"(ch.w[2]), "=r"(ch.w[3]) : "l"(src));
    }
    const uint32_t g = static_cast<uint32_t>((static_cast<uint64_t>(col) * kV) >> p.g_log2);
    const float* sp = p.x_scale + static_cast<int64_t>(e) * p.se + static_cast<int64_t>(r) * p.sm;
    ch.sc0 = __ldg(sp + static_cast<int64_t>(g) * p.sg);
    ch.sc1 = ch.sc0;
    if (kV == 32 && p.g_log2 == 4u) ch.sc1 = __ldg(sp + static_cast<int64_t>(g + 1u) * p.sg);
  };

  const float oscale = *p.output_scale;                 // in flight with masked_m
  int32_t m_lane = 0;
  if (masked && lane < p.experts) m_lane = __ldg(p.masked_m + lane);
  // The warp's first task is loaded as if its rows were live (every row r < m lies inside
  // x), right after the reads of masked_m and the output scale are issued, so the three are
  // in flight together; whether it is live is settled when masked_m arrives (2.45 -> 2.27
  // us on the page's shape; issued ahead of the masked_m read it was slower, 2.53 us).
  Chunk first_ch;
  uint32_t f_r, f_e, f_c;
  {
    f_c = (warp_id << 5) + lane;
    const uint32_t S = udiv(f_c, p.cpr, p.cpr_magic);
    const uint32_t col = f_c - S * p.cpr;
    f_r = udiv(S, p.experts, p.e_magic);
    f_e = S - f_r * p.experts;
    first_ch.off = (static_cast<int64_t>(f_e) * p.m + f_r) * p.k + static_cast<int64_t>(col) * kV;
    first_ch.live = f_r < p.m;
    if (first_ch.live) load(first_ch, f_e, f_r, col);
  }

  // Live rows of expert `lane` (E <= 32), and the largest live count of any expert.
  uint32_t my_live = 0u, max_live = p.m;
  if (masked) {
    uint32_t mx = lane < p.experts ? (m_lane < 0 ? 0u : min(static_cast<uint32_t>(m_lane), p.m)) : 0u;
    my_live = mx;
    for (uint32_t e = lane + 32u; e < p.experts; e += 32u) {
      const int32_t v = __ldg(p.masked_m + e);
      mx = max(mx, v < 0 ? 0u : min(static_cast<uint32_t>(v), p.m));
    }
    max_live = redux_max(mx, 0xFFFFFFFFu);
  }
  const float inv = __frcp_rn(oscale);
  const uint64_t inv2 = pk2(inv, inv);

  // Tasks that can hold live chunks: those of the first max_live * E slots.
  const uint64_t live_chunks = static_cast<uint64_t>(max_live) * p.experts * p.cpr;
  const uint32_t tasks = static_cast<uint32_t>((live_chunks + 31u) >> 5);

  // Live rows of expert e (every lane of the warp calls this).
  auto live_rows_of = [&](uint32_t e) -> uint32_t {
    if (!masked) return p.m;
    if (p.experts <= 32u) return __shfl_sync(0xFFFFFFFFu, my_live, e & 31u);
    const int32_t v = __ldg(p.masked_m + e);
    return v < 0 ? 0u : min(static_cast<uint32_t>(v), p.m);
  };
  {
    const uint32_t live_e = live_rows_of(f_e);
    first_ch.live = first_ch.live && static_cast<uint64_t>(f_c) < live_chunks && f_r < live_e;
  }

  auto issue = [&](uint32_t t, Chunk& ch) {
    const uint32_t c = (t << 5) + lane;
    const uint32_t S = udiv(c, p.cpr, p.cpr_magic);
    const uint32_t col = c - S * p.cpr;
    const uint32_t r = udiv(S, p.experts, p.e_magic);
    const uint32_t e = S - r * p.experts;
    const uint32_t live_e = live_rows_of(e);
    ch.live = static_cast<uint64_t>(c) < live_chunks && r < live_e;
    ch.off = (static_cast<int64_t>(e) * p.m + r) * p.k + static_cast<int64_t>(col) * kV;
    if (ch.live) load(ch, e, r, col);
  };

  // (v * sc) * inv for 4 codes of one 32-bit word, two at a time (mul.rn.f32x2 rounds
  // each product like __fmul_rn), re-encoded with the saturating conversion.
  auto word = [&](uint32_t w, float sc) {
    const uint64_t sc2 = pk2(sc, sc);
    uint32_t c[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t f16x2;
      const uint16_t pair = static_cast<uint16_t>(w >> (16 * h));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f16x2) : "h"(pair));
      c[h] = e4m3x2_pair(mul2(mul2(widen2<true>(f16x2), sc2), inv2));
    }
    return c[0] | (c[1] << 16);
  };

  auto finish = [&](const Chunk& ch) {
    if (!ch.live) return;
    uint32_t o[kWords];
#pragma unroll
    for (int i = 0; i < kWords; ++i) o[i] = word(ch.w[i], i < kWords / 2 ? ch.sc0 : ch.sc1);
    uint8_t* dst = p.out + ch.off;
    if constexpr (kV == 32) {
      asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "r"(o[0]),
                   "r"(o[1]), "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                   : "memory");
    } else {
      st_128(dst, o[0], o[1], o[2], o[3]);
    }
  };

  uint32_t t = warp_id;
  if (t < tasks) {                         // the first task, already loaded
    if (t + stride < tasks) {
      Chunk b;
      issue(t + stride, b);
      finish(first_ch);
      finish(b);
      t += 2u * stride;
    } else {
      finish(first_ch);
      t += stride;
    }
  }
  if (t + stride < tasks) {                // at least two tasks: batches of two
    for (; t + stride < tasks; t += 2u * stride) {
      Chunk a, b;
      issue(t, a);
      issue(t + stride, b);
      finish(a);
      finish(b);
    }
  }
  if (t < tasks) {
    Chunk a;
    issue(t, a);
    finish(a);
  }
}

namespace {

std::mutex g_mu;
std::map<std::tuple<const void*, int, size_t>, int> g_occ;   // (kernel, device, smem) -> blocks/SM
std::map<int, int> g_sms;
std::map<std::pair<const void*, int>, size_t> g_smem_attr;   // (kernel, device) -> attribute set

// Resident CTAs per SM of `fn` at this shared-memory size and CTA size (raising the
// kernel's dynamic shared-memory limit first when needed), and the SM count.  0 or -1.
int occupancy(const void* fn, size_t smem, int threads, int* blocks_per_sm, int* sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  auto s = g_sms.find(dev);
  if (s == g_sms.end()) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    s = g_sms.emplace(dev, n).first;
  }
  // The dynamic shared-memory limit of a kernel is only ever raised, so a launch with a
  // size seen earlier stays valid after launches with smaller sizes.
  if (smem > 48 * 1024) {
    auto a = g_smem_attr.find({fn, dev});
    if (a == g_smem_attr.end() || a->second < smem) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem)) != cudaSuccess) {
        cudaGetLastError();
        return -1;
      }
      g_smem_attr[{fn, dev}] = smem;
    }
  }
  auto o = g_occ.find(std::make_tuple(fn, dev, smem + static_cast<size_t>(threads) * 1000000u));
  if (o == g_occ.end()) {
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, threads, smem) != cudaSuccess || nb < 1) {
      cudaGetLastError();
      return -1;
    }
    o = g_occ.emplace(std::make_tuple(fn, dev, smem + static_cast<size_t>(threads) * 1000000u), nb).first;
  }
  *blocks_per_sm = o->second;
  *sm_count = s->second;
  return 0;
}

int grid_for(const void* fn, size_t smem, int64_t want, int threads = kThreads) {
  int bps = 0, sms = 0;
  if (occupancy(fn, smem, threads, &bps, &sms) != 0) return -1;
  const int64_t full = static_cast<int64_t>(bps) * sms;
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, full)));
}

int launch(const void* fn, int grid, size_t smem, ptgq_stream_t stream, void** args,
           int threads = kThreads) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // A failed launch is reported through the status code and its error is cleared from the
  // runtime's state, so it does not surface later in the caller's own CUDA calls.  After a
  // successful launch the error state is left alone: an error pending from the caller's
  // earlier work is theirs to see, not this call's to report or clear.
  if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
    cudaGetLastError();
    return PTGQ_ERR_CUDA;
  }
  return PTGQ_OK;
}

const void* per_token_reg_fn(int dtype, bool wide) {
  switch (dtype * 2 + (wide ? 1 : 0)) {
    case 0: return reinterpret_cast<const void*>(&per_token_reg_kernel<0, 8>);
    case 1: return reinterpret_cast<const void*>(&per_token_reg_kernel<0, 16>);
    case 2: return reinterpret_cast<const void*>(&per_token_reg_kernel<1, 8>);
    case 3: return reinterpret_cast<const void*>(&per_token_reg_kernel<1, 16>);
    default: return reinterpret_cast<const void*>(&per_token_reg_kernel<2, 16>);
  }
}

const void* per_token_cta_fn(int dtype, int threads) {
  switch (dtype * 2 + (threads == 128 ? 1 : 0)) {
    case 0: return reinterpret_cast<const void*>(&per_token_cta_kernel<0, 256>);
    case 1: return reinterpret_cast<const void*>(&per_token_cta_kernel<0, 128>);
    case 2: return reinterpret_cast<const void*>(&per_token_cta_kernel<1, 256>);
    case 3: return reinterpret_cast<const void*>(&per_token_cta_kernel<1, 128>);
    case 4: return reinterpret_cast<const void*>(&per_token_cta_kernel<2, 256>);
    default: return reinterpret_cast<const void*>(&per_token_cta_kernel<2, 128>);
  }
}

// Calls of at most this many rows per SM take the CTA-per-row kernel.
constexpr int64_t kPtCtaRowsPerSm = 4;
// Calls of at most this many rows per SM (and more than kPtCtaRowsPerSm), with rows of at
// most kPtHalfCtaRowBytes, take CTAs of 4 warps per row ([1024, 4096]: 3.09 -> 2.81 us,
// [1600, 4096]: 4.05 -> 3.72 us, [1216, 7168]: 5.19 -> 5.04 us; longer rows re-read more of
// themselves from L2 with half the threads, [1024, 16384]: 10.08 -> 11.91 us).
constexpr int64_t kPtHalfCtaRowsPerSm = 12;
constexpr int64_t kPtHalfCtaRowBytes = 16 * 1024;

const void* per_token_smem_fn(int dtype, int bufs) {
  switch (dtype * 2 + (bufs == 2 ? 1 : 0)) {
    case 0: return reinterpret_cast<const void*>(&per_token_smem_kernel<0, 1>);
    case 1: return reinterpret_cast<const void*>(&per_token_smem_kernel<0, 2>);
    case 2: return reinterpret_cast<const void*>(&per_token_smem_kernel<1, 1>);
    case 3: return reinterpret_cast<const void*>(&per_token_smem_kernel<1, 2>);
    case 4: return reinterpret_cast<const void*>(&per_token_smem_kernel<2, 1>);
    default: return reinterpret_cast<const void*>(&per_token_smem_kernel<2, 2>);
  }
}

// Shape of the staged per-token launch: warps per CTA, row buffers per warp, CTAs.
struct PtShape {
  int warps = 0, bufs = 0, grid = 0;
  size_t smem = 0;
  const void* fn = nullptr;
};

// Rows are whole work units (a row's max must be known before any of its codes), so the
// last round of rows leaves warps idle unless the warps divide the rows evenly.  Each SM
// streams its resident warps' rows at its share of HBM bandwidth, so the time is about
// rounds * (warps per SM), with the CTAs of the grid spread evenly over the SMs; the shape
// minimizing that product wins, ties going to more warps in total.  One buffer per warp
// is allowed only when every warp takes at most one row (nothing to overlap).  Returns
// false when no shape fits.
bool per_token_shape(int dtype, int64_t tokens, int64_t row_bytes, PtShape* out) {
  constexpr int64_t kMaxSmem = 227 * 1024;
  int64_t best_cost = -1, best_total = 0;
  for (int bufs = 2; bufs >= 1; --bufs) {
    const void* fn = per_token_smem_fn(dtype, bufs);
    for (int wc = 1; wc <= kWarps; ++wc) {
      const int64_t smem = static_cast<int64_t>(wc) * bufs * row_bytes;
      if (smem > kMaxSmem) break;
      int bps = 0, sms = 0;
      if (occupancy(fn, static_cast<size_t>(smem), 32 * wc, &bps, &sms) != 0 || bps < 1)
        continue;                                   // this shape does not fit
      const int64_t total = static_cast<int64_t>(sms) * bps * wc;
      const int64_t rounds = (tokens + total - 1) / total;
      if (bufs == 1 && rounds > 1) continue;
      const int64_t grid = std::min<int64_t>(static_cast<int64_t>(sms) * bps, (tokens + wc - 1) / wc);
      const int64_t used = grid * wc;
      const int64_t cost = rounds * ((grid + sms - 1) / sms) * wc;
      if (best_cost < 0 || cost < best_cost || (cost == best_cost && used > best_total)) {
        best_cost = cost;
        best_total = used;
        out->warps = wc;
        out->bufs = bufs;
        out->smem = static_cast<size_t>(smem);
        out->fn = fn;
        out->grid = static_cast<int>(grid);
      }
    }
  }
  return best_cost >= 0;
}

}  // namespace
}  // namespace ptgq

using namespace ptgq;

extern "C" int ptgq_per_token_quant(const void* x, int dtype, int64_t num_tokens, int64_t hidden,
                                    void* out_q, float* out_s, ptgq_stream_t stream) {
  if (dtype != PTGQ_BF16 && dtype != PTGQ_FP16 && dtype != PTGQ_FP32) return PTGQ_ERR_DTYPE;
  if (hidden <= 0 || hidden % 4 != 0) return PTGQ_ERR_HIDDEN;
  if (num_tokens < 0) return PTGQ_ERR_SHAPE;
  if (num_tokens > 0 && hidden > (int64_t(1) << 62) / num_tokens) return PTGQ_ERR_TOO_LARGE;
  if (num_tokens == 0) return PTGQ_OK;
  if (x == nullptr || out_q == nullptr || out_s == nullptr) return PTGQ_ERR_NULL;
  const int esize = dtype == PTGQ_FP32 ? 4 : 2;
  // 16-byte vectors when every row start is 16-byte aligned, else 8-byte vectors (16-bit
  // rows whose length is a multiple of 4 but not of 8).
  const bool wide = dtype == PTGQ_FP32 || hidden % 8 == 0;
  const uintptr_t need = wide ? 16 : 8;
  if (reinterpret_cast<uintptr_t>(x) % need != 0 || reinterpret_cast<uintptr_t>(out_q) % (wide && esize == 2 ? 8 : 4) != 0 ||
      reinterpret_cast<uintptr_t>(out_s) % 4 != 0)
    return PTGQ_ERR_ALIGN;
  PerTokenParams p{x, static_cast<uint8_t*>(out_q), out_s, num_tokens, hidden};
  void* args[] = {&p};
  // Staged kernel: rows that are a multiple of 16 bytes, at least 512 bytes long, and of
  // which two fit in a CTA's shared memory.
  const int64_t row_bytes = hidden * esize;
  if (row_bytes % 16 == 0 && row_bytes >= 512 && reinterpret_cast<uintptr_t>(x) % 16 == 0) {
    for (const int threads : {256, 128}) {
      const void* fn = per_token_cta_fn(dtype, threads);
      int bps = 0, sms = 0;
      if (occupancy(fn, 0, threads, &bps, &sms) != 0) return PTGQ_ERR_CUDA;
      const int64_t limit = threads == 256 ? kPtCtaRowsPerSm * sms
                            : (row_bytes <= kPtHalfCtaRowBytes ? kPtHalfCtaRowsPerSm * sms : 0);
      if (num_tokens <= limit) {
        const int grid = static_cast<int>(std::min<int64_t>(num_tokens, static_cast<int64_t>(bps) * sms));
        return launch(fn, grid, 0, stream, args, threads);
      }
    }
  }
  if (row_bytes % 16 == 0 && row_bytes >= 512 && 2 * row_bytes <= 227 * 1024 &&
      reinterpret_cast<uintptr_t>(x) % 16 == 0) {
    PtShape sh;
    if (!per_token_shape(dtype, num_tokens, row_bytes, &sh)) return PTGQ_ERR_CUDA;
    return launch(sh.fn, sh.grid, sh.smem, stream, args, 32 * sh.warps);
  }
  const void* fn = per_token_reg_fn(dtype, wide);
  const int grid = grid_for(fn, 0, (num_tokens + kWarps - 1) / kWarps);
  if (grid < 0) return PTGQ_ERR_CUDA;
  return launch(fn, grid, 0, stream, args);
}

extern "C" int ptgq_requant_per_tensor(const void* x, const float* x_scale, int64_t scale_stride_e,
                                       int64_t scale_stride_m, int64_t scale_stride_g,
                                       const int32_t* masked_m, const float* output_scale,
                                       void* out, int64_t num_experts, int64_t m, int64_t k,
                                       int group_size, ptgq_stream_t stream) {
  if (group_size != 16 && group_size != 32 && group_size != 64 && group_size != 128)
    return PTGQ_ERR_GROUP;
  if (k <= 0 || k % group_size != 0) return PTGQ_ERR_HIDDEN;
  if (num_experts < 0 || m < 0 || (masked_m != nullptr && num_experts > kMaxExperts))
    return PTGQ_ERR_SHAPE;
  // Lane chunks (16 codes at least) are numbered in 32 bits on the device: each factor is
  // bounded on its own before the product is formed, so nothing overflows.
  const int64_t kLimit = int64_t(1) << 31;
  if (num_experts >= kLimit || m >= kLimit || k >= (int64_t(1) << 40) ||
      (num_experts > 0 && m > kLimit / num_experts) ||
      (num_experts * m > 0 && k / 16 > (kLimit - 1) / (num_experts * m)))
    return PTGQ_ERR_TOO_LARGE;
  if (num_experts * m == 0) return PTGQ_OK;
  if (x == nullptr || x_scale == nullptr || output_scale == nullptr || out == nullptr)
    return PTGQ_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0 || reinterpret_cast<uintptr_t>(out) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(x_scale) % 4 != 0 || reinterpret_cast<uintptr_t>(output_scale) % 4 != 0 ||
      reinterpret_cast<uintptr_t>(masked_m) % 4 != 0)
    return PTGQ_ERR_ALIGN;
  // 32 codes per lane when every row start is 32-byte aligned, else 16.
  const bool wide = k % 32 == 0 && reinterpret_cast<uintptr_t>(x) % 32 == 0 &&
                    reinterpret_cast<uintptr_t>(out) % 32 == 0;
  const int V = wide ? 32 : 16;
  RequantParams p{};
  p.x = static_cast<const uint8_t*>(x);
  p.x_scale = x_scale;
  p.masked_m = masked_m;
  p.output_scale = output_scale;
  p.out = static_cast<uint8_t*>(out);
  p.experts = static_cast<uint32_t>(num_experts);
  p.m = static_cast<uint32_t>(m);
  p.k = k;
  p.se = scale_stride_e;
  p.sm = scale_stride_m;
  p.sg = scale_stride_g;
  p.cpr = static_cast<uint32_t>(k / V);
  p.cpr_magic = p.cpr == 1 ? 0xFFFFFFFFu : static_cast<uint32_t>((uint64_t(1) << 32) / p.cpr);
  p.e_magic = p.experts == 1 ? 0xFFFFFFFFu : static_cast<uint32_t>((uint64_t(1) << 32) / p.experts);
  p.g_log2 = static_cast<uint32_t>(__builtin_ctz(static_cast<unsigned>(group_size)));
  const void* fn = wide ? reinterpret_cast<const void*>(&requant_kernel<32>)
                        : reinterpret_cast<const void*>(&requant_kernel<16>);
  const int64_t tasks = (num_experts * m * p.cpr + 31) / 32;
  int bps = 0, sms = 0;
  if (occupancy(fn, 0, kThreads, &bps, &sms) != 0) return PTGQ_ERR_CUDA;
  const int64_t wave = static_cast<int64_t>(std::min(bps, kRequantBlocksPerSm)) * sms;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((tasks + kWarps - 1) / kWarps, wave)));
  if (grid < 0) return PTGQ_ERR_CUDA;
  void* args[] = {&p};
  return launch(fn, grid, 0, stream, args);
}
