// ptgq_kernel.cuh -- the per-token-group quantization kernel for sm_103a.
//
// One persistent, grid-strided kernel serves both schedulers of the pages
// (sglang PR #30924, "Implementation breakdown" item 1: flat and masked
// schedulers; sglang PR #27449, "Summary": NaiveScheduler and
// MaskedLayoutScheduler):
//   flat   : every row of x [T, H_in] is live; padding rows of out_q and of the
//            scales are zero-filled (vLLM PR #41326, "Implementation breakdown"
//            item 4).
//   masked : x [E, tokens_pad, H_in]; only rows t < masked_m[e] are read or
//            written (sglang PR #35593, "Key source snippets",
//            test_masked_rows_and_k_tail).  Each CTA turns masked_m into a prefix
//            sum in shared memory, so work is dealt out over live rows only and no
//            CTA is spent on dead rows.
// Per lane: one 256-bit load of 16 contiguous 16-bit elements (two with silu:
// gate and up), amax in registers, group amax with redux.sync over the G/16
// lanes of the group, scale and codes in binary32, one 128-bit store of 16
// codes.  Packed UE8M0 exponents of four groups are OR-reduced into one int32
// word and stored by one lane.  Launched with programmatic dependent launch: the
// kernel waits on griddepcontrol before its first access to caller memory.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "ptgq_device.cuh"
#include "ptgq_internal.h"
#include "ptgq_math.cuh"
#include "silu_tables.inc"

namespace ptgq {

constexpr int kExpIntWords = 2 * (PTGQ_EXP_INT_MAX - PTGQ_EXP_INT_MIN + 1);
constexpr int kExpFracWords = 2 * (PTGQ_EXP_FRAC_JMAX - PTGQ_EXP_FRAC_JMIN + 1);
constexpr int kSiluBf16Words = 2 * PTGQ_SILU_BF16_SPAN;

template <bool kFp16, bool kSilu>
struct SmemTables {
  // bf16 silu reads the precomputed table of results; fp16 silu rebuilds exp
  // from the (hi, lo) exp tables.
  static constexpr int words = !kSilu ? 0 : (kFp16 ? kExpIntWords + kExpFracWords : kSiluBf16Words);
  static constexpr int bytes = (words * 4 + 15) / 16 * 16;
};

// One lane's share of a warp task.
struct Slot {
  const uint16_t* src;   // first input element (gate half with silu)
  uint8_t* dst;          // first code byte
  int64_t s_base;        // scale block base (elements)
  uint32_t row;          // row within the block
  uint32_t g;            // group within the row
  uint32_t c;            // unit within the row
  bool unit_valid;       // the unit exists
  bool valid;            // the unit exists and this lane's group is inside the row
};

template <bool kFp16, bool kInt8, bool kPow2, bool kSilu>
__global__ void __launch_bounds__(kThreads) quant_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  using Tab = SmemTables<kFp16, kSilu>;
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + Tab::bytes);

  // Module constants first: they do not depend on the previous grid.
  if constexpr (kSilu) {
    uint4* dst = reinterpret_cast<uint4*>(smem);
    if constexpr (kFp16) {
      const uint32_t* a = kExpIntHL;
      const uint32_t* b = kExpFracHL;
      uint32_t* d32 = reinterpret_cast<uint32_t*>(smem);
      for (int i = threadIdx.x; i < kExpIntWords; i += kThreads) d32[i] = a[i];
      for (int i = threadIdx.x; i < kExpFracWords; i += kThreads) d32[kExpIntWords + i] = b[i];
      (void)dst;
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(kSiluBf16);
      for (int i = threadIdx.x; i < kSiluBf16Words / 4; i += kThreads) dst[i] = src[i];
    }
  }

  griddep_wait();
  griddep_launch_dependents();

  const bool masked = p.masked_m != nullptr;
  uint32_t total_units = p.units_flat;
  if (masked) {
    masked_prefix(p.masked_m, p.n, p.rows, prefix);
  }
  __syncthreads();
  if (masked) total_units = static_cast<uint32_t>(prefix[p.n]) * p.upr;

  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t lu_log2 = p.lg_log2 + p.ug_log2;            // log2(lanes per unit)
  const uint32_t upw_log2 = 5u - lu_log2;                    // log2(units per warp task)
  const uint32_t lg = 1u << p.lg_log2;
  const uint32_t lu = 1u << lu_log2;
  const uint32_t local = lane & (lu - 1u);
  const uint32_t gj = local >> p.lg_log2;                    // group within the unit
  const uint32_t kk = local & (lg - 1u);                     // lane within the group
  const uint32_t gmask = (lg == 32u ? 0xFFFFFFFFu : ((1u << lg) - 1u)) << (lane & ~(lg - 1u));
  const uint32_t umask = (lu == 32u ? 0xFFFFFFFFu : ((1u << lu) - 1u)) << (lane & ~(lu - 1u));
  const uint32_t G = 16u << p.lg_log2;
  const uint32_t total_tasks = (total_units + (1u << upw_log2) - 1u) >> upw_log2;
  const uint32_t stride = gridDim.x * kWarps;
  const uint32_t first = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const uint16_t* __restrict__ x = static_cast<const uint16_t*>(p.x);
  uint8_t* __restrict__ q = static_cast<uint8_t*>(p.q);
  const float* silu_tab = reinterpret_cast<const float*>(smem);

  auto prep = [&](uint32_t t) {
    Slot sl;
    const uint32_t u = (t << upw_log2) + (lane >> lu_log2);
    sl.unit_valid = t < total_tasks && u < total_units;
    const uint32_t uu = sl.unit_valid ? u : 0u;
    const uint32_t R = udiv(uu, p.upr, p.upr_magic);
    sl.c = uu - R * p.upr;
    sl.g = (sl.c << p.ug_log2) + gj;
    sl.valid = sl.unit_valid && sl.g < p.ng;
    int64_t blk = 0;
    uint32_t r = R;
    if (masked) {
      const int e = expert_of(prefix, static_cast<int>(p.n), R);
      r = R - static_cast<uint32_t>(prefix[e]);
      blk = e;
    }
    sl.row = r;
    const int64_t grow = blk * p.rows + r;
    const int64_t col = static_cast<int64_t>(sl.g) * G + kk * 16u;
    sl.src = x + grow * p.in_row + col;
    sl.dst = q + grow * p.hidden + col;
    sl.s_base = blk * p.s_per_block;
    return sl;
  };

  auto finish = [&](const Slot& sl, const Raw16& a, const Raw16& b) {
    float v[16];
    uint32_t amax_bits;
    if constexpr (kSilu) {
      amax_bits = 0u;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float s0, s1;
        if constexpr (kFp16) {
          const float2* ei = reinterpret_cast<const float2*>(silu_tab);
          const float2* ef = ei + kExpIntWords / 2;
          s0 = silu_generic(widen_lo<true>(a.w[i]), ei, ef, PTGQ_EXP_INT_MIN, PTGQ_EXP_FRAC_JMIN);
          s1 = silu_generic(widen_hi<true>(a.w[i]), ei, ef, PTGQ_EXP_INT_MIN, PTGQ_EXP_FRAC_JMIN);
        } else {
          s0 = silu_bf16(a.w[i] & 0xFFFFu, silu_tab, PTGQ_SILU_BF16_FIELD_LO, PTGQ_SILU_BF16_SPAN);
          s1 = silu_bf16(a.w[i] >> 16, silu_tab, PTGQ_SILU_BF16_FIELD_LO, PTGQ_SILU_BF16_SPAN);
        }
        v[2 * i] = __fmul_rn(s0, widen_lo<kFp16>(b.w[i]));
        v[2 * i + 1] = __fmul_rn(s1, widen_hi<kFp16>(b.w[i]));
        amax_bits = max(amax_bits, f2u(v[2 * i]) & 0x7FFFFFFFu);
        amax_bits = max(amax_bits, f2u(v[2 * i + 1]) & 0x7FFFFFFFu);
      }
    } else {
      // |x| of 16-bit floats orders like the unsigned bit patterns without the sign.
      uint32_t m = 0u;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        m = __vmaxu2(m, a.w[i] & 0x7FFF7FFFu);
        v[2 * i] = widen_lo<kFp16>(a.w[i]);
        v[2 * i + 1] = widen_hi<kFp16>(a.w[i]);
      }
      const uint32_t hm = max(m & 0xFFFFu, m >> 16);
      amax_bits = f2u(widen_lo<kFp16>(hm));
      (void)b;
    }
    amax_bits = redux_max(sl.valid ? amax_bits : 0u, gmask);
    const float amax = fmaxf(u2f(amax_bits), p.eps);
    float s = __fdiv_rn(amax, p.fmax);
    uint32_t e = 0u;
    float y[16];
    if constexpr (kPow2) {
      if (p.scale_floor) s = fmaxf(s, 1e-10f);
      e = ue8m0_exponent(s);
      const float inv = ue8m0_inverse(e);
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = __fmul_rn(v[i], inv);
    } else {
      const float r = __frcp_rn(s);
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = div_by_scale(v[i], s, r);
    }
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (kInt8) o[i] = s8x4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
      else o[i] = e4m3x4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
    }
    if (sl.valid) st_128(sl.dst, o[0], o[1], o[2], o[3]);

    // scales
    if (p.scale_fmt == 1) {
      const uint32_t word = redux_or(sl.valid && kk == 0u ? (e << (8u * gj)) : 0u, umask);
      if (sl.unit_valid && local == 0u) {
        const int64_t idx = p.col_major ? sl.s_base + static_cast<int64_t>(sl.c) * p.s_mn_pad + sl.row
                                        : sl.s_base + static_cast<int64_t>(sl.row) * p.s_ncol + sl.c;
        static_cast<uint32_t*>(p.s)[idx] = word;
      }
    } else if (sl.valid && kk == 0u) {
      const float sv = p.scale_fmt == 0 ? s : u2f(e << 23);
      const int64_t idx = p.col_major ? sl.s_base + static_cast<int64_t>(sl.g) * p.s_mn_pad + sl.row
                                      : sl.s_base + static_cast<int64_t>(sl.row) * p.s_ncol + sl.g;
      static_cast<float*>(p.s)[idx] = sv;
    }
  };

  // Two tasks in flight per warp: both loads are issued before either is used.
  for (uint32_t t = first; t < total_tasks; t += 2u * stride) {
    const Slot s0 = prep(t);
    const Slot s1 = prep(t + stride);
    Raw16 a0, a1, b0, b1;
    if (s0.valid) ld_stream_256(a0, s0.src);
    if (s1.valid) ld_stream_256(a1, s1.src);
    if constexpr (kSilu) {
      if (s0.valid) ld_stream_256(b0, s0.src + p.hidden);
      if (s1.valid) ld_stream_256(b1, s1.src + p.hidden);
    }
    if (!s0.valid) {
#pragma unroll
      for (int i = 0; i < 8; ++i) a0.w[i] = b0.w[i] = 0u;
    }
    if (!s1.valid) {
#pragma unroll
      for (int i = 0; i < 8; ++i) a1.w[i] = b1.w[i] = 0u;
    }
    finish(s0, a0, b0);
    finish(s1, a1, b1);
  }

  // Flat scheduler: zero the padding rows of out_q and of the scales.
  if (!masked) {
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t off = p.zero_q_begin + tid * 16; off < p.zero_q_end; off += nthr * 16)
      st_128(q + off, 0u, 0u, 0u, 0u);
    const int64_t nz = p.zero_s_rows * p.s_ncol;
    uint32_t* s32 = static_cast<uint32_t*>(p.s);
    for (int64_t i = tid; i < nz; i += nthr) {
      const int64_t rr = p.n + i / p.s_ncol;
      const int64_t cc = i % p.s_ncol;
      s32[p.col_major ? cc * p.s_mn_pad + rr : rr * p.s_ncol + cc] = 0u;
    }
  }
}

}  // namespace ptgq
