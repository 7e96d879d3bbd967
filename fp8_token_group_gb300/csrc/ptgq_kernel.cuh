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
// gate and up), amax in registers, group amax with a butterfly of shuffles over
// the G/16 lanes of the group, scale and codes in binary32, one 128-bit store of 16
// codes.  Packed UE8M0 exponents of four groups are OR-reduced into one int32
// word and stored by one lane.  Launched with programmatic dependent launch: the
// kernel waits on griddepcontrol before its first access to caller memory.
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "ptgq_device.cuh"
#include "ptgq_internal.h"
#include "ptgq_math.cuh"
#include "silu_tables.inc"

namespace ptgq {

constexpr int kSiluF16Words = (PTGQ_SILU_F16_ENTRIES + 3) / 4 * 4;
constexpr int kSiluBf16Words = 2 * PTGQ_SILU_BF16_SPAN;
// Range of amax over which the fast scale and quotient arithmetic is proven exact (checked
// for every pair of 16-bit values and 1.3e9 sampled binary32 pairs down to this amax).  The
// launcher takes the checked instances (kChecked) when eps is below it; ptgq_api.cu holds
// the same bound.
constexpr float kExactAmaxMin = 1e-24f;
constexpr float kFltMax = 3.40282346638528859812e+38f;

// IEEE quotient v / scale for the warps outside that range, made ready for the code
// conversion: a NaN quotient (inf / inf, an infinite element of a group whose amax is
// infinite) becomes the positive NaN, which the saturating e4m3 conversion encodes 0x7F,
// or 0 for int8 (NaN has no integer value).
template <bool kInt8>
__device__ __forceinline__ float exact_quotient(float v, float scale) {
  const float y = __fdiv_rn(v, scale);
  if (y == y) return y;
  return kInt8 ? 0.0f : __uint_as_float(0x7FFFFFFFu);
}

template <bool kFp16, bool kSilu>
struct SmemTables {
  // The fused-silu instances read precomputed binary32 silu results from shared memory.
  static constexpr int words = !kSilu ? 0 : (kFp16 ? kSiluF16Words : kSiluBf16Words);
  static constexpr int bytes = (words * 4 + 15) / 16 * 16;
};

// What finish() needs of one lane's share of a warp task (issue() computes it).
struct Slot {
  uint8_t* dst;          // first code byte of the lane's 16 elements
  int64_t sidx;          // scale element this lane stores (group or unit leader)
  bool unit_valid;       // the unit exists
  bool valid;            // the unit exists and this lane's group is inside the row
};

// Tuning, per instance (compile-time), from sweeps on GB300: tasks per warp batch, whether
// the next batch's loads are issued before the current batch is computed, and the CTAs per
// SM the register budget is sized for.  Without silu: two tasks loaded then computed, 4
// CTAs/SM (64 registers).  bf16 silu: one task pipelined, flat at 3 CTAs/SM, masked in one
// CTA of 24 warps per SM (80 registers; masked silu [32, 384, 2x4096]: 23.09 us against
// 23.84 us for two tasks loaded then computed).  fp16 silu: one CTA of quant_threads() per
// SM (its table fills most of the shared memory), one task pipelined.
// The light flavour of the plain flat instances (kLight): one task per batch at 6 CTAs/SM
// (40 registers, 48 warps per SM).  It ramps up faster when each warp has only a few
// tasks, and the launcher takes it below about 8 tasks per warp of the standard grid
// (4096 x 4096, G = 128: 9.8 us against the standard 10.05 us; at 4096 x 7168 the standard
// flavour is the faster one, 14.7 us against 15.4 us).
template <bool kFp16, bool kSilu, bool kMasked, bool kLight = false>
struct Tuning {
  static_assert(!kLight || (!kSilu && !kMasked), "the light flavour is plain flat only");
  static constexpr bool f16_silu = kFp16 && kSilu;
  static constexpr int threads = quant_threads(kFp16, kSilu, kMasked);
  // Tasks dealt round-robin over the CTAs (consecutive tasks to consecutive CTAs) instead
  // of in blocks of one per warp, in masked calls and in flat calls with fewer tasks than
  // warps: see quant_small_tasks_per_cta.  (Large flat calls keep the blocks: 14.8 us
  // against 15.2 us round-robin for fp16 silu [8192, 2x2048]; masked silu [32, 384,
  // 2x4096]: 22.9 us round-robin against 23.3 us.)
  static constexpr bool round_robin = f16_silu || (kSilu && kMasked);
  static constexpr int batch = (kSilu || kLight) ? 1 : 2;
  static constexpr bool pipeline = kSilu;
  static constexpr int min_blocks = (f16_silu || (kSilu && kMasked)) ? 1 : (kLight ? 6 : (!kSilu ? 4 : 3));
};

// kFmt: 0 fp32 scales, 1 UE8M0 packed four per int32, 2 UE8M0 as fp32, 3 fp32 scales with
// the element quotients taken by approximate division (fast-math interop).  The scale
// format is a template parameter so that only the packed instances carry the exponent OR.
// kChecked: every warp votes on whether all its groups' amax lie in [kExactAmaxMin, FLT_MAX]
// and otherwise takes IEEE division (below).  Needed when eps < kExactAmaxMin; the int8
// instances always vote, since a NaN quotient (an infinite element of a group whose amax is
// infinite) has no integer code without a select per element.
template <bool kFp16, bool kInt8, int kFmt, bool kSilu, bool kMasked, int kLight = 0,
          bool kChecked = false>
__global__ void __launch_bounds__((Tuning<kFp16, kSilu, kMasked, kLight != 0>::threads),
                                  (Tuning<kFp16, kSilu, kMasked, kLight != 0>::min_blocks))
    quant_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr bool kPow2 = kFmt == 1 || kFmt == 2;
  constexpr bool packed = kFmt == 1;
  using Tab = SmemTables<kFp16, kSilu>;
  using Tune = Tuning<kFp16, kSilu, kMasked, kLight != 0>;
  constexpr int kB = Tune::batch;
  constexpr int kT = Tune::threads;
  constexpr int kW = kT / 32;
  // This warp's first task, round-robin or in blocks per CTA; the warp then strides by all
  // the grid's warps.
  auto first_task = [&](bool rr) {
    return rr ? blockIdx.x + gridDim.x * (threadIdx.x >> 5) : blockIdx.x * kW + (threadIdx.x >> 5);
  };
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + Tab::bytes);

  // Module constants first (asynchronously): they do not depend on the previous grid.  The
  // masked fp16 silu instances issue their 162 KB table copy after the row prefetches below
  // instead (with the copy first, the unhinted guess made the large masked call 17% slower;
  // after them, the unhinted decode batch 2.75 -> 2.59 us and the large call 22.58 -> 22.49
  // us), the others before.
  constexpr bool kCopyFirst = !(kFp16 && kSilu && kMasked);
  if constexpr (kSilu && kCopyFirst) {
    if constexpr (kFp16) copy_to_smem_async<kT>(smem, kSiluF16, kSiluF16Words / 4);
    else copy_to_smem_async<kT>(smem, kSiluBf16, kSiluBf16Words / 4);
  }

  // The rows of this warp's first batch go to L2 before the dependency wait.  A prefetch
  // reads no value into the kernel and L2 is the point of coherence for device memory, so
  // whatever the previous kernel writes to x, the loads after the wait see it; when x was
  // not written by that kernel, the first DRAM round trip of this call overlaps its tail
  // (back-to-back calls on independent buffers, benchmarked workload: 14.95 -> 14.27 us;
  // fused silu [8192, 2x2048]: 15.01 -> 14.29 us; [64, 4096]: 1.88 -> 1.51 us).
  //   flat  : the exact tasks of the first batch (the first task and the batch's strides).
  //   masked: with a hint of the live rows per expert, the rows of the first task guessed
  //           as if every expert had exactly rows_hint live rows (hinted decode batch, bf16
  //           silu: 3.16 -> 2.91 us; fp16 silu: 3.68 -> 3.62 us); without one, as if every
  //           expert had one live row, the rows a decode batch has (unhinted decode batch,
  //           bf16 silu: 2.78 -> 2.00 us, plain 2.33 -> 2.07 us, large masked silu 23.05 ->
  //           22.90 us).  The guess only decides what is prefetched: rows below
  //           max(rows_hint, 1) <= rows of experts below n, so every prefetched address lies
  //           inside x.
  {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t lu_log2 = p.lg_log2 + p.ug_log2;
    const uint32_t local = lane & ((1u << lu_log2) - 1u);
    const uint32_t kk0 = local & ((1u << p.lg_log2) - 1u);
    auto prefetch_row = [&](int64_t grow, uint32_t g) {
      const uint16_t* src = static_cast<const uint16_t*>(p.x) + grow * p.in_row +
                            (static_cast<int64_t>(g) << (4u + p.lg_log2)) + kk0 * 16u;
      prefetch_l2(src);
      if constexpr (kSilu) prefetch_l2(src + p.hidden);
    };
    if constexpr (kMasked) {
      {
        const uint32_t rh = p.rows_hint > 0u ? p.rows_hint : 1u;
        const uint32_t rhm = p.rows_hint > 0u ? p.rows_hint_magic : 0xFFFFFFFFu;
        const uint32_t u = (first_task(Tune::round_robin) << (5u - lu_log2)) + (lane >> lu_log2);
        const uint32_t R = udiv(u, p.upr, p.upr_magic);
        const uint32_t e = udiv(R, rh, rhm);
        const uint32_t g = ((u - R * p.upr) << p.ug_log2) + (local >> p.lg_log2);
        if (e < p.n && g < p.ng)
          prefetch_row(static_cast<int64_t>(e) * p.rows + (R - e * rh), g);
      }
    } else {
      const uint32_t upw_log2 = 5u - lu_log2;
      const uint32_t tasks = (p.units_flat + (1u << upw_log2) - 1u) >> upw_log2;
      const uint32_t stride = gridDim.x * kW;
      const uint32_t t0 = first_task(Tune::round_robin && tasks < stride);
      // The light flavour prefetches a warp's second task too when the call has at most three
      // tasks per warp, so most of the input is on its way to L2 before the wait ([4096, 2048]
      // G = 128, 2.25 tasks per warp: 5.64 -> 5.23 us; [1024, 7168]: 4.77 -> 4.54 us; with
      // more tasks per warp the second prefetch was slower: [4096, 4096], 4.5 tasks per warp,
      // 9.42 -> 9.99 us).
      constexpr int kPre = kLight != 0 ? 2 : kB;
      const int nb = (kB > 1 && tasks <= stride) ? 1 : ((kLight != 0 && tasks <= 3u * stride) ? 2 : kB);
#pragma unroll
      for (int b = 0; b < kPre; ++b) {
        const uint32_t u = ((t0 + b * stride) << upw_log2) + (lane >> lu_log2);
        if (b < nb && u < p.units_flat) {
          const uint32_t R = udiv(u, p.upr, p.upr_magic);
          const uint32_t g = ((u - R * p.upr) << p.ug_log2) + (local >> p.lg_log2);
          if (g < p.ng) prefetch_row(R, g);
        }
      }
    }
  }

  if constexpr (kSilu && !kCopyFirst) copy_to_smem_async<kT>(smem, kSiluF16, kSiluF16Words / 4);

  griddep_wait();
  griddep_launch_dependents();

  constexpr bool masked = kMasked;
  int32_t* bucket = prefix + (p.n + 1);
  uint32_t bshift = 0u;
  uint32_t live_rows = 0u;
  // Masked calls of at most 32 experts: every warp reads masked_m itself (one expert per
  // lane) and scans it with shuffles, so no block barrier stands between the live counts
  // and the row loads.  w_key is the exclusive prefix of expert `lane` (all ones for lanes
  // past the experts).  When no warp has more than one task (decode-sized work), a lane
  // finds its expert with a five-step search over the warp's w_key by shuffles (wlookup);
  // larger calls copy the prefix to shared memory and use the row-to-expert buckets, whose
  // lookup is cheaper per task.  Decode batch, bf16 silu, one live row in each of 32
  // experts: 3.44 -> 2.70 us without a hint, 2.76 -> 2.09 us with expected_m = 1.
  uint32_t w_key = 0xFFFFFFFFu;
  bool wlookup = false;
  if constexpr (kMasked) {
    if (p.n <= 32) {
      const uint32_t ln = threadIdx.x & 31u;
      const int32_t mm = ln < p.n ? __ldg(p.masked_m + ln) : 0;
      const uint32_t c = mm < 0 ? 0u : min(static_cast<uint32_t>(mm), static_cast<uint32_t>(p.rows));
      uint32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (ln >= static_cast<uint32_t>(o)) incl += v;
      }
      if (ln < p.n) w_key = incl - c;
      live_rows = __shfl_sync(0xFFFFFFFFu, incl, 31);
    } else {
      masked_prefix<kT>(p.masked_m, p.n, p.rows, prefix);
      __syncthreads();
      live_rows = static_cast<uint32_t>(prefix[p.n]);
    }
    // A grid sized without knowing the live counts (no hint) often has CTAs with no task:
    // they return here, before the row-to-expert buckets (the condition is uniform).
    const uint32_t upw_log2 = 5u - (p.lg_log2 + p.ug_log2);
    const uint32_t tasks = (live_rows * p.upr + (1u << upw_log2) - 1u) >> upw_log2;
    if ((Tune::round_robin ? blockIdx.x : blockIdx.x * kW) >= tasks) {
      if constexpr (kSilu) copy_to_smem_wait();    // no copy outlives its CTA
      return;
    }
    wlookup = p.n <= 32 && tasks <= gridDim.x * kW;
    if (!wlookup) {
      if (p.n <= 32) {
        if (threadIdx.x < p.n) prefix[threadIdx.x] = static_cast<int32_t>(w_key);
        if (threadIdx.x == 0u) prefix[p.n] = static_cast<int32_t>(live_rows);
        __syncthreads();
      }
      bshift = bucket_shift(live_rows);
      build_buckets<kT>(prefix, static_cast<int>(p.n), live_rows, bshift, bucket);
    }
  }
  // A pipelined instance waits for its table only once its first loads are in flight, or,
  // in decode-sized masked calls (wlookup), right before its one task (below), so no barrier
  // is needed here then (unhinted decode batch, bf16 silu: 2.80 -> 2.66 us).
  if constexpr (kSilu && !Tune::pipeline) copy_to_smem_wait();
  if ((kSilu && !Tune::pipeline) || !wlookup) __syncthreads();
  const uint32_t total_units = masked ? live_rows * p.upr : p.units_flat;

  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t lu_log2 = p.lg_log2 + p.ug_log2;            // log2(lanes per unit)
  const uint32_t upw_log2 = 5u - lu_log2;                    // log2(units per warp task)
  const uint32_t lg = 1u << p.lg_log2;
  const uint32_t lu = 1u << lu_log2;
  const uint32_t local = lane & (lu - 1u);
  const uint32_t lane_unit = lane >> lu_log2;                // unit within the warp task
  const uint32_t gj = local >> p.lg_log2;                    // group within the unit
  const uint32_t kk = local & (lg - 1u);                     // lane within the group
  const uint32_t G = 16u << p.lg_log2;
  const uint32_t total_tasks = (total_units + (1u << upw_log2) - 1u) >> upw_log2;
  const uint32_t stride = gridDim.x * kW;
  const uint32_t first = first_task(Tune::round_robin && (kMasked || total_tasks < stride));
  const uint16_t* __restrict__ x = static_cast<const uint16_t*>(p.x);
  uint8_t* __restrict__ q = static_cast<uint8_t*>(p.q);
  const float* silu_tab = reinterpret_cast<const float*>(smem);
  const float rfmax = p.fmax == 448.0f ? (1.0f / 448.0f) : (1.0f / 127.0f);

  // Address the lane's 16 elements of task t and start its loads.  Lanes past the end
  // (or in the unused groups of a partial unit) read a valid address of the last unit
  // and are masked off later, so no load is ever predicated away.
  // WS (masked calls with wlookup): the expert comes from the warp's w_key, else from the
  // shared-memory prefix and buckets.
  auto issue = [&](auto ws, uint32_t t, Slot& sl, Raw16& a, Raw16& b) {
    [[maybe_unused]] constexpr bool WS = decltype(ws)::value;
    const uint32_t u0 = (t << upw_log2) + lane_unit;
    sl.unit_valid = u0 < total_units;
    const uint32_t u = sl.unit_valid ? u0 : total_units - 1u;
    const uint32_t R = udiv(u, p.upr, p.upr_magic);
    const uint32_t c = u - R * p.upr;
    const uint32_t g = (c << p.ug_log2) + gj;
    sl.valid = sl.unit_valid && g < p.ng;
    const uint32_t ge = g < p.ng ? g : p.ng - 1u;
    int64_t grow = R, sbase = 0;
    uint32_t row = R;
    if constexpr (kMasked) {
      int e;
      if constexpr (WS) {
        // largest e with w_key[e] <= R (w_key is nondecreasing, w_key[0] = 0)
        int lo = 0;
        uint32_t base = 0u;
#pragma unroll
        for (int step = 16; step > 0; step >>= 1) {
          const uint32_t v = __shfl_sync(0xFFFFFFFFu, w_key, lo + step);
          if (v <= R) {
            lo += step;
            base = v;
          }
        }
        e = lo;
        row = R - base;
      } else {
        const uint32_t b = R >> bshift;
        e = expert_in(prefix, bucket[b], bucket[b + 1], R);
        row = R - static_cast<uint32_t>(prefix[e]);
      }
      grow = static_cast<int64_t>(e) * p.rows + row;
      sbase = static_cast<int64_t>(e) * p.s_per_block;
    }
    const int64_t col = static_cast<int64_t>(ge) * G + kk * 16u;
    const uint16_t* src = x + grow * p.in_row + col;
    ld_stream_256(a, src);
    if constexpr (kSilu) ld_stream_256(b, src + p.hidden);
    sl.dst = q + grow * p.hidden + col;
    const uint32_t sc = packed ? c : g;
    sl.sidx = sbase + (p.col_major ? static_cast<int64_t>(sc) * p.s_mn_pad + row
                                   : static_cast<int64_t>(row) * p.s_ncol + sc);
  };

  auto finish = [&](const Slot& sl, const Raw16& a, const Raw16& b) {
    uint64_t v[8];                  // the 16 values as f32x2 pairs
    uint32_t amax_bits;
    if constexpr (kSilu) {
      if constexpr (kFp16) {
        static_assert(PTGQ_SILU_F16_POS + 0x7FFF < 0x10000 && PTGQ_SILU_F16_ENTRIES <= 0x10000,
                      "packed table indices need 16 bits per half");
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t idx = silu_f16_index2(a.w[i], PTGQ_SILU_F16_POS, PTGQ_SILU_F16_ENTRIES);
          const float s0 = silu_f16_pick(a.w[i] & 0xFFFFu, silu_tab[idx & 0xFFFFu], PTGQ_SILU_F16_POS);
          const float s1 = silu_f16_pick(a.w[i] >> 16, silu_tab[idx >> 16], PTGQ_SILU_F16_POS);
          v[i] = mul2(pk2(s0, s1), widen2<true>(b.w[i]));
        }
      } else {
        // Table entry (|bits| - FIELD_LO*128), plus SPAN for a negative gate.  Both 16-bit
        // halves of a word are offset at once: bit 15 of each half is set before the
        // subtraction (so no borrow crosses halves) and flipped back after it, leaving
        // t = |bits| - FIELD_LO*128 per half, wrapped to >= 0x8000 for a gate below the
        // table (|g| < 2^-25, zero included) and >= SPAN = 0x1000 for one above it
        // (|g| >= 128).  A warp whose OR of all t has no bit at 12 or above in either half
        // reads only inside the table (byte offsets <= 0x7FFC of 0x8000); otherwise the
        // warp takes the full definition (silu_bf16).
        static_assert(PTGQ_SILU_BF16_SPAN == 4096, "the range check assumes SPAN = 2^12");
        constexpr uint32_t kBase = PTGQ_SILU_BF16_FIELD_LO << 7;
        constexpr uint32_t kBase2 = kBase | (kBase << 16);
        constexpr uint32_t kSpan = PTGQ_SILU_BF16_SPAN;
        uint32_t t[8];
        uint32_t acc = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          t[i] = ((a.w[i] | 0x80008000u) - kBase2) ^ 0x80008000u;
          acc |= t[i];
        }
        const bool oob = (acc & 0xF000F000u) != 0u;
        if (!__any_sync(0xFFFFFFFFu, oob)) {
          const char* tab = reinterpret_cast<const char*>(silu_tab);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t w = a.w[i];
            // byte offsets 4*t (positive gate) or 4*(SPAN + t) = 0x4000 + 4*t (negative)
            const uint32_t o0 = ((t[i] << 2) & 0x3FFCu) | ((w >> 1) & 0x4000u);
            const uint32_t o1 = ((t[i] >> 14) & 0x3FFCu) | ((w >> 17) & 0x4000u);
            const float s0 = *reinterpret_cast<const float*>(tab + o0);
            const float s1 = *reinterpret_cast<const float*>(tab + o1);
            v[i] = mul2(pk2(s0, s1), widen2<false>(b.w[i]));
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float s0 = silu_bf16(a.w[i] & 0xFFFFu, silu_tab, PTGQ_SILU_BF16_FIELD_LO, kSpan);
            const float s1 = silu_bf16(a.w[i] >> 16, silu_tab, PTGQ_SILU_BF16_FIELD_LO, kSpan);
            v[i] = mul2(pk2(s0, s1), widen2<false>(b.w[i]));
          }
        }
      }
      // max |v| as floats (for finite non-negative floats the order of the values is the
      // order of their bit patterns, so this is the same maximum)
      float amax_f = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float y0, y1;
        upk2(v[i], y0, y1);
        amax_f = fmaxf(amax_f, fmaxf(fabsf(y0), fabsf(y1)));
      }
      amax_bits = f2u(amax_f);
    } else {
      uint32_t m01 = maxabs2<kFp16>(a.w[0], a.w[1]), m23 = maxabs2<kFp16>(a.w[2], a.w[3]);
      uint32_t m45 = maxabs2<kFp16>(a.w[4], a.w[5]), m67 = maxabs2<kFp16>(a.w[6], a.w[7]);
      const uint32_t m = maxabs2<kFp16>(maxabs2<kFp16>(m01, m23), maxabs2<kFp16>(m45, m67)) &
                         0x7FFF7FFFu;
      const uint32_t hm = max(m & 0xFFFFu, m >> 16);
      amax_bits = f2u(widen_lo<kFp16>(hm));
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = widen2<kFp16>(a.w[i]);
      (void)b;
    }
    amax_bits = group_max(sl.valid ? amax_bits : 0u, lg);
    const float amax = fmaxf(u2f(amax_bits), p.eps);
    float s;
    uint32_t e = 0u;
    uint64_t y[8];
    // The scale and quotients below (constant reciprocal with one correction, reciprocal
    // with an exact residual) give the IEEE results for kExactAmaxMin <= amax <= FLT_MAX.
    // amax >= eps, so only an infinite amax (an infinite element, or a silu product that
    // overflows binary32) lies outside that range unless eps < kExactAmaxMin.  The e4m3
    // instances handle it with three selects: s = +inf, and the quotients v / +inf formed
    // as v * 0 (UE8M0: the inverse of 2^128 taken as 0) or through the residual step with
    // r = 1/s = 0 and -s taken as 0: +-0 for finite v, NaN (0x7F) for infinite v.  The
    // checked, int8 and fast-divide instances vote instead: a warp with any group outside
    // the range takes IEEE division for the scale and every quotient (uniform branch).  The
    // vote and its branch cost 1-4% (sweep [32768, 7168] G = 128: 103.1 against 99.3 us
    // with the selects; masked silu fp16: 23.24 against 22.53 us).
    constexpr bool kVote = kInt8 || kChecked || kFmt == 3;
    if (!kVote || __all_sync(0xFFFFFFFFu, amax >= kExactAmaxMin && amax <= kFltMax)) {
      s = div_by_const(amax, p.fmax, rfmax);
      if constexpr (!kVote) s = amax > kFltMax ? amax : s;     // the quotient is NaN for +inf
      if constexpr (kPow2) {
        s = fmaxf(s, p.scale_floor);
        e = ue8m0_exponent(s);
        const float inv = (!kVote && e == 255u) ? 0.0f : ue8m0_inverse(e);
        const uint64_t inv2 = pk2(inv, inv);
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = mul2(v[i], inv2);
      } else if constexpr (kFmt == 3) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float v0, v1;
          upk2(v[i], v0, v1);
          y[i] = pk2(__fdividef(v0, s), __fdividef(v1, s));
        }
      } else {
        const float r = __frcp_rn(s);
        const float ns = (!kVote && s > kFltMax) ? 0.0f : -s;
        const uint64_t r2 = pk2(r, r), ns2 = pk2(ns, ns);
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = div2_by_scale(v[i], r2, ns2);
      }
    } else {
      s = __fdiv_rn(amax, p.fmax);
      float scale = s;
      if constexpr (kPow2) {
        s = fmaxf(s, p.scale_floor);
        e = ue8m0_exponent(s);
        scale = u2f(e << 23);        // 2^(e - 127): e >= 1 since s > 0; +inf for e = 255
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float v0, v1;
        upk2(v[i], v0, v1);
        y[i] = pk2(exact_quotient<kInt8>(v0, scale), exact_quotient<kInt8>(v1, scale));
      }
    }
    uint32_t o[4];
    if constexpr (kInt8) {
      // + 1.5 * 2^23 rounds |y| <= 127 to the nearest integer (ties to even) in the low byte
      const uint64_t magic = pk2(12582912.0f, 12582912.0f);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float a0, a1, b0, b1;
        upk2(add2(y[2 * i], magic), a0, a1);
        upk2(add2(y[2 * i + 1], magic), b0, b1);
        o[i] = __byte_perm(__byte_perm(f2u(a0), f2u(a1), 0x0040u),
                           __byte_perm(f2u(b0), f2u(b1), 0x0040u), 0x5410u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = e4m3x2_pair(y[2 * i]) | (e4m3x2_pair(y[2 * i + 1]) << 16);
    }
    st_128_if(sl.valid, sl.dst, o[0], o[1], o[2], o[3]);

    // One predicated store per lane: the packed word (unit leader), or the float scale /
    // power of two (group leader).
    uint32_t sval;
    bool sp;
    if constexpr (packed) {
      sval = unit_or(sl.valid ? (e << (8u * gj)) : 0u, lg);
      sp = sl.unit_valid && local == 0u;
    } else {
      sval = kPow2 ? (e << 23) : f2u(s);
      sp = sl.valid && kk == 0u;
    }
    st_32_if(sp, static_cast<uint32_t*>(p.s) + sl.sidx, sval);
  };

  // Batches of KB tasks: all their loads are issued, then all are computed.
  // With PF (plain flat calls on a grid of several waves, p.prefetch_next), the lanes also
  // prefetch the next batch's chunks into L2 while this batch computes, so the next loads
  // mostly hit L2: [32768, 7168] G = 128 104.1 -> 102.1 us, G = 16 109.3 -> 106.7 us,
  // [32768, 2048] 32.1 -> 31.4 us.  Only chunks of units below the call's units and groups
  // below the row's groups are prefetched, so every address lies inside x.
  auto batches = [&](auto kb, auto pf) {
    constexpr int KB = decltype(kb)::value;
    constexpr bool PF = decltype(pf)::value;
    for (uint32_t t = first; t < total_tasks; t += KB * stride) {
      Slot cur[KB];
      Raw16 ca[KB], cb[KB];
#pragma unroll
      for (int i = 0; i < KB; ++i) issue(std::false_type{}, t + i * stride, cur[i], ca[i], cb[i]);
      if constexpr (PF && !kMasked && kLight != 1) {
#pragma unroll
        for (int i = 0; i < KB; ++i) {
          const uint64_t tn = t + static_cast<uint64_t>(KB + i) * stride;
          const uint64_t un = (tn << upw_log2) + lane_unit;
          if (un < total_units) {
            const uint32_t R = udiv(static_cast<uint32_t>(un), p.upr, p.upr_magic);
            const uint32_t g = ((static_cast<uint32_t>(un) - R * p.upr) << p.ug_log2) + gj;
            if (g < p.ng) {
              const uint16_t* src = x + static_cast<int64_t>(R) * p.in_row +
                                    static_cast<int64_t>(g) * G + kk * 16u;
              prefetch_l2(src);
              if constexpr (kSilu) prefetch_l2(src + p.hidden);
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < KB; ++i) finish(cur[i], ca[i], cb[i]);
    }
  };
  // Software pipeline: the next batch's loads are in flight while this batch computes.
  auto pipelined = [&]() {
    uint32_t t = first;
    Slot cur[kB];
    Raw16 ca[kB], cb[kB];
#pragma unroll
    for (int i = 0; i < kB; ++i) issue(std::false_type{}, t + i * stride, cur[i], ca[i], cb[i]);
    if constexpr (kSilu) {          // uniform: every thread reaches this barrier
      copy_to_smem_wait();
      __syncthreads();
    }
    while (t < total_tasks) {
      Slot nxt[kB];
      Raw16 na[kB], nb[kB];
#pragma unroll
      for (int i = 0; i < kB; ++i) issue(std::false_type{}, t + (kB + i) * stride, nxt[i], na[i], nb[i]);
#pragma unroll
      for (int i = 0; i < kB; ++i) finish(cur[i], ca[i], cb[i]);
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        cur[i] = nxt[i];
        ca[i] = na[i];
        cb[i] = nb[i];
      }
      t += kB * stride;
    }
  };
  // The loop is chosen per call (the choice is uniform over the CTA).  The warp-lookup
  // path has a loop of its own, a single task per warp: sharing the batch loops with the
  // shared-memory lookup cost the large masked silu call 4-6% (24.3 -> 25.3-25.8 us).
  const std::false_type no{};
  const std::true_type yes{};
  const std::integral_constant<int, 1> one{};
  const std::integral_constant<int, kB> wide{};
  bool done = false;
  if constexpr (kMasked) {
    if (total_units > 0u && wlookup) {      // at most one task per warp
      Slot cur;
      Raw16 ca, cb;
      const bool has = first < total_tasks;   // uniform over the warp
      // The table is waited for before the loads here, unlike in the pipelined loop (hinted
      // decode batch, bf16 silu: 2.08 us against 2.22 us with the wait after the loads).
      if constexpr (kSilu && Tune::pipeline) {    // uniform: every thread reaches this barrier
        copy_to_smem_wait();
        __syncthreads();
      }
      if (has) issue(yes, first, cur, ca, cb);
      if (has) finish(cur, ca, cb);
      done = true;
    }
  }
  if (done || total_units == 0u) {
  } else if (!Tune::pipeline) {
    // When no warp has a second task (small or decode-sized work), one-task batches: the
    // empty slots of a wider batch would still be computed and only lengthen the call.
    if (kB > 1 && total_tasks <= stride) batches(one, no);
    else if (!kMasked && kLight != 1 && p.prefetch_next) batches(wide, yes);
    else batches(wide, no);
  } else {
    pipelined();
  }

  if constexpr (kSilu && Tune::pipeline) copy_to_smem_wait();   // no copy outlives its CTA

  // Flat scheduler: zero the padding rows of out_q and of the scales.
  if constexpr (!kMasked) {
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kT + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * kT;
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
