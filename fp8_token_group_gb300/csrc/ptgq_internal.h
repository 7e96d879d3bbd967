// ptgq_internal.h -- launch parameters shared by the kernel translation units and the
// C ABI layer.  Not part of the public interface (that is include/ptgq.h).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ptgq {

constexpr int kThreads = 256;                 // 8 warps per CTA (the plain and flat silu instances)
constexpr int kWarps = kThreads / 32;
// Threads per CTA of a quantizer instance.  The fp16 fused-silu instances hold a 162 KB
// table of silu results in shared memory, so one CTA per SM carries all their warps.  The
// bf16 masked silu instances also take one CTA of 24 warps per SM: a masked grid is sized
// without knowing the live rows, and its CTAs that find no task cost less as a third as
// many larger CTAs (decode batch without a hint: 4.07 -> 3.48 us; [32, 384, 2x4096] with
// 6360 live rows: 24.42 -> 24.02 us).
constexpr int quant_threads(bool fp16, bool silu, bool masked) {
  return fp16 && silu ? 1024 : (silu && masked ? 768 : kThreads);
}
// Tasks a CTA of an instance takes in a call too small to fill the grid: one per warp,
// except in the one-CTA-per-SM silu instances, whose large CTAs then deal consecutive tasks
// round-robin over the grid and are given 8 each, so a small call spreads over as many SMs
// as 8-warp CTAs would (each SM's ingress from memory, not its warps, bounds such a call:
// a fp16 [64, 2x2048] call takes 2.3 us instead of 3.6 us).
constexpr int quant_small_tasks_per_cta(bool fp16, bool silu, bool masked) {
  return silu && (fp16 || masked) ? 8 : quant_threads(fp16, silu, masked) / 32;
}
constexpr int kMaxExperts = 4096;             // masked scheduler: E <= kMaxExperts
constexpr int kBuckets = 256;                 // masked scheduler: row-to-expert buckets

// Work decomposition.  A "unit" is one group (float scale formats) or four
// consecutive groups of one row (packed UE8M0, so one unit fills one int32 word).
// One lane handles 16 consecutive elements of a group (32 bytes of bf16/fp16),
// so a group spans G/16 lanes and a unit 4*G/16 or G/16 lanes; a warp task is 32
// lanes = 32 / (lanes per unit) consecutive units.  Units are numbered row by row
// over the live rows (flat: all T rows; masked: expert by expert, live rows only).
struct Params {
  const void* x;             // input (bf16/fp16)
  void* q;                   // codes (e4m3/int8)
  void* s;                   // scales
  const int32_t* masked_m;   // nullptr: flat scheduler
  int64_t n;                 // flat: live rows T; masked: experts E
  int64_t rows;              // rows per block of x/q (flat: tokens_pad or T; masked: tokens_pad)
  int64_t hidden;            // H
  int64_t in_row;            // elements per input row (H, or 2H with silu)
  uint32_t lg_log2;          // log2(lanes per group) = log2(G / 16)
  uint32_t ug_log2;          // log2(groups per unit): 2 for packed UE8M0, else 0
  uint32_t ng;               // groups per row
  uint32_t upr;              // units per row = ceil(ng / groups per unit)
  uint32_t upr_magic;        // floor(2^32 / upr), or 0xFFFFFFFF when upr == 1
  uint32_t units_flat;       // flat: T * upr (< 2^32); masked: unused
  int32_t scale_fmt;         // 0 fp32, 1 packed UE8M0, 2 UE8M0 as fp32
  int32_t col_major;         // scales column-major (TMA-aligned)
  int64_t s_ncol;            // scale columns (ng, or ceil(ng/4) words)
  int64_t s_mn_pad;          // column pitch of the column-major layout
  int64_t s_per_block;       // scale elements per block (per expert)
  float eps;                 // amax floor
  float fmax;                // 448 (e4m3) or 127 (int8)
  float scale_floor;         // UE8M0 only: s = max(s, scale_floor); 1e-10 for the vLLM
                             // semantics, else 0 (a no-op since s > 0)
  uint32_t rows_hint;        // masked: the caller's expected live rows per expert,
                             // min(expected_m, rows); 0 without a hint
  uint32_t rows_hint_magic;  // floor(2^32 / rows_hint), or 0xFFFFFFFF when rows_hint <= 1
  uint32_t prefetch_next;    // plain flat calls on several waves: 1 to prefetch the next batch
  // Flat zero-fill of padding (rows [T, rows) of q; scale rows past T).
  int64_t zero_q_begin;      // byte offsets into q, multiples of 16
  int64_t zero_q_end;
  int64_t zero_s_rows;       // scale rows to zero per column: [T, T + zero_s_rows)
};

// One kernel instance per (input type, output type, scale arithmetic, silu, scheduler).
struct KernelKey {
  int fp16;       // input is fp16 (else bf16)
  int int8;       // output is int8 (else e4m3)
  int fmt;        // 0 fp32, 1 UE8M0 packed, 2 UE8M0 as fp32, 3 fp32 with approximate division
  int silu;       // fused silu(gate) * up
  int masked;     // masked (EP-MoE) scheduler (else flat)
  int light;      // plain flat only: 1 the flavour for a few tasks per warp, 2 the same with
                  // the next-batch prefetch (more than one task per warp)
  int checked;    // e4m3, fmt 0..2: the instances that vote on the amax range (eps below
                  // kExactAmaxEps)
};

// Lower end of the amax range over which the kernels' fast scale and quotient arithmetic is
// exact (the same bound as kExactAmaxMin in ptgq_kernel.cuh): calls with a smaller eps take
// the checked instances.
constexpr float kExactAmaxEps = 1e-24f;

// Returns the __global__ function of an instance (defined in the instance TUs).
const void* kernel_for(const KernelKey& k);
// Dynamic shared memory the instance needs for `experts` masked blocks (0: flat).
size_t dynamic_smem_bytes(const KernelKey& k, int64_t experts);

}  // namespace ptgq
