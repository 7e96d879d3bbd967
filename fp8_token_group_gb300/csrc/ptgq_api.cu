// ptgq_api.cu -- the C ABI (include/ptgq.h): argument validation, launch geometry,
// one kernel launch per call.  Host-side checks follow the style of the sglang
// per-token quant host contract (sglang PR #34257, "Key source snippets": output
// rows >= input rows, explicit shape checks) but report status codes instead of
// throwing.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include <cuda_runtime.h>

#include "../../include/ptgq.h"
#include "ptgq_internal.h"

namespace ptgq {

const void* kernel_for_bf16_flat(int int8, int fmt, int silu);
const void* kernel_for_bf16_masked(int int8, int fmt, int silu);
const void* kernel_for_fp16_flat(int int8, int fmt, int silu);
const void* kernel_for_fp16_masked(int int8, int fmt, int silu);
const void* kernel_for_bf16_flat_light(int int8, int fmt);
const void* kernel_for_fp16_flat_light(int int8, int fmt);
const void* kernel_for_bf16_flat_light_pf(int int8, int fmt);
const void* kernel_for_bf16_flat_checked(int fmt, int silu);
const void* kernel_for_bf16_masked_checked(int fmt, int silu);
const void* kernel_for_fp16_flat_checked(int fmt, int silu);
const void* kernel_for_fp16_masked_checked(int fmt, int silu);
const void* kernel_for_fp16_flat_light_pf(int int8, int fmt);
int table_bytes_bf16(int silu);
int table_bytes_fp16(int silu);

const void* kernel_for(const KernelKey& k) {
  if (k.checked && !k.int8 && k.fmt != 3) {
    if (k.fp16)
      return k.masked ? kernel_for_fp16_masked_checked(k.fmt, k.silu) : kernel_for_fp16_flat_checked(k.fmt, k.silu);
    return k.masked ? kernel_for_bf16_masked_checked(k.fmt, k.silu) : kernel_for_bf16_flat_checked(k.fmt, k.silu);
  }
  if (k.light == 2 && !k.masked && !k.silu)
    return k.fp16 ? kernel_for_fp16_flat_light_pf(k.int8, k.fmt) : kernel_for_bf16_flat_light_pf(k.int8, k.fmt);
  if (k.light && !k.masked && !k.silu)
    return k.fp16 ? kernel_for_fp16_flat_light(k.int8, k.fmt) : kernel_for_bf16_flat_light(k.int8, k.fmt);
  if (k.fp16)
    return k.masked ? kernel_for_fp16_masked(k.int8, k.fmt, k.silu)
                    : kernel_for_fp16_flat(k.int8, k.fmt, k.silu);
  return k.masked ? kernel_for_bf16_masked(k.int8, k.fmt, k.silu)
                  : kernel_for_bf16_flat(k.int8, k.fmt, k.silu);
}

size_t dynamic_smem_bytes(const KernelKey& k, int64_t experts) {
  const size_t tab = static_cast<size_t>(k.fp16 ? table_bytes_fp16(k.silu) : table_bytes_bf16(k.silu));
  // masked: prefix of the live-row counts (E + 1) and the row-to-expert buckets
  return tab + (experts > 0 ? static_cast<size_t>(experts + 1 + kBuckets + 1) * sizeof(int32_t) : 0);
}

namespace {

struct Geometry {
  int64_t rows;       // rows per block of x / out_q
  int64_t in_row;     // input row length in elements
  int64_t ng;         // groups per row
  int64_t ncol;       // scale columns
  int64_t mn_pad;     // column pitch of the column-major layout
  int64_t per_block;  // scale elements per block
  int64_t blocks;     // 1 (flat) or E (masked)
  int64_t upr;        // units per row
  int ug_log2;        // log2(groups per unit)
};

bool mul_ok(int64_t a, int64_t b, int64_t limit) { return a == 0 || b <= limit / a; }

int geometry(int64_t n, int64_t tokens_pad, int64_t hidden, int group_size, int scale_fmt,
             int scale_layout, int fuse_silu, bool masked, Geometry* g) {
  const int64_t kLimit = int64_t(1) << 62;
  g->rows = masked ? tokens_pad : (tokens_pad ? tokens_pad : n);
  g->in_row = fuse_silu ? 2 * hidden : hidden;
  g->ng = hidden / group_size;
  g->ncol = scale_fmt == PTGQ_SCALE_UE8M0_PACKED ? (g->ng + 3) / 4 : g->ng;
  g->mn_pad = (g->rows + 3) / 4 * 4;
  g->blocks = masked ? n : 1;
  g->ug_log2 = scale_fmt == PTGQ_SCALE_UE8M0_PACKED ? 2 : 0;
  g->upr = (g->ng + (int64_t(1) << g->ug_log2) - 1) >> g->ug_log2;
  if (!mul_ok(g->rows, g->ncol, kLimit) || !mul_ok(g->ncol, g->mn_pad, kLimit)) return PTGQ_ERR_TOO_LARGE;
  g->per_block = scale_layout == PTGQ_ROW_MAJOR ? g->rows * g->ncol : g->ncol * g->mn_pad;
  if (!mul_ok(g->blocks, g->per_block, kLimit)) return PTGQ_ERR_TOO_LARGE;
  if (!mul_ok(g->blocks, g->rows, kLimit) || !mul_ok(g->blocks * g->rows, g->in_row, kLimit))
    return PTGQ_ERR_TOO_LARGE;
  // Units (one lane-group of work each) are numbered in 31 bits on the device.
  const int64_t live_rows_max = masked ? g->blocks * g->rows : n;
  if (!mul_ok(live_rows_max, g->upr, (int64_t(1) << 31) - 1)) return PTGQ_ERR_TOO_LARGE;
  return PTGQ_OK;
}

int validate(const void* x, int dtype, int64_t n, int64_t tokens_pad, int64_t hidden,
             int group_size, const void* out_q, int out_dtype, const void* out_s, int scale_fmt,
             int scale_layout, int fuse_silu, const int32_t* masked_m, float eps, unsigned flags,
             Geometry* g) {
  if (dtype != PTGQ_BF16 && dtype != PTGQ_FP16) return PTGQ_ERR_DTYPE;
  if (out_dtype != PTGQ_E4M3 && out_dtype != PTGQ_INT8) return PTGQ_ERR_OUT_DTYPE;
  if (scale_fmt < PTGQ_SCALE_FP32 || scale_fmt > PTGQ_SCALE_UE8M0_FP32) return PTGQ_ERR_SCALE_FMT;
  if (scale_layout != PTGQ_ROW_MAJOR && scale_layout != PTGQ_COL_MAJOR_TMA) return PTGQ_ERR_LAYOUT;
  if (group_size != 16 && group_size != 32 && group_size != 64 && group_size != 128)
    return PTGQ_ERR_GROUP;
  if (hidden <= 0 || hidden % group_size != 0) return PTGQ_ERR_HIDDEN;
  if ((fuse_silu != 0 && fuse_silu != 1) ||
      (flags & ~static_cast<unsigned>(PTGQ_FLAG_NO_PDL | PTGQ_FLAG_UE8M0_SCALE_FLOOR |
                                   PTGQ_FLAG_FAST_DIVIDE)) != 0)
    return PTGQ_ERR_FLAG;
  const bool masked = masked_m != nullptr;
  if (n < 0 || tokens_pad < 0) return PTGQ_ERR_SHAPE;
  if (!masked && tokens_pad != 0 && tokens_pad < n) return PTGQ_ERR_SHAPE;
  if (masked && n > kMaxExperts) return PTGQ_ERR_SHAPE;
  if (!std::isfinite(eps) || !(eps >= PTGQ_EPS_MIN)) return PTGQ_ERR_EPS;
  const int rc = geometry(n, tokens_pad, hidden, group_size, scale_fmt, scale_layout, fuse_silu,
                          masked, g);
  if (rc != PTGQ_OK) return rc;
  // x is read only when live rows can exist; the outputs are written whenever rows exist
  // (flat padding rows are zero-filled even with no live rows).
  const bool any_rows = g->blocks * g->rows > 0;
  const bool any_live = masked ? any_rows : n > 0;
  if ((any_live && x == nullptr) || (any_rows && (out_q == nullptr || out_s == nullptr)))
    return PTGQ_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(x) % 32 != 0 || reinterpret_cast<uintptr_t>(out_q) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(out_s) % 4 != 0 || reinterpret_cast<uintptr_t>(masked_m) % 4 != 0)
    return PTGQ_ERR_ALIGN;
  return PTGQ_OK;
}

struct DeviceInfo {
  int sm_count = 0;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;
// (kernel, device, smem): each kernel is always launched with the same CTA size
std::map<std::tuple<const void*, int, size_t>, int> g_occupancy;
std::map<std::pair<const void*, int>, size_t> g_smem_attr;          // (kernel, device) -> max set

int launch_blocks(const void* fn, int dev, size_t smem, int threads, int* blocks_per_sm,
                  int* sm_count) {
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_devices.find(dev);
  if (it == g_devices.end()) {
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PTGQ_ERR_CUDA;
    it = g_devices.emplace(dev, d).first;
  }
  *sm_count = it->second.sm_count;
  const auto akey = std::make_pair(fn, dev);
  auto at = g_smem_attr.find(akey);
  if (smem > 48 * 1024 && (at == g_smem_attr.end() || at->second < smem)) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess) {
      cudaGetLastError();
      return PTGQ_ERR_CUDA;
    }
    g_smem_attr[akey] = smem;
  }
  const auto okey = std::make_tuple(fn, dev, smem);
  auto ot = g_occupancy.find(okey);
  if (ot == g_occupancy.end()) {
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, threads, smem) != cudaSuccess || nb < 1) {
      cudaGetLastError();
      return PTGQ_ERR_CUDA;
    }
    ot = g_occupancy.emplace(okey, nb).first;
  }
  *blocks_per_sm = ot->second;
  return PTGQ_OK;
}

}  // namespace
}  // namespace ptgq

using namespace ptgq;

namespace ptgq {
namespace masked_count {

// The optional out-of-range count of ptgq_quant_ex: one CTA adds the number of experts whose
// masked_m lies outside [0, rows] to *err.  A kernel of its own, launched after the quantizer
// in stream order only when the caller asks for the count, so the quantizer's code is the
// same whether or not it is counted (counting inside its masked prologue cost the fp16
// masked silu call 2%).
__global__ void __launch_bounds__(256) masked_m_error_kernel(const int32_t* __restrict__ masked_m,
                                                             int64_t n, int64_t rows,
                                                             int32_t* err) {
  int bad = 0;
  for (int64_t e = threadIdx.x; e < n; e += blockDim.x) {
    const int32_t m = masked_m[e];
    bad += (m < 0 || m > rows) ? 1 : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xFFFFFFFFu, bad, o);
  if ((threadIdx.x & 31u) == 0u && bad != 0) atomicAdd(err, bad);
}

int count_masked_errors(const int32_t* masked_m, int64_t n, int64_t rows, int32_t* err,
                        ptgq_stream_t stream) {
  if (err == nullptr || masked_m == nullptr || n == 0) return PTGQ_OK;
  void* args[] = {&masked_m, &n, &rows, &err};
  // As for the quantizer's launch: only this launch's own failure is reported and cleared.
  if (cudaLaunchKernel(reinterpret_cast<const void*>(&masked_m_error_kernel), dim3(1), dim3(256),
                       args, 0, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return PTGQ_ERR_CUDA;
  }
  return PTGQ_OK;
}

}  // namespace masked_count
}  // namespace ptgq

extern "C" int ptgq_quant_ex(const void* x, int dtype, int64_t n, int64_t tokens_pad,
                             int64_t hidden, int group_size, void* out_q, int out_dtype,
                             void* out_s, int scale_fmt, int scale_layout, int fuse_silu,
                             const int32_t* masked_m, float eps, ptgq_stream_t stream,
                             unsigned flags, int64_t expected_m, int32_t* masked_m_errors) {
  Geometry g;
  int rc = validate(x, dtype, n, tokens_pad, hidden, group_size, out_q, out_dtype, out_s,
                    scale_fmt, scale_layout, fuse_silu, masked_m, eps, flags, &g);
  if (rc != PTGQ_OK) return rc;
  if (expected_m < 0) return PTGQ_ERR_SHAPE;
  const bool masked = masked_m != nullptr;
  if (masked && masked_m_errors != nullptr &&
      reinterpret_cast<uintptr_t>(masked_m_errors) % 4 != 0)
    return PTGQ_ERR_ALIGN;
  using ptgq::masked_count::count_masked_errors;
  if (g.blocks * g.rows == 0)                   // nothing to read or write
    return masked ? count_masked_errors(masked_m, n, g.rows, masked_m_errors, stream) : PTGQ_OK;

  Params p{};
  p.x = x;
  p.q = out_q;
  p.s = out_s;
  p.masked_m = masked_m;
  p.n = n;
  p.rows = g.rows;
  p.hidden = hidden;
  p.in_row = g.in_row;
  p.lg_log2 = static_cast<uint32_t>(__builtin_ctz(static_cast<unsigned>(group_size / 16)));
  p.ug_log2 = static_cast<uint32_t>(g.ug_log2);
  p.ng = static_cast<uint32_t>(g.ng);
  p.upr = static_cast<uint32_t>(g.upr);
  p.upr_magic = g.upr == 1 ? 0xFFFFFFFFu
                           : static_cast<uint32_t>((uint64_t(1) << 32) / static_cast<uint64_t>(g.upr));
  p.units_flat = masked ? 0u : static_cast<uint32_t>(n * g.upr);
  p.scale_fmt = scale_fmt;
  p.col_major = scale_layout == PTGQ_COL_MAJOR_TMA;
  p.s_ncol = g.ncol;
  p.s_mn_pad = g.mn_pad;
  p.s_per_block = g.per_block;
  p.eps = eps;
  p.fmax = out_dtype == PTGQ_E4M3 ? 448.0f : 127.0f;
  p.scale_floor = (flags & PTGQ_FLAG_UE8M0_SCALE_FLOOR) ? 1e-10f : 0.0f;
  p.rows_hint = masked && expected_m > 0
                    ? static_cast<uint32_t>(std::min<int64_t>(expected_m, g.rows)) : 0u;
  p.rows_hint_magic = p.rows_hint <= 1u ? 0xFFFFFFFFu
                                        : static_cast<uint32_t>((uint64_t(1) << 32) / p.rows_hint);
  if (!masked) {
    p.zero_q_begin = n * hidden;
    p.zero_q_end = g.rows * hidden;
    p.zero_s_rows = (scale_layout == PTGQ_ROW_MAJOR ? g.rows : g.mn_pad) - n;
  }

  // Internal format 3: fp32 scales with approximate element division (fast-math interop).
  const int kfmt = (scale_fmt == PTGQ_SCALE_FP32 && (flags & PTGQ_FLAG_FAST_DIVIDE)) ? 3 : scale_fmt;
  KernelKey key{dtype == PTGQ_FP16, out_dtype == PTGQ_INT8, kfmt, fuse_silu, masked, 0, eps < kExactAmaxEps};
  const void* fn = kernel_for(key);
  const size_t smem = dynamic_smem_bytes(key, masked ? n : 0);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PTGQ_ERR_CUDA;
  const int threads = quant_threads(key.fp16 != 0, key.silu != 0, key.masked != 0);
  int per_sm = 0, sms = 0;
  rc = launch_blocks(fn, dev, smem, threads, &per_sm, &sms);
  if (rc != PTGQ_OK) return rc;

  // Grid: at most one full wave, fewer when the work is small (masked: as small as the
  // expected live rows need, when the caller gives a hint); the kernel strides over tasks.
  const int64_t lanes_per_unit = (int64_t(group_size) / 16) << g.ug_log2;
  const int64_t rows_hint = expected_m > 0 ? std::min<int64_t>(expected_m, g.rows) : g.rows;
  const int64_t units_max = (masked ? g.blocks * rows_hint : n) * g.upr;
  const int64_t tasks = (units_max * lanes_per_unit + 31) / 32;
  // Plain flat work of at most about 8 tasks per warp of the standard grid: the light
  // flavour (one task per batch, more warps per SM) ramps up faster.
  if (!masked && !fuse_silu && !key.checked && tasks <= 8 * static_cast<int64_t>(per_sm) * sms * kWarps) {
    key.light = 1;
    fn = kernel_for(key);
    rc = launch_blocks(fn, dev, smem, threads, &per_sm, &sms);
    if (rc != PTGQ_OK) return rc;
    // Above three tasks per warp of the light grid, the instances with the next-batch
    // prefetch; up to three, the kernel prefetches a warp's first two tasks before its
    // dependency wait instead, and the rolling prefetch only costs issue slots ([4096, 2048]:
    // 5.23 -> 4.92 us, [1024, 7168]: 4.55 -> 4.24 us without it).
    if (tasks > 3 * static_cast<int64_t>(per_sm) * sms * kWarps) {
      key.light = 2;
      p.prefetch_next = 1u;
      fn = kernel_for(key);
      rc = launch_blocks(fn, dev, smem, threads, &per_sm, &sms);
      if (rc != PTGQ_OK) return rc;
    }
  }
  const int per_cta = quant_small_tasks_per_cta(key.fp16 != 0, key.silu != 0, key.masked != 0);
  int64_t want = (tasks + per_cta - 1) / per_cta;
  int64_t full = static_cast<int64_t>(per_sm) * sms;
  // Large plain flat calls (more than 16 tasks per warp of one wave): CTAs of 8 tasks per warp
  // instead of one persistent wave.  A persistent wave finishes unevenly (on each SM the CTA
  // dispatched first ends about 1.4 us before the last one, and SMs differ by up to 2 us);
  // with several waves of shorter CTAs the block scheduler hands the later CTAs to the SMs
  // that free up first.  [32768, 7168]: 105.2 -> 103.9 us at G = 128, 123.7 -> 109.6 us at
  // G = 16; [8192, 7168] G = 16: 30.2 -> 29.4 us.  Below the threshold (the benchmarked
  // [4096, 7168] has 11.8 tasks per warp) one wave stays faster (14.9 against 15.7 us).
  if (!masked && !fuse_silu && !key.light && tasks > 16 * full * kWarps) {
    want = (tasks + per_cta * 8 - 1) / (per_cta * 8);
    full = want;
    p.prefetch_next = 1u;
  }
  if (!masked) {
    const int64_t zero_chunks = (p.zero_q_end - p.zero_q_begin) / 16 + p.zero_s_rows * g.ncol;
    want = std::max<int64_t>(want, (zero_chunks + threads - 1) / threads);
  }
  const unsigned grid = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(want, std::max(full, int64_t(1)))));

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (flags & PTGQ_FLAG_NO_PDL) ? 0 : 1;
  void* args[] = {&p};
  // A failed launch is reported through the status code and its error is cleared from the
  // runtime's state, so it does not surface later in the caller's own CUDA calls.  After a
  // successful launch the error state is left alone: an error pending from the caller's
  // earlier work is theirs to see, not this call's to report or clear.
  if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) {
    cudaGetLastError();
    return PTGQ_ERR_CUDA;
  }
  return masked ? count_masked_errors(masked_m, n, g.rows, masked_m_errors, stream) : PTGQ_OK;
}

extern "C" int ptgq_quant(const void* x, int dtype, int64_t n, int64_t tokens_pad, int64_t hidden,
                          int group_size, void* out_q, int out_dtype, void* out_s, int scale_fmt,
                          int scale_layout, int fuse_silu, const int32_t* masked_m, float eps,
                          ptgq_stream_t stream) {
  return ptgq_quant_ex(x, dtype, n, tokens_pad, hidden, group_size, out_q, out_dtype, out_s,
                       scale_fmt, scale_layout, fuse_silu, masked_m, eps, stream, 0u, 0, nullptr);
}

extern "C" int ptgq_scale_elems(int64_t n, int64_t tokens_pad, int64_t hidden, int group_size,
                                int scale_fmt, int scale_layout, int masked, int64_t* n_out) {
  if (n_out == nullptr) return PTGQ_ERR_NULL;
  if (scale_fmt < PTGQ_SCALE_FP32 || scale_fmt > PTGQ_SCALE_UE8M0_FP32) return PTGQ_ERR_SCALE_FMT;
  if (scale_layout != PTGQ_ROW_MAJOR && scale_layout != PTGQ_COL_MAJOR_TMA) return PTGQ_ERR_LAYOUT;
  if (group_size != 16 && group_size != 32 && group_size != 64 && group_size != 128)
    return PTGQ_ERR_GROUP;
  if (hidden <= 0 || hidden % group_size != 0) return PTGQ_ERR_HIDDEN;
  if (n < 0 || tokens_pad < 0 || (!masked && tokens_pad != 0 && tokens_pad < n)) return PTGQ_ERR_SHAPE;
  Geometry g;
  const int rc = geometry(n, tokens_pad, hidden, group_size, scale_fmt, scale_layout, 0, masked != 0, &g);
  if (rc != PTGQ_OK) return rc;
  *n_out = g.blocks * g.per_block;
  return PTGQ_OK;
}

extern "C" const char* ptgq_strerror(int status) {
  switch (status) {
    case PTGQ_OK: return "ok";
    case PTGQ_ERR_NULL: return "a required pointer is NULL";
    case PTGQ_ERR_DTYPE: return "unknown input dtype";
    case PTGQ_ERR_OUT_DTYPE: return "unknown output dtype";
    case PTGQ_ERR_GROUP: return "group_size must be 16, 32, 64 or 128";
    case PTGQ_ERR_HIDDEN: return "hidden must be positive and a multiple of group_size";
    case PTGQ_ERR_SHAPE: return "invalid row counts (negative, tokens_pad < num_tokens, or too many experts)";
    case PTGQ_ERR_ALIGN: return "misaligned pointer (x 32 B, out_q 16 B, out_s and masked_m 4 B)";
    case PTGQ_ERR_SCALE_FMT: return "unknown scale format";
    case PTGQ_ERR_LAYOUT: return "unknown scale layout";
    case PTGQ_ERR_EPS: return "eps must be finite and >= PTGQ_EPS_MIN (2^-140)";
    case PTGQ_ERR_FLAG: return "fuse_silu must be 0 or 1 and flags must be PTGQ_FLAG_* bits";
    case PTGQ_ERR_TOO_LARGE: return "sizes exceed the supported index range";
    case PTGQ_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}
