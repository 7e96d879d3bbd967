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
// vector loads and stores, PDL, no shared-memory staging beyond the masked prefix.
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
  griddep_wait();
  griddep_launch_dependents();
  const int warps = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
    for (int64_t c = lane; c < chunks; c += 32) {
      uint32_t w[4];
      chunk(slot, c, w);
      quantize16<kIn>(w, inv, qrow + c * kPer16);
    }
    if (lane == 0) p.s[row] = s;
    issue(row + kPtBufs * W, slot);                        // refill this buffer
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
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
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
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
  auto quantize_store = [&](int64_t row, int64_t i, const uint32_t (&w)[kWords], float inv) {
    uint8_t* dst = p.q + row * p.hidden + i * kElems;
    if constexpr (kVecBytes == 16) {
      quantize16<kIn>(w, inv, dst);
    } else {       // 16-bit, 4 elements
      constexpr bool h = kIn == 1;
      const uint32_t o = e4m3x4(__fmul_rn(widen_lo<h>(w[0]), inv), __fmul_rn(widen_hi<h>(w[0]), inv),
                                __fmul_rn(widen_lo<h>(w[1]), inv), __fmul_rn(widen_hi<h>(w[1]), inv));
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
#pragma unroll
    for (int j = 0; j < kCache; ++j) {
      const int64_t i = lane + 32 * j;
      if (i < nvec) quantize_store(row, i, cache[j], inv);
    }
    for (int64_t i = lane + 32 * kCache; i < nvec; i += 32) {
      uint32_t w[kWords];
      load(row, i, w);
      quantize_store(row, i, w, inv);
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
  int64_t experts;
  int64_t m;                     // rows per expert
  int64_t k;                     // row length
  int64_t se, sm, sg;            // x_scale strides (elements)
  uint32_t lg_log2;              // log2(lanes per group) = log2(G / 16)
  uint32_t gpr;                  // groups per row
  uint32_t gpr_magic;            // floor(2^32 / gpr), or 0xFFFFFFFF when gpr == 1
};

// Each lane requantizes 16 codes (16 bytes) of one group; G/16 lanes share a group's scale.
__global__ void __launch_bounds__(kThreads) requant_kernel(const RequantParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  int32_t* prefix = reinterpret_cast<int32_t*>(smem);
  griddep_wait();
  griddep_launch_dependents();
  const float oscale = *p.output_scale;                 // in flight during the prefix sum
  const bool masked = p.masked_m != nullptr;
  uint32_t live_rows = static_cast<uint32_t>(p.experts * p.m);
  if (masked) masked_prefix(p.masked_m, p.experts, p.m, prefix);
  __syncthreads();
  if (masked) live_rows = static_cast<uint32_t>(prefix[p.experts]);
  const float inv = __frcp_rn(oscale);

  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t lg = 1u << p.lg_log2;
  const uint32_t kk = lane & (lg - 1u);
  const uint32_t gpw_log2 = 5u - p.lg_log2;                 // groups per warp task
  const uint32_t total_groups = live_rows * p.gpr;
  const uint32_t tasks = (total_groups + (1u << gpw_log2) - 1u) >> gpw_log2;
  const uint32_t stride = gridDim.x * kWarps;
  for (uint32_t t = blockIdx.x * kWarps + (threadIdx.x >> 5); t < tasks; t += stride) {
    const uint32_t gi = (t << gpw_log2) + (lane >> p.lg_log2);
    if (gi >= total_groups) continue;
    const uint32_t R = udiv(gi, p.gpr, p.gpr_magic);
    const uint32_t g = gi - R * p.gpr;
    int64_t e = 0, r = R;
    if (masked) {
      e = expert_of(prefix, static_cast<int>(p.experts), R);
      r = R - prefix[e];
    } else {
      e = R / p.m;
      r = R - e * p.m;
    }
    const int64_t off = (e * p.m + r) * p.k + (static_cast<int64_t>(g) << (p.lg_log2 + 4)) + kk * 16;
    uint32_t w[4];
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "l"(p.x + off));
    const float sc = p.x_scale[e * p.se + r * p.sm + static_cast<int64_t>(g) * p.sg];
    // (v * sc) * inv two codes at a time: mul.rn.f32x2 rounds each product like __fmul_rn
    const uint64_t sc2 = pk2(sc, sc), inv2 = pk2(inv, inv);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t c[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t f16x2;
        const uint16_t pair = static_cast<uint16_t>(w[i] >> (16 * h));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f16x2) : "h"(pair));
        c[h] = e4m3x2_pair(mul2(mul2(widen2<true>(f16x2), sc2), inv2));
      }
      o[i] = c[0] | (c[1] << 16);
    }
    st_128(p.out + off, o[0], o[1], o[2], o[3]);
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
// false when no shape fits.  PTGQ_PT_FORCE_BUFS / _WARPS restrict the choice (sweeps).
bool per_token_shape(int dtype, int64_t tokens, int64_t row_bytes, PtShape* out) {
  constexpr int64_t kMaxSmem = 227 * 1024;
  int64_t best_cost = -1, best_total = 0;
  for (int bufs = 2; bufs >= 1; --bufs) {
#ifdef PTGQ_PT_FORCE_BUFS
    if (bufs != PTGQ_PT_FORCE_BUFS) continue;
#endif
    const void* fn = per_token_smem_fn(dtype, bufs);
    for (int wc = 1; wc <= kWarps; ++wc) {
#ifdef PTGQ_PT_FORCE_WARPS
      if (wc != PTGQ_PT_FORCE_WARPS) continue;
#endif
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
  if (num_experts > 0 && m > 0 &&
      (num_experts * m > (int64_t(1) << 31) / (k / group_size) || m > (int64_t(1) << 31)))
    return PTGQ_ERR_TOO_LARGE;
  if (num_experts * m == 0) return PTGQ_OK;
  if (x == nullptr || x_scale == nullptr || output_scale == nullptr || out == nullptr)
    return PTGQ_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0 || reinterpret_cast<uintptr_t>(out) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(x_scale) % 4 != 0 || reinterpret_cast<uintptr_t>(output_scale) % 4 != 0 ||
      reinterpret_cast<uintptr_t>(masked_m) % 4 != 0)
    return PTGQ_ERR_ALIGN;
  RequantParams p{};
  p.x = static_cast<const uint8_t*>(x);
  p.x_scale = x_scale;
  p.masked_m = masked_m;
  p.output_scale = output_scale;
  p.out = static_cast<uint8_t*>(out);
  p.experts = num_experts;
  p.m = m;
  p.k = k;
  p.se = scale_stride_e;
  p.sm = scale_stride_m;
  p.sg = scale_stride_g;
  p.lg_log2 = static_cast<uint32_t>(__builtin_ctz(static_cast<unsigned>(group_size / 16)));
  p.gpr = static_cast<uint32_t>(k / group_size);
  p.gpr_magic = p.gpr == 1 ? 0xFFFFFFFFu : static_cast<uint32_t>((uint64_t(1) << 32) / p.gpr);
  const size_t smem = masked_m ? static_cast<size_t>(num_experts + 1) * sizeof(int32_t) : 0;
  const void* fn = reinterpret_cast<const void*>(&requant_kernel);
  const int64_t groups = num_experts * m * (k / group_size);
  const int64_t tasks = (groups * (group_size / 16) + 31) / 32;
  const int grid = grid_for(fn, smem, (tasks + kWarps - 1) / kWarps);
  if (grid < 0) return PTGQ_ERR_CUDA;
  void* args[] = {&p};
  return launch(fn, grid, smem, stream, args);
}
