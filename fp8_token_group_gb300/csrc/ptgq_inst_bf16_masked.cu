// ptgq_inst_bf16_masked.cu -- kernel instances for bf16 input, masked scheduler (one translation
// unit per input type and scheduler, so the instances compile in parallel).
#include "ptgq_kernel.cuh"

namespace ptgq {

const void* kernel_for_bf16_masked(int int8, int fmt, int silu) {
  static const void* const table[16] = {
      reinterpret_cast<const void*>(&quant_kernel<false, false, 0, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 0, true, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 1, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 1, true, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 2, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 2, true, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 3, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 3, true, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 0, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 0, true, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 1, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 1, true, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 2, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 2, true, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 3, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 3, true, true>),
  };
  return table[(int8 ? 8 : 0) + fmt * 2 + (silu ? 1 : 0)];
}

// e4m3 instances that vote on the amax range (eps below the fast arithmetic's range);
// fmt 0..2 (the fast-divide and int8 instances always vote).
const void* kernel_for_bf16_masked_checked(int fmt, int silu) {
  static const void* const table[6] = {
      reinterpret_cast<const void*>(&quant_kernel<false, false, 0, false, true, 0, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 0, true, true, 0, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 1, false, true, 0, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 1, true, true, 0, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 2, false, true, 0, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 2, true, true, 0, true>),
  };
  return table[fmt * 2 + (silu ? 1 : 0)];
}

}  // namespace ptgq
