// ptgq_inst_bf16_flat.cu -- kernel instances for bf16 input, flat scheduler (one translation
// unit per input type and scheduler, so the instances compile in parallel).
#include "ptgq_kernel.cuh"

namespace ptgq {

const void* kernel_for_bf16_flat(int int8, int fmt, int silu) {
  static const void* const table[16] = {
      reinterpret_cast<const void*>(&quant_kernel<false, false, 0, false, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 0, true, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 1, false, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 1, true, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 2, false, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 2, true, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 3, false, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 3, true, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 0, false, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 0, true, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 1, false, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 1, true, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 2, false, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 2, true, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 3, false, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 3, true, false>),
  };
  return table[(int8 ? 8 : 0) + fmt * 2 + (silu ? 1 : 0)];
}

const void* kernel_for_bf16_flat_light(int int8, int fmt) {
  static const void* const table[8] = {
      reinterpret_cast<const void*>(&quant_kernel<false, false, 0, false, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 1, false, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 2, false, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 3, false, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 0, false, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 1, false, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 2, false, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 3, false, false, true>),
  };
  return table[(int8 ? 4 : 0) + fmt];
}

const void* kernel_for_bf16_flat_light_pf(int int8, int fmt) {
  static const void* const table[8] = {
      reinterpret_cast<const void*>(&quant_kernel<false, false, 0, false, false, 2>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 1, false, false, 2>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 2, false, false, 2>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 3, false, false, 2>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 0, false, false, 2>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 1, false, false, 2>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 2, false, false, 2>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, 3, false, false, 2>),
  };
  return table[(int8 ? 4 : 0) + fmt];
}

int table_bytes_bf16(int silu) { return silu ? SmemTables<false, true>::bytes : 0; }

// e4m3 instances that vote on the amax range (eps below the fast arithmetic's range);
// fmt 0..2 (the fast-divide and int8 instances always vote).
const void* kernel_for_bf16_flat_checked(int fmt, int silu) {
  static const void* const table[6] = {
      reinterpret_cast<const void*>(&quant_kernel<false, false, 0, false, false, 0, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 0, true, false, 0, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 1, false, false, 0, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 1, true, false, 0, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 2, false, false, 0, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, 2, true, false, 0, true>),
  };
  return table[fmt * 2 + (silu ? 1 : 0)];
}

}  // namespace ptgq
