// ptgq_inst_bf16.cu -- kernel instances for bf16 input (one translation unit per input
// type so the instances compile in parallel).
#include "ptgq_kernel.cuh"

namespace ptgq {

const void* kernel_for_bf16(int int8, int pow2, int silu) {
  static const void* const table[8] = {
      reinterpret_cast<const void*>(&quant_kernel<false, false, false, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, true, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, false, true, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, false, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, true, false>),
      reinterpret_cast<const void*>(&quant_kernel<false, true, true, true>),
  };
  return table[(int8 ? 4 : 0) + (pow2 ? 2 : 0) + (silu ? 1 : 0)];
}

int table_bytes_bf16(int silu) { return silu ? SmemTables<false, true>::bytes : 0; }

}  // namespace ptgq
