// ptgq_inst_fp16.cu -- kernel instances for fp16 input (one translation unit per input
// type so the instances compile in parallel).
#include "ptgq_kernel.cuh"

namespace ptgq {

const void* kernel_for_fp16(int int8, int pow2, int silu) {
  static const void* const table[8] = {
      reinterpret_cast<const void*>(&quant_kernel<true, false, false, false>),
      reinterpret_cast<const void*>(&quant_kernel<true, false, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<true, false, true, false>),
      reinterpret_cast<const void*>(&quant_kernel<true, false, true, true>),
      reinterpret_cast<const void*>(&quant_kernel<true, true, false, false>),
      reinterpret_cast<const void*>(&quant_kernel<true, true, false, true>),
      reinterpret_cast<const void*>(&quant_kernel<true, true, true, false>),
      reinterpret_cast<const void*>(&quant_kernel<true, true, true, true>),
  };
  return table[(int8 ? 4 : 0) + (pow2 ? 2 : 0) + (silu ? 1 : 0)];
}

int table_bytes_fp16(int silu) { return silu ? SmemTables<true, true>::bytes : 0; }

}  // namespace ptgq
