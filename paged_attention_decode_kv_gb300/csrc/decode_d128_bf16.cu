// Decode kernel variants for head_dim 128, bf16 storage: group tiles 1, 2, 4, 8.
#include "kernel_variants.cuh"

namespace vt {

const VariantInfo* variants_d128_bf16(int* count) {
  static const VariantInfo table[] = {
      Variant<128, __nv_bfloat16, 1, 4, 2, 6>::info(),
      Variant<128, __nv_bfloat16, 2, 4, 2, 6>::info(),
      Variant<128, __nv_bfloat16, 4, 4, 2, 6>::info(),
      Variant<128, __nv_bfloat16, 8, 4, 2, 6>::info(),
  };
  *count = 4;
  return table;
}

}  // namespace vt
