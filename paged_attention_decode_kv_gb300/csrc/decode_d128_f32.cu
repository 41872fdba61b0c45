// Decode kernel variants for head_dim 128, f32 storage, CUDA-core consumer:
// group tiles 1, 2, 4, 8.
#include "kernel_variants.cuh"

namespace vt {

const VariantInfo* variants_d128_f32(int* count) {
  static const VariantInfo table[] = {
      Variant<128, float, 1, 4, 2, 4, Math::kSimt>::info(),
      Variant<128, float, 2, 4, 2, 4, Math::kSimt>::info(),
      Variant<128, float, 4, 4, 2, 4, Math::kSimt>::info(),
      Variant<128, float, 8, 4, 2, 4, Math::kSimt>::info(),
  };
  *count = 4;
  return table;
}

}  // namespace vt
