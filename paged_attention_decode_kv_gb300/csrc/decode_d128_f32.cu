// Decode kernel variants for head_dim 128, f32 storage, CUDA-core consumer:
// group tiles 1, 2, 4, 8.  Group tile 8 keeps 8 x 8 q and accumulator values
// per lane and runs one CTA per SM (236 registers, no spills; two CTAs cap a
// thread at 168 registers, which spilled and ran 8% slower).
#include "kernel_variants.cuh"

namespace vt {

const VariantInfo* variants_d128_f32(int* count) {
  static const VariantInfo table[] = {
      Variant<128, float, 1, 4, 2, 4, Math::kSimt>::info(),
      Variant<128, float, 2, 4, 2, 4, Math::kSimt>::info(),
      Variant<128, float, 4, 4, 2, 4, Math::kSimt>::info(),
      Variant<128, float, 8, 4, 1, 4, Math::kSimt>::info(),
  };
  *count = 4;
  return table;
}

}  // namespace vt
