// Decode kernel variants for head_dim 64: bf16 storage on the tensor-core
// (mma.sync) consumer, group tiles 8 and 16; fp32 storage on the CUDA-core
// consumer, group tiles 1, 2, 4, 8.  A 64-column page tile is 4 KB, so the
// bf16 ring is deeper (up to 8 stages) for the same bytes in flight.
#include "kernel_variants.cuh"

namespace vt {

const VariantInfo* variants_d64_bf16(int* count) {
  static const VariantInfo table[] = {
      Variant<64, __nv_bfloat16, 8, 4, 3, 8, Math::kMma>::info(),
      Variant<64, __nv_bfloat16, 16, 4, 2, 8, Math::kMma>::info(),
  };
  *count = 2;
  return table;
}

const VariantInfo* variants_d64_f32(int* count) {
  static const VariantInfo table[] = {
      Variant<64, float, 1, 4, 2, 6, Math::kSimt>::info(),
      Variant<64, float, 2, 4, 2, 6, Math::kSimt>::info(),
      Variant<64, float, 4, 4, 2, 6, Math::kSimt>::info(),
      Variant<64, float, 8, 4, 1, 6, Math::kSimt>::info(),
  };
  *count = 4;
  return table;
}

}  // namespace vt
