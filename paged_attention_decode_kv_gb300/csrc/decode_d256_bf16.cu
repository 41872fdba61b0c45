// Decode kernel variants for head_dim 256, bf16 storage, tensor-core (mma.sync) consumer:
// group tiles 8, 16.  Group tile 8 keeps a 3-stage ring (1 CTA/SM, 96 KB of
// pages in flight per SM): 4, 5 and 6 stages measured slower on GB300.
#include "kernel_variants.cuh"

namespace vt {

const VariantInfo* variants_d256_bf16(int* count) {
  static const VariantInfo table[] = {
      Variant<256, __nv_bfloat16, 8, 4, 1, 3, Math::kMma>::info(),
      Variant<256, __nv_bfloat16, 16, 4, 1, 6, Math::kMma>::info(),
  };
  *count = 2;
  return table;
}

}  // namespace vt
