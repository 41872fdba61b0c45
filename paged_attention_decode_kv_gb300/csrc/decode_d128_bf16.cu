// Decode kernel variants for head_dim 128, bf16 storage, tensor-core (mma.sync) consumer:
// group tiles 8, 16.  Group tile 8 keeps a 4-stage ring (2 CTAs/SM, 128 KB of
// pages in flight per SM): 3, 5 and 6 stages measured slower on GB300 (deeper
// rings queue more requests at HBM without streaming faster).
#include "kernel_variants.cuh"

namespace vt {

const VariantInfo* variants_d128_bf16(int* count) {
  static const VariantInfo table[] = {
      Variant<128, __nv_bfloat16, 8, 4, 2, 4, Math::kMma>::info(),
      Variant<128, __nv_bfloat16, 16, 4, 2, 6, Math::kMma>::info(),
  };
  *count = 2;
  return table;
}

}  // namespace vt
