// Decode kernel variants for head_dim 256, f32 storage, CUDA-core consumer:
// group tiles 1, 2, 4, 8.  A 2-stage ring (1 CTA/SM, 128 KB of pages in flight
// per SM): 3 stages measured slower on GB300.  Group tile 8 keeps 8 x 8 q and
// accumulator values per lane, so it runs four consumer warps (243 registers,
// no spills; eight warps capped at 168 spilled and ran 10% slower).
#include "kernel_variants.cuh"

namespace vt {

const VariantInfo* variants_d256_f32(int* count) {
  static const VariantInfo table[] = {
      Variant<256, float, 1, 8, 1, 2, Math::kSimt>::info(),
      Variant<256, float, 2, 8, 1, 2, Math::kSimt>::info(),
      Variant<256, float, 4, 8, 1, 2, Math::kSimt>::info(),
      Variant<256, float, 8, 4, 1, 2, Math::kSimt>::info(),
  };
  *count = 4;
  return table;
}

}  // namespace vt
