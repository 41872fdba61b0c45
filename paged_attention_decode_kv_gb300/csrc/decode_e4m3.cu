// Decode kernel variants for an FP8 (E4M3) K/V cache with per-kv-head scales,
// bf16 queries and output: tensor-core consumer (codes widened to f16 in
// registers, mma.sync f16), group tiles 8 and 16, head_dim 64, 128 and 256.  A
// page tile is half the bytes of bf16, so the rings are deeper for the same
// bytes in flight.
#include "kernel_variants.cuh"

namespace vt {

const VariantInfo* variants_d64_e4m3(int* count) {
  static const VariantInfo table[] = {
      Variant<64, __nv_bfloat16, 8, 4, 3, 8, Math::kMma8>::info(),
      Variant<64, __nv_bfloat16, 16, 4, 2, 8, Math::kMma8>::info(),
  };
  *count = 2;
  return table;
}

const VariantInfo* variants_d128_e4m3(int* count) {
  static const VariantInfo table[] = {
      Variant<128, __nv_bfloat16, 8, 4, 2, 8, Math::kMma8>::info(),
      Variant<128, __nv_bfloat16, 16, 4, 2, 8, Math::kMma8>::info(),
  };
  *count = 2;
  return table;
}

const VariantInfo* variants_d256_e4m3(int* count) {
  static const VariantInfo table[] = {
      Variant<256, __nv_bfloat16, 8, 4, 1, 6, Math::kMma8>::info(),
      Variant<256, __nv_bfloat16, 16, 4, 1, 6, Math::kMma8>::info(),
  };
  *count = 2;
  return table;
}

}  // namespace vt
