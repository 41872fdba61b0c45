// Decode kernel variant for head_dim 512, bf16 storage, tensor-core (mma.sync)
// consumer: group tile 8 (larger groups run as several query subgroups).  A
// page tile is 32 KB per K or V, so the CTA holds a 2-stage ring and is alone
// on its SM; eight consumer warps split the head_dim four ways for PV, and
// the Q^T fragments come from shared memory (see Smem::qs).
#include "kernel_variants.cuh"

namespace vt {

const VariantInfo* variants_d512_bf16(int* count) {
  static const VariantInfo table[] = {
      Variant<512, __nv_bfloat16, 8, 8, 1, 2, Math::kMma>::info(),
  };
  *count = 1;
  return table;
}

}  // namespace vt
