// Compile-time variants of the decode kernel and their launch descriptors.
#pragma once

#include "decode_kernel.cuh"

namespace vt {

struct VariantInfo {
  int head_dim;
  int dtype;           // 0 bf16, 1 fp32
  int group_tile;      // G
  int consumer_warps;  // NCW
  int stages;          // NSTAGE
  int threads;
  int min_blocks;      // launch-bounds residency target
  size_t smem_bytes;   // dynamic shared memory (includes 1 KB alignment slack)
  const void* func;
  cudaError_t (*launch)(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& args, int grid,
                        cudaStream_t stream);
};

// Shared memory an SM offers (228 KB) less the 1 KB the hardware reserves per CTA.
constexpr size_t kSmemPerSm = 233472;
constexpr size_t kSmemReservedPerCta = 1024;

// Deepest ring (<= ST stages) whose CTA still fits MINB times on an SM.
template <int D, typename T, int G, int NCW, int MINB, int ST>
struct StagePick {
  static constexpr size_t bytes = sizeof(Smem<D, T, G, NCW, ST>) + 1024;
  static constexpr int value =
      (bytes + kSmemReservedPerCta) * MINB <= kSmemPerSm ? ST : StagePick<D, T, G, NCW, MINB, ST - 1>::value;
};
template <int D, typename T, int G, int NCW, int MINB>
struct StagePick<D, T, G, NCW, MINB, 0> {
  static constexpr int value = 0;
};

template <int D, typename T, int G, int NCW, int MINB, int MAXST>
struct Variant {
  static constexpr int NSTAGE = StagePick<D, T, G, NCW, MINB, MAXST>::value;
  static_assert(NSTAGE >= 2, "variant does not fit two stages in shared memory");
  using S = Smem<D, T, G, NCW, NSTAGE>;
  static constexpr size_t smem = sizeof(S) + 1024;

  static cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& args, int grid,
                            cudaStream_t stream) {
    paged_decode_kernel<D, T, G, NCW, NSTAGE, MINB><<<grid, (NCW + 1) * 32, smem, stream>>>(tk, tv, args);
    return cudaGetLastError();
  }

  static VariantInfo info() {
    return VariantInfo{D,
                       sizeof(T) == 2 ? 0 : 1,
                       G,
                       NCW,
                       NSTAGE,
                       (NCW + 1) * 32,
                       MINB,
                       smem,
                       reinterpret_cast<const void*>(&paged_decode_kernel<D, T, G, NCW, NSTAGE, MINB>),
                       &launch};
  }
};

// One table per (head_dim, dtype); each defined in its own translation unit
// so the variants compile in parallel.
const VariantInfo* variants_d128_bf16(int* count);
const VariantInfo* variants_d256_bf16(int* count);
const VariantInfo* variants_d128_f32(int* count);
const VariantInfo* variants_d256_f32(int* count);

}  // namespace vt
