// Compile-time variants of the decode kernel and their launch descriptors.
#pragma once

#include "decode_kernel.cuh"

namespace vt {

struct VariantInfo {
  int head_dim;
  int tensor_cores;    // 1: mma.sync consumer (bf16 or fp8 K/V), 0: CUDA-core consumer
  int dtype;           // K/V storage: 0 bf16, 1 fp32, 2 FP8 E4M3 codes (bf16 q and out)
  int group_tile;      // G
  int consumer_warps;  // NCW
  int stages;          // NSTAGE
  int threads;
  int min_blocks;      // launch-bounds residency target
  size_t smem_bytes;   // dynamic shared memory (includes 1 KB alignment slack)
  const void* func;
  cudaError_t (*launch)(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& args, int grid,
                        cudaStream_t stream, bool overlap);
};

// Shared memory an SM offers (228 KB) less the 1 KB the hardware reserves per CTA.
constexpr size_t kSmemPerSm = 233472;
constexpr size_t kSmemReservedPerCta = 1024;

// Deepest ring (<= ST stages) whose CTA still fits MINB times on an SM; a
// multiple of the alternate-page pairs (Smem::NPAR).
template <int D, typename T, int G, int NCW, int MINB, Math M, int ST>
struct StagePick {
  static constexpr size_t bytes = sizeof(Smem<D, T, G, NCW, ST, M>) + 1024;
  static constexpr bool fits =
      (bytes + kSmemReservedPerCta) * MINB <= kSmemPerSm && ST % Smem<D, T, G, NCW, ST, M>::NPAR == 0;
  static constexpr int value = fits ? ST : StagePick<D, T, G, NCW, MINB, M, ST - 1>::value;
};
template <int D, typename T, int G, int NCW, int MINB, Math M>
struct StagePick<D, T, G, NCW, MINB, M, 0> {
  static constexpr int value = 0;
};

// Spare shared memory (bytes, multiple of 1024, at most 64 KB) a CTA with
// this ring still has within its share of the SM: the split-KV combine
// stages partial records into the ring plus these bytes.
template <int D, typename T, int G, int NCW, int MINB, Math M, int NSTAGE>
struct ExtPick {
  static constexpr size_t budget = kSmemPerSm / MINB - kSmemReservedPerCta - 1024;
  static constexpr size_t used = sizeof(Smem<D, T, G, NCW, NSTAGE, M, 0>) - 1024;  // without ext's own KB
  static constexpr size_t spare = budget > used ? (budget - used) / 1024 * 1024 : 0;
  static constexpr int value = static_cast<int>(spare < 65536 ? spare : 65536);
};

template <int D, typename T, int G, int NCW, int MINB, int MAXST, Math M>
struct Variant {
  static constexpr int NSTAGE = StagePick<D, T, G, NCW, MINB, M, MAXST>::value;
  static_assert(NSTAGE >= 2, "variant does not fit two stages in shared memory");
  static constexpr int EXT = ExtPick<D, T, G, NCW, MINB, M, NSTAGE>::value;
  using S = Smem<D, T, G, NCW, NSTAGE, M, EXT>;
  static constexpr size_t smem = sizeof(S) + 1024;
  static_assert((smem + kSmemReservedPerCta) * MINB <= kSmemPerSm, "variant does not fit its CTAs per SM");

  // overlap: launch as a programmatic dependent of the previous kernel on the
  // stream, so this grid's CTAs may start (and read context lengths and block
  // tables) while that kernel finishes.
  static cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& args, int grid,
                            cudaStream_t stream, bool overlap) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((NCW + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, T, G, NCW, NSTAGE, MINB, M, EXT>, tk, tv, args);
  }

  static VariantInfo info() {
    return VariantInfo{D,
                       M != Math::kSimt ? 1 : 0,
                       M == Math::kMma8 ? 2 : (sizeof(T) == 2 ? 0 : 1),
                       G,
                       NCW,
                       NSTAGE,
                       (NCW + 1) * 32,
                       MINB,
                       smem,
                       reinterpret_cast<const void*>(&paged_decode_kernel<D, T, G, NCW, NSTAGE, MINB, M, EXT>),
                       &launch};
  }
};

// One table per (head_dim, dtype); each defined in its own translation unit
// so the variants compile in parallel.
const VariantInfo* variants_d64_bf16(int* count);
const VariantInfo* variants_d64_f32(int* count);
const VariantInfo* variants_d128_bf16(int* count);
const VariantInfo* variants_d256_bf16(int* count);
const VariantInfo* variants_d512_bf16(int* count);
const VariantInfo* variants_d128_f32(int* count);
const VariantInfo* variants_d256_f32(int* count);
const VariantInfo* variants_d64_e4m3(int* count);
const VariantInfo* variants_d128_e4m3(int* count);
const VariantInfo* variants_d256_e4m3(int* count);

}  // namespace vt
