// C-ABI front end of the paged decode library: argument validation, launch
// plan, the split scratch (library-owned, caller-owned or static), TMA
// descriptors, launch, and the device status word.
//
// Every decode entry point goes through the same three steps, so they cannot
// drift apart: validate() checks the arguments, make_plan() picks the kernel
// variant and the grid, launch() encodes the tensor maps, fills the kernel
// arguments and records the plan.  The entry points differ only in where the
// split scratch comes from.
//
// Declarations and the contract of every entry point: include/vt_paged_attn.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/vt_paged_attn.h"
#include "kernel_variants.cuh"

namespace {

using vt::DecodeArgs;
using vt::VariantInfo;

constexpr int kVersion = 10100;  // 1.1.0
constexpr int kMaxGroupTile = 8;
constexpr int kDefaultMinUnits = 2;
// A segment boundary weighs about two tiles of bf16 or fp32 streaming; an FP8
// tile (half the bytes) or a multi-token one (a longer epilogue per boundary)
// is worth less against it: measured best at six.
constexpr int kDefaultSegCost = 2;
constexpr int kDefaultSegCostFp8OrMulti = 6;
constexpr size_t kStatusBytes = 256;

thread_local int g_override_grid = 0;
thread_local bool g_overlap = false;
thread_local int g_override_min_units = 0;
thread_local int g_seg_cost = -1;  // < 0: default
thread_local long long g_test_wait_limit = 0;  // <= 0: kWaitLimitCycles
thread_local int g_test_withhold_cta = -1;
thread_local int g_test_withhold_tile = -1;
thread_local vt_plan g_last_plan{};
thread_local bool g_have_plan = false;
thread_local std::string g_last_cuda_error;

vt_status cuda_fail(cudaError_t e, const char* where) {
  g_last_cuda_error = std::string(where) + ": " + cudaGetErrorString(e);
  return VT_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Variant lookup
// ---------------------------------------------------------------------------
const VariantInfo* find_variant(int head_dim, vt_dtype dtype, int group_tile) {
  int n = 0;
  const VariantInfo* table = nullptr;
  if (head_dim == 64 && dtype == VT_BF16) table = vt::variants_d64_bf16(&n);
  if (head_dim == 64 && dtype == VT_F32) table = vt::variants_d64_f32(&n);
  if (head_dim == 128 && dtype == VT_BF16) table = vt::variants_d128_bf16(&n);
  if (head_dim == 256 && dtype == VT_BF16) table = vt::variants_d256_bf16(&n);
  if (head_dim == 512 && dtype == VT_BF16) table = vt::variants_d512_bf16(&n);
  if (head_dim == 128 && dtype == VT_F32) table = vt::variants_d128_f32(&n);
  if (head_dim == 256 && dtype == VT_F32) table = vt::variants_d256_f32(&n);
  if (head_dim == 64 && dtype == VT_E4M3) table = vt::variants_d64_e4m3(&n);
  if (head_dim == 128 && dtype == VT_E4M3) table = vt::variants_d128_e4m3(&n);
  if (head_dim == 256 && dtype == VT_E4M3) table = vt::variants_d256_e4m3(&n);
  for (int k = 0; k < n; ++k)
    if (table[k].group_tile == group_tile) return &table[k];
  return nullptr;
}

// Query rows computed per kv head and CTA.  bf16 runs on tensor cores with
// the queries as the N dimension of m16n8k16: one tile of 8 (or 16) rows
// covers any group up to that size (head_dim 512: 8, larger groups become
// query subgroups).  fp32 runs on CUDA cores, where every padded row costs
// FMAs: the next power of two, at most 8.
int group_tile_for(int group, vt_dtype dtype, int head_dim) {
  if (dtype != VT_F32) return (group <= 8 || head_dim >= 512) ? 8 : 16;
  int g = 1;
  while (g < group && g < kMaxGroupTile) g <<= 1;
  return g;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Split scratch layout: [status words (256 B) | arrival counters | partial
// records].  Arrival counters are zero between calls (every kernel leaves
// them so; vt_paged_attn_device_status clears them after a give-up), so the
// region that held counters must never receive partials: partials start
// after the largest counter region the scratch has served.
struct WsNeed {
  size_t counters_bytes;  // counters this call uses
  size_t part_bytes;      // partial records: per row (m, l, 0, 0), then the rows
};

WsNeed ws_need(int num_seqs, int nvh, int grid, int group_tile, int head_dim) {
  WsNeed n;
  n.counters_bytes = static_cast<size_t>(num_seqs) * nvh * sizeof(int);
  const size_t slots = 2 * static_cast<size_t>(grid);
  n.part_bytes = slots * group_tile * (4 + head_dim) * sizeof(float);
  return n;
}

size_t ws_total(const WsNeed& n) { return kStatusBytes + align_up(n.counters_bytes, 256) + n.part_bytes; }

struct Scratch {
  char* base = nullptr;
  size_t bytes = 0;
  size_t counters_cap = 0;  // bytes after the status words that hold zeroed counters
};

// ---------------------------------------------------------------------------
// Per-device state
// ---------------------------------------------------------------------------
struct DeviceState {
  bool init = false;
  int num_sms = 0;
  Scratch lib;               // library-owned (cudaMallocAsync, grows)
  Scratch user;              // caller-owned (vt_paged_attn_set_workspace)
  char* noalloc = nullptr;   // device address of the static array, once looked up
  std::vector<std::pair<const void*, int>> occupancy;
};

std::mutex g_mutex;
std::vector<DeviceState> g_devices;

DeviceState& device_state(int dev) {
  if (static_cast<int>(g_devices.size()) <= dev) g_devices.resize(dev + 1);
  return g_devices[dev];
}

vt_status prepare_device(int dev, DeviceState& ds) {
  if (ds.init) return VT_OK;
  int sms = 0;
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  ds.num_sms = sms;
  ds.init = true;
  return VT_OK;
}

vt_status prepare_variant(DeviceState& ds, const VariantInfo& v, int* ctas_per_sm) {
  for (auto& p : ds.occupancy)
    if (p.first == v.func) {
      *ctas_per_sm = p.second;
      return VT_OK;
    }
  cudaError_t e = cudaFuncSetAttribute(v.func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(v.smem_bytes));
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, v.func, v.threads, v.smem_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  if (n < 1) {
    g_last_cuda_error = "decode kernel variant cannot be resident on this device";
    return VT_ERR_UNSUPPORTED;
  }
  ds.occupancy.emplace_back(v.func, n);
  *ctas_per_sm = n;
  return VT_OK;
}

// Library-owned scratch: grows (never shrinks).  A new buffer's status words
// and counter region are zeroed on `stream` before any kernel uses them.
vt_status ensure_library_scratch(Scratch& w, const WsNeed& n, cudaStream_t stream) {
  if (w.base && w.counters_cap >= n.counters_bytes &&
      w.bytes - kStatusBytes - w.counters_cap >= n.part_bytes)
    return VT_OK;
  const size_t old_part = w.base ? w.bytes - kStatusBytes - w.counters_cap : 0;
  size_t counters = w.counters_cap > n.counters_bytes ? w.counters_cap : n.counters_bytes;
  counters = align_up(counters + counters / 4 + 1024, 256);
  size_t partial = old_part > n.part_bytes ? old_part : n.part_bytes;
  partial = align_up(partial + partial / 4, 1 << 16);
  const size_t bytes = kStatusBytes + counters + partial;
  if (w.base) {
    cudaError_t e = cudaFreeAsync(w.base, stream);
    w = Scratch{};
    if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync");
  }
  void* p = nullptr;
  cudaError_t e = cudaMallocAsync(&p, bytes, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    g_last_cuda_error = std::string("cudaMallocAsync: ") + cudaGetErrorString(e);
    return VT_ERR_OOM;
  }
  e = cudaMemsetAsync(p, 0, kStatusBytes + counters, stream);
  if (e != cudaSuccess) {
    cudaFreeAsync(p, stream);
    return cuda_fail(e, "cudaMemsetAsync");
  }
  w.base = static_cast<char*>(p);
  w.bytes = bytes;
  w.counters_cap = counters;
  return VT_OK;
}

// Caller-owned scratch of fixed size: the counter region grows in place (its
// new part zeroed on `stream`, ahead of the kernel) as long as the buffer
// holds it and the call's partials after it.
vt_status fit_user_scratch(Scratch& w, const WsNeed& n, cudaStream_t stream) {
  const size_t counters = align_up(n.counters_bytes, 256);
  const size_t cap = counters > w.counters_cap ? counters : w.counters_cap;
  const size_t total = kStatusBytes + cap + n.part_bytes;
  if (total > w.bytes) {
    g_last_cuda_error = "vt_paged_attn_decode: this call needs " + std::to_string(total) +
                        " bytes of workspace; the caller's workspace holds " + std::to_string(w.bytes);
    return VT_ERR_SCRATCH_LIMIT;
  }
  if (cap > w.counters_cap) {
    cudaError_t e = cudaMemsetAsync(w.base + kStatusBytes + w.counters_cap, 0, cap - w.counters_cap, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    w.counters_cap = cap;
  }
  return VT_OK;
}

// ---------------------------------------------------------------------------
// TMA descriptors: tiled views of a page pool (4-D for bf16, 3-D for fp32).
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct MapKey {
  const void* ptr;
  int head_dim, num_kv_heads, num_blocks, dtype, device;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && head_dim == o.head_dim && num_kv_heads == o.num_kv_heads &&
           num_blocks == o.num_blocks && dtype == o.dtype && device == o.device;
  }
};

struct MapCache {
  static constexpr int kSlots = 16;
  MapKey key[kSlots];
  CUtensorMap map[kSlots];
  int used = 0, next = 0;
};
thread_local MapCache g_maps;

vt_status tensor_map(const MapKey& k, CUtensorMap* out) {
  for (int i = 0; i < g_maps.used; ++i)
    if (g_maps.key[i] == k) {
      *out = g_maps.map[i];
      return VT_OK;
    }
  auto fn = encode_fn();
  if (!fn) {
    g_last_cuda_error = "cuTensorMapEncodeTiled entry point unavailable";
    return VT_ERR_CUDA;
  }
  const size_t es = k.dtype == VT_BF16 ? 2 : (k.dtype == VT_E4M3 ? 1 : 4);
  const cuuint64_t tokens = static_cast<cuuint64_t>(k.num_blocks) * vt::kPageTokens;
  const cuuint64_t row = static_cast<cuuint64_t>(k.head_dim) * k.num_kv_heads * es;  // bytes per token
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  // L2 promotion no wider than one head's token row: a 128-byte row (FP8 at
  // head_dim 128, bf16 at 64) promoted to 256 bytes would also pull the next
  // kv head's row, which another CTA reads at another time.
  const CUtensorMapL2promotion promo =
      static_cast<size_t>(k.head_dim) * es <= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  CUtensorMap m;
  CUresult r;
  if (k.dtype == VT_E4M3) {
    // FP8 consumer: the same 4-D view as bf16 over bytes, column blocks of
    // 128 codes (one 128-byte swizzle row) at head_dim 128 or 256, one block
    // of 64 codes with the 64-byte swizzle at head_dim 64.
    const cuuint64_t kCols = k.head_dim >= 128 ? 128 : 64;
    const cuuint64_t dims[4] = {kCols, tokens, static_cast<cuuint64_t>(k.head_dim) / kCols,
                                static_cast<cuuint64_t>(k.num_kv_heads)};
    const cuuint64_t strides[3] = {row, kCols, static_cast<cuuint64_t>(k.head_dim)};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(kCols), static_cast<cuuint32_t>(vt::kPageTokens),
                               static_cast<cuuint32_t>(k.head_dim / kCols), 1u};
    r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(k.ptr), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, kCols == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
           promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else if (k.dtype == VT_BF16) {
    // Tensor-core consumer: a 4-D view (64 columns, token, column block, kv
    // head) so one box brings a whole [32 tokens][head_dim] tile of one head,
    // stored as head_dim/64 sub-tiles of [token][64 columns] with the 128-byte
    // swizzle (bank-conflict-free ldmatrix reads).
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(vt::kSwizzleCols), tokens,
                                static_cast<cuuint64_t>(k.head_dim / vt::kSwizzleCols),
                                static_cast<cuuint64_t>(k.num_kv_heads)};
    const cuuint64_t strides[3] = {row, static_cast<cuuint64_t>(vt::kSwizzleCols) * es,
                                   static_cast<cuuint64_t>(k.head_dim) * es};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(vt::kSwizzleCols), static_cast<cuuint32_t>(vt::kPageTokens),
                               static_cast<cuuint32_t>(k.head_dim / vt::kSwizzleCols), 1u};
    r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(k.ptr), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    // CUDA-core consumer: a 3-D view (column, kv head, token) and one
    // unswizzled box of head_dim x 32 tokens.
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(k.head_dim), static_cast<cuuint64_t>(k.num_kv_heads), tokens};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(k.head_dim) * es, row};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(k.head_dim), 1u, static_cast<cuuint32_t>(vt::kPageTokens)};
    r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(k.ptr), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, promo,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) {
    g_last_cuda_error = "cuTensorMapEncodeTiled failed (code " + std::to_string(static_cast<int>(r)) + ")";
    return VT_ERR_CUDA;
  }
  const int slot = g_maps.next;
  g_maps.key[slot] = k;
  g_maps.map[slot] = m;
  g_maps.next = (slot + 1) % MapCache::kSlots;
  if (g_maps.used < MapCache::kSlots) ++g_maps.used;
  *out = m;
  return VT_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------------------
// The shared call path
// ---------------------------------------------------------------------------
struct Call {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
  float scale;
  int window;
  cudaStream_t stream;
  int max_blocks_per_seq, num_blocks;
  vt_dtype dtype;                  // K/V storage (VT_E4M3: bf16 q and out)
  const float* k_scale = nullptr;  // VT_E4M3 only: [num_kv_heads] dequantisation scales
  const float* v_scale = nullptr;
  int q_len = 1;                   // new tokens per sequence (vt_paged_attn_decode_multi)
};

struct Plan {
  const VariantInfo* v = nullptr;
  int dev = 0, grid = 0, per_sm = 0, min_units = 0, num_sms = 0;
  int group = 0, rows = 0, gt = 0, subgroups = 0;
  long long nvh = 0;
  WsNeed need{};
};

// Argument checks that need no device: every error returns before any
// launch.  (num_seqs == 0 is handled by the caller as a no-op.)
vt_status validate(const Call& c) {
  if (c.num_seqs < 0 || c.q_len < 1) return VT_ERR_INVALID_ARG;
  if (!c.out || !c.q || !c.k_cache || !c.v_cache || !c.block_tables || !c.context_lens) return VT_ERR_INVALID_ARG;
  if (c.dtype != VT_BF16 && c.dtype != VT_F32 && c.dtype != VT_E4M3) return VT_ERR_INVALID_ARG;
  // an FP8 cache comes with its scales, and only through vt_paged_attn_decode_fp8
  if ((c.dtype == VT_E4M3) != (c.k_scale != nullptr) || (c.k_scale == nullptr) != (c.v_scale == nullptr))
    return VT_ERR_INVALID_ARG;
  if (c.k_scale && (!aligned(c.k_scale, 4) || !aligned(c.v_scale, 4))) return VT_ERR_INVALID_ARG;
  if (c.num_q_heads <= 0 || c.num_kv_heads <= 0 || c.num_q_heads % c.num_kv_heads != 0) return VT_ERR_INVALID_ARG;
  if (c.max_blocks_per_seq <= 0 || c.num_blocks <= 0 || c.block_size <= 0 || c.head_dim <= 0)
    return VT_ERR_INVALID_ARG;
  if (!std::isfinite(c.scale)) return VT_ERR_INVALID_ARG;
  if (!aligned(c.out, 16) || !aligned(c.q, 16) || !aligned(c.k_cache, 16) || !aligned(c.v_cache, 16) ||
      !aligned(c.block_tables, 4) || !aligned(c.context_lens, 4))
    return VT_ERR_INVALID_ARG;
  if (c.head_dim != 64 && c.head_dim != 128 && c.head_dim != 256 && c.head_dim != 512) return VT_ERR_UNSUPPORTED;
  if (c.dtype == VT_E4M3 && c.head_dim == 512) return VT_ERR_UNSUPPORTED;
  if (c.dtype == VT_F32 && c.head_dim == 512) return VT_ERR_UNSUPPORTED;
  if (c.block_size != vt::kPageTokens) return VT_ERR_UNSUPPORTED;
  if (static_cast<long long>(c.num_blocks) * vt::kPageTokens > 0x7fffffffLL) return VT_ERR_UNSUPPORTED;
  if (static_cast<long long>(c.max_blocks_per_seq) * vt::kPageTokens > 0x7fffffffLL) return VT_ERR_UNSUPPORTED;
  return VT_OK;
}

// Variant, grid and scratch need of a validated call on the current device.
// Caller holds g_mutex.
vt_status make_plan(const Call& c, Plan* p) {
  p->group = c.num_q_heads / c.num_kv_heads;
  const long long rows = static_cast<long long>(p->group) * c.q_len;  // query rows per kv head
  if (rows > 4096) return VT_ERR_UNSUPPORTED;
  p->rows = static_cast<int>(rows);
  p->gt = group_tile_for(p->rows, c.dtype, c.head_dim);
  p->subgroups = (p->rows + p->gt - 1) / p->gt;
  p->nvh = static_cast<long long>(c.num_kv_heads) * p->subgroups;
  if (p->nvh * c.num_seqs > 0x7fffffffLL) return VT_ERR_UNSUPPORTED;
  p->v = find_variant(c.head_dim, c.dtype, p->gt);
  if (!p->v) return VT_ERR_UNSUPPORTED;
  cudaError_t e = cudaGetDevice(&p->dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DeviceState& ds = device_state(p->dev);
  vt_status st = prepare_device(p->dev, ds);
  if (st != VT_OK) return st;
  st = prepare_variant(ds, *p->v, &p->per_sm);
  if (st != VT_OK) return st;
  p->num_sms = ds.num_sms;
  p->grid = g_override_grid > 0 ? g_override_grid : ds.num_sms * p->per_sm;
  p->min_units = g_override_min_units > 0 ? g_override_min_units : kDefaultMinUnits;
  p->need = ws_need(c.num_seqs, static_cast<int>(p->nvh), p->grid, p->gt, c.head_dim);
  return VT_OK;
}

// Encodes the tensor maps, fills the kernel arguments from the plan and the
// chosen scratch (status words at `base`, counters after them, partials at
// `base + 256 + counters_region`), launches, and records the plan.
vt_status launch(const Call& c, const Plan& p, char* base, size_t counters_region, size_t scratch_used,
                 int scratch_source) {
  CUtensorMap tk, tv;
  vt_status st = tensor_map(MapKey{c.k_cache, c.head_dim, c.num_kv_heads, c.num_blocks, c.dtype, p.dev}, &tk);
  if (st != VT_OK) return st;
  st = tensor_map(MapKey{c.v_cache, c.head_dim, c.num_kv_heads, c.num_blocks, c.dtype, p.dev}, &tv);
  if (st != VT_OK) return st;

  DecodeArgs args{};
  args.status = reinterpret_cast<unsigned*>(base);
  args.counters = reinterpret_cast<int*>(base + kStatusBytes);
  args.part = reinterpret_cast<float*>(base + kStatusBytes + counters_region);
  args.out = c.out;
  args.q = c.q;
  args.block_tables = c.block_tables;
  args.context_lens = c.context_lens;
  args.num_seqs = c.num_seqs;
  args.num_q_heads = c.num_q_heads;
  args.num_kv_heads = c.num_kv_heads;
  args.q_len = c.q_len;
  args.rows = p.rows;
  args.group = p.group;
  args.subgroups = p.subgroups;
  args.max_blocks = c.max_blocks_per_seq;
  args.num_blocks = c.num_blocks;
  args.window = c.window > 0 ? c.window : 0;
  args.scale_log2 = c.scale * 1.4426950408889634f;
  args.min_units = p.min_units;
  args.seg_cost = g_seg_cost >= 0 ? g_seg_cost
                 : (c.dtype == VT_E4M3 || c.q_len > 1) ? kDefaultSegCostFp8OrMulti
                                                       : kDefaultSegCost;
  args.wait_limit = g_test_wait_limit > 0 ? g_test_wait_limit : vt::kWaitLimitCycles;
  args.withhold_cta = g_test_withhold_tile >= 0 ? g_test_withhold_cta : -1;
  args.withhold_tile = g_test_withhold_tile;
  args.k_scale = c.k_scale;
  args.v_scale = c.v_scale;

  cudaError_t e = p.v->launch(tk, tv, args, p.grid, c.stream, g_overlap);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");

  vt_plan& r = g_last_plan;
  r.grid_ctas = p.grid;
  r.ctas_per_sm = p.per_sm;
  r.num_sms = p.num_sms;
  r.consumer_warps = p.v->consumer_warps;
  r.tensor_cores = p.v->tensor_cores;
  r.stages = p.v->stages;
  r.group_tile = p.gt;
  r.subgroups = p.subgroups;
  r.min_units_per_cta = p.min_units;
  r.head_dim = c.head_dim;
  r.dtype = c.dtype;
  r.smem_bytes = p.v->smem_bytes;
  r.workspace_bytes = scratch_used;
  r.launch_overlap = g_overlap ? 1 : 0;
  r.segment_cost = args.seg_cost;
  r.scratch_source = scratch_source;
  r.q_len = c.q_len;
  g_have_plan = true;
  return VT_OK;
}

Call make_call(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
               const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
               int block_size, float scale, int window, vt_stream_t stream, int max_blocks_per_seq,
               int num_blocks, vt_dtype dtype) {
  return Call{out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
              head_dim, block_size, scale, window, reinterpret_cast<cudaStream_t>(stream), max_blocks_per_seq,
              num_blocks, dtype, nullptr, nullptr, 1};
}

// ---------------------------------------------------------------------------
// Allocation-free variant: the split scratch is a fixed, file-scope device
// array instead of the library's lazily allocated per-device workspace.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = VT_NOALLOC_SCRATCH_BYTES;  // held on every device that loads the library
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// In host code the array's name is only a host-side stand-in: its device
// address must be looked up, once per device, with that device current.
// Caller holds g_mutex.
vt_status noalloc_scratch(DeviceState& ds, char** ptr) {
  if (!ds.noalloc) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
    ds.noalloc = static_cast<char*>(p);
  }
  *ptr = ds.noalloc;
  return VT_OK;
}

// The status areas a kernel on this device may have written, library-owned
// scratch first.  Caller holds g_mutex.
std::vector<std::pair<char*, size_t>> status_areas(DeviceState& ds) {
  std::vector<std::pair<char*, size_t>> areas;  // (base, bytes to clear on a give-up)
  if (ds.lib.base) areas.emplace_back(ds.lib.base, kStatusBytes + ds.lib.counters_cap);
  if (ds.user.base) areas.emplace_back(ds.user.base, kStatusBytes + ds.user.counters_cap);
  if (ds.noalloc) areas.emplace_back(ds.noalloc, kStatusBytes);  // its calls clear their counters themselves
  return areas;
}

}  // namespace

extern "C" {

const char* vt_status_string(vt_status s) {
  switch (s) {
    case VT_OK: return "ok";
    case VT_ERR_INVALID_ARG: return "invalid argument";
    case VT_ERR_UNSUPPORTED: return "unsupported configuration";
    case VT_ERR_CUDA: return "CUDA error";
    case VT_ERR_OOM: return "out of device memory";
    case VT_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case VT_ERR_SCRATCH_LIMIT: return "call needs more scratch than the fixed buffer (static or caller's) holds";
  }
  return "unknown status";
}

const char* vt_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

int vt_paged_attn_version(void) { return kVersion; }

vt_status vt_paged_attn_set_override(int grid_ctas, int min_units_per_cta) {
  if (grid_ctas < 0 || min_units_per_cta < 0) return VT_ERR_INVALID_ARG;
  g_override_grid = grid_ctas;
  g_override_min_units = min_units_per_cta;
  return VT_OK;
}

vt_status vt_paged_attn_set_overlap(int enabled) {
  if (enabled != 0 && enabled != 1) return VT_ERR_INVALID_ARG;
  g_overlap = enabled != 0;
  return VT_OK;
}

vt_status vt_paged_attn_set_segment_cost(int tiles) {
  if (tiles > 64) return VT_ERR_INVALID_ARG;
  g_seg_cost = tiles;
  return VT_OK;
}

vt_status vt_paged_attn_set_test_wait(long long wait_limit_cycles, int withhold_cta, int withhold_tile) {
  if (withhold_tile >= 0 && withhold_cta < 0) return VT_ERR_INVALID_ARG;
  g_test_wait_limit = wait_limit_cycles > 0 ? wait_limit_cycles : 0;
  g_test_withhold_cta = withhold_tile >= 0 ? withhold_cta : -1;
  g_test_withhold_tile = withhold_tile >= 0 ? withhold_tile : -1;
  return VT_OK;
}

vt_status vt_paged_attn_last_plan(vt_plan* plan) {
  if (!plan) return VT_ERR_INVALID_ARG;
  if (!g_have_plan) return VT_ERR_INVALID_ARG;
  *plan = g_last_plan;
  return VT_OK;
}

size_t vt_paged_attn_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                     vt_dtype dtype) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return 0;
  const int group = num_q_heads / num_kv_heads;
  const int gt = group_tile_for(group, dtype, head_dim);
  const VariantInfo* v = find_variant(head_dim, dtype, gt);
  if (!v) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& ds = device_state(dev);
  if (prepare_device(dev, ds) != VT_OK) return 0;
  int per_sm = 0;
  if (prepare_variant(ds, *v, &per_sm) != VT_OK) return 0;
  const int grid = g_override_grid > 0 ? g_override_grid : ds.num_sms * per_sm;
  const int nvh = num_kv_heads * ((group + gt - 1) / gt);
  return ws_total(ws_need(num_seqs, nvh, grid, gt, head_dim));
}

vt_status vt_paged_attn_set_workspace(void* dev_ptr, size_t bytes, vt_stream_t stream_handle) {
  if (dev_ptr && (!aligned(dev_ptr, 256) || bytes < VT_MIN_WORKSPACE_BYTES)) return VT_ERR_INVALID_ARG;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& ds = device_state(dev);
  if (!dev_ptr) {
    ds.user = Scratch{};
    return VT_OK;
  }
  e = cudaMemsetAsync(dev_ptr, 0, kStatusBytes, reinterpret_cast<cudaStream_t>(stream_handle));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  ds.user = Scratch{static_cast<char*>(dev_ptr), bytes, 0};
  return VT_OK;
}

}  // extern "C"

namespace {

// A call on the device's workspace: the caller's (vt_paged_attn_set_workspace)
// when one is set, else the library's own.
vt_status decode_on_workspace(const Call& c) {
  if (c.num_seqs == 0) return VT_OK;
  vt_status st = validate(c);
  if (st != VT_OK) return st;
  Plan p;
  Scratch w;
  int source = 0;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    st = make_plan(c, &p);
    if (st != VT_OK) return st;
    DeviceState& ds = device_state(p.dev);
    if (ds.user.base) {
      st = fit_user_scratch(ds.user, p.need, c.stream);
      w = ds.user;
      source = 1;
    } else {
      st = ensure_library_scratch(ds.lib, p.need, c.stream);
      w = ds.lib;
    }
    if (st != VT_OK) return st;
  }
  const size_t used = kStatusBytes + w.counters_cap + p.need.part_bytes;
  return launch(c, p, w.base, w.counters_cap, used, source);
}

}  // namespace

extern "C" {

vt_status vt_paged_attn_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                               int num_q_heads, int num_kv_heads, int head_dim, int block_size, float scale,
                               int window, vt_stream_t stream, int max_blocks_per_seq, int num_blocks,
                               vt_dtype dtype) {
  return decode_on_workspace(make_call(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                       num_q_heads, num_kv_heads, head_dim, block_size, scale, window, stream,
                                       max_blocks_per_seq, num_blocks, dtype));
}

vt_status vt_paged_attn_decode_multi(void* out, const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                     int q_len, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                     float scale, int window, vt_stream_t stream, int max_blocks_per_seq,
                                     int num_blocks, vt_dtype dtype) {
  Call c = make_call(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, block_size, scale, window, stream, max_blocks_per_seq, num_blocks, dtype);
  if (dtype == VT_E4M3) return VT_ERR_INVALID_ARG;
  c.q_len = q_len;
  return decode_on_workspace(c);
}

vt_status vt_paged_attn_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                                   const float* k_scale, const float* v_scale, const int32_t* block_tables,
                                   const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                                   int head_dim, int block_size, float scale, int window, vt_stream_t stream,
                                   int max_blocks_per_seq, int num_blocks) {
  Call c = make_call(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, block_size, scale, window, stream, max_blocks_per_seq, num_blocks, VT_E4M3);
  if (!k_scale || !v_scale) return VT_ERR_INVALID_ARG;
  c.k_scale = k_scale;
  c.v_scale = v_scale;
  return decode_on_workspace(c);
}

vt_status vt_paged_attn_decode_multi_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                                         const float* k_scale, const float* v_scale, const int32_t* block_tables,
                                         const int32_t* context_lens, int num_seqs, int q_len, int num_q_heads,
                                         int num_kv_heads, int head_dim, int block_size, float scale, int window,
                                         vt_stream_t stream, int max_blocks_per_seq, int num_blocks) {
  Call c = make_call(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads, num_kv_heads,
                     head_dim, block_size, scale, window, stream, max_blocks_per_seq, num_blocks, VT_E4M3);
  if (!k_scale || !v_scale) return VT_ERR_INVALID_ARG;
  c.k_scale = k_scale;
  c.v_scale = v_scale;
  c.q_len = q_len;
  return decode_on_workspace(c);
}

vt_status vt_paged_attn_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                       float scale, int window, vt_stream_t stream, int max_blocks_per_seq,
                                       int num_blocks, vt_dtype dtype) {
  const Call c = make_call(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                           num_kv_heads, head_dim, block_size, scale, window, stream, max_blocks_per_seq,
                           num_blocks, dtype);
  if (num_seqs == 0) return VT_OK;
  vt_status st = validate(c);
  if (st != VT_OK) return st;
  Plan p;
  char* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    st = make_plan(c, &p);
    if (st != VT_OK) return st;
    const size_t total = ws_total(p.need);
    if (total > kNoAllocScratchBytes) {
      g_last_cuda_error = "vt_paged_attn_decode_noalloc: this call needs " + std::to_string(total) +
                          " bytes of scratch; the static buffer holds " + std::to_string(kNoAllocScratchBytes);
      return VT_ERR_SCRATCH_LIMIT;
    }
    st = noalloc_scratch(device_state(p.dev), &base);
    if (st != VT_OK) return st;
  }
  // The array keeps the previous call's contents (partials of any earlier
  // call may sit where this call's counters go): the status words and the
  // arrival counters must start at zero.
  const size_t counters_region = align_up(p.need.counters_bytes, 256);
  cudaError_t e = cudaMemsetAsync(base, 0, kStatusBytes + counters_region, c.stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  return launch(c, p, base, counters_region, ws_total(p.need), 2);
}

vt_status vt_paged_attn_device_status(vt_stream_t stream_handle, unsigned* status) {
  if (!status) return VT_ERR_INVALID_ARG;
  *status = 0;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  std::lock_guard<std::mutex> lock(g_mutex);
  unsigned all = 0;
  for (const auto& area : status_areas(device_state(dev))) {
    unsigned word = 0;
    e = cudaMemcpy(&word, area.first, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy");
    if (word == 0) continue;
    all |= word;
    // A kernel gave up: clear its status words and every arrival counter it
    // may have left behind.
    e = cudaMemset(area.first, 0, area.second);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
  }
  *status = all;
  return all ? VT_ERR_DEVICE_TIMEOUT : VT_OK;
}

vt_status vt_paged_attn_device_status_detail(vt_stream_t stream_handle, unsigned* words, int n_words) {
  if (!words || n_words < 0 || n_words > 8) return VT_ERR_INVALID_ARG;
  for (int k = 0; k < n_words; ++k) words[k] = 0;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if (n_words == 0) return VT_OK;
  std::lock_guard<std::mutex> lock(g_mutex);
  // the first area whose status word is set (else all zeros)
  for (const auto& area : status_areas(device_state(dev))) {
    unsigned buf[8] = {0};
    e = cudaMemcpy(buf, area.first, sizeof(unsigned) * n_words, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy");
    if (buf[0] == 0) continue;
    for (int k = 0; k < n_words; ++k) words[k] = buf[k];
    break;
  }
  return VT_OK;
}

void vt_paged_attn_release(void) {
  std::lock_guard<std::mutex> lock(g_mutex);
  int cur = 0;
  cudaGetDevice(&cur);
  for (size_t d = 0; d < g_devices.size(); ++d) {
    DeviceState& ds = g_devices[d];
    if (ds.lib.base) {
      cudaSetDevice(static_cast<int>(d));
      cudaFree(ds.lib.base);
      ds.lib = Scratch{};
    }
  }
  cudaSetDevice(cur);
}

}  // extern "C"
