// C-ABI front end of the paged decode library: argument validation, launch
// plan, per-device split workspace, TMA descriptors, launch.
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

constexpr int kVersion = 10000;  // 1.0.0
constexpr int kMaxGroupTile = 8;
constexpr int kDefaultMinUnits = 2;
constexpr int kDefaultSegCost = 2;  // a segment boundary weighs about two tiles of streaming

thread_local int g_override_grid = 0;
thread_local bool g_overlap = false;
thread_local int g_override_min_units = 0;
thread_local int g_seg_cost = -1;  // < 0: default
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
  if (head_dim == 128 && dtype == VT_F32) table = vt::variants_d128_f32(&n);
  if (head_dim == 256 && dtype == VT_F32) table = vt::variants_d256_f32(&n);
  for (int k = 0; k < n; ++k)
    if (table[k].group_tile == group_tile) return &table[k];
  return nullptr;
}

// Query rows computed per kv head and CTA.  bf16 runs on tensor cores with
// the queries as the M dimension of m16n8k16: one tile of 8 (or 16) rows
// covers any group up to that size.  fp32 runs on CUDA cores, where every
// padded row costs FMAs: the next power of two, at most 8.
int group_tile_for(int group, vt_dtype dtype) {
  if (dtype == VT_BF16) return group <= 8 ? 8 : 16;
  int g = 1;
  while (g < group && g < kMaxGroupTile) g <<= 1;
  return g;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout: [status word (256 B) | counter region | partial (m, l, 0, 0) | partial rows].
// The counter region is reserved at allocation and never holds anything but
// arrival counters, which every kernel leaves at zero; partials start after it.
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

size_t ws_total(const WsNeed& n) { return 256 + align_up(n.counters_bytes, 256) + n.part_bytes; }

// ---------------------------------------------------------------------------
// Per-device state
// ---------------------------------------------------------------------------
struct DeviceState {
  bool init = false;
  int num_sms = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  size_t counters_cap = 0;  // bytes reserved for arrival counters (after the status word)
  size_t partial_cap = 0;   // bytes for partials, starting at 256 + counters_cap
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

// Grows (never shrinks) the device's workspace.  A new buffer is zeroed on
// `stream` before any kernel that uses it, so all counters start at 0.
vt_status ensure_workspace(DeviceState& ds, const WsNeed& n, cudaStream_t stream) {
  if (ds.ws && ds.counters_cap >= n.counters_bytes && ds.partial_cap >= n.part_bytes) return VT_OK;
  size_t counters = ds.counters_cap > n.counters_bytes ? ds.counters_cap : n.counters_bytes;
  counters = align_up(counters + counters / 4 + 1024, 256);
  size_t partial = ds.partial_cap > n.part_bytes ? ds.partial_cap : n.part_bytes;
  partial = align_up(partial + partial / 4, 1 << 16);
  const size_t bytes = 256 + counters + partial;
  if (ds.ws) {
    cudaError_t e = cudaFreeAsync(ds.ws, stream);
    ds.ws = nullptr;
    ds.ws_bytes = ds.counters_cap = ds.partial_cap = 0;
    if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync");
  }
  void* p = nullptr;
  cudaError_t e = cudaMallocAsync(&p, bytes, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    g_last_cuda_error = std::string("cudaMallocAsync: ") + cudaGetErrorString(e);
    return VT_ERR_OOM;
  }
  e = cudaMemsetAsync(p, 0, 256 + counters, stream);
  if (e != cudaSuccess) {
    cudaFreeAsync(p, stream);
    return cuda_fail(e, "cudaMemsetAsync");
  }
  ds.ws = p;
  ds.ws_bytes = bytes;
  ds.counters_cap = counters;
  ds.partial_cap = partial;
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
  const size_t es = k.dtype == VT_BF16 ? 2 : 4;
  const cuuint64_t tokens = static_cast<cuuint64_t>(k.num_blocks) * vt::kPageTokens;
  const cuuint64_t row = static_cast<cuuint64_t>(k.head_dim) * k.num_kv_heads * es;  // bytes per token
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUtensorMap m;
  CUresult r;
  if (k.dtype == VT_BF16) {
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
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    // CUDA-core consumer: a 3-D view (column, kv head, token) and one
    // unswizzled box of head_dim x 32 tokens.
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(k.head_dim), static_cast<cuuint64_t>(k.num_kv_heads), tokens};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(k.head_dim) * es, row};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(k.head_dim), 1u, static_cast<cuuint32_t>(vt::kPageTokens)};
    r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(k.ptr), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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
    case VT_ERR_SCRATCH_LIMIT: return "call needs more scratch than the static buffer holds";
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
  const int gt = group_tile_for(group, dtype);
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

vt_status vt_paged_attn_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                               int num_q_heads, int num_kv_heads, int head_dim, int block_size, float scale,
                               int window, vt_stream_t stream_handle, int max_blocks_per_seq, int num_blocks,
                               vt_dtype dtype) {
  if (num_seqs < 0) return VT_ERR_INVALID_ARG;
  if (num_seqs == 0) return VT_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return VT_ERR_INVALID_ARG;
  if (dtype != VT_BF16 && dtype != VT_F32) return VT_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return VT_ERR_INVALID_ARG;
  if (max_blocks_per_seq <= 0 || num_blocks <= 0 || block_size <= 0 || head_dim <= 0) return VT_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return VT_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return VT_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return VT_ERR_UNSUPPORTED;
  if (block_size != vt::kPageTokens) return VT_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * vt::kPageTokens > 0x7fffffffLL) return VT_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_blocks_per_seq) * vt::kPageTokens > 0x7fffffffLL) return VT_ERR_UNSUPPORTED;

  const int group = num_q_heads / num_kv_heads;
  const int gt = group_tile_for(group, dtype);
  const int subgroups = (group + gt - 1) / gt;
  const long long nvh = static_cast<long long>(num_kv_heads) * subgroups;
  if (nvh * num_seqs > 0x7fffffffLL) return VT_ERR_UNSUPPORTED;
  const VariantInfo* v = find_variant(head_dim, dtype, gt);
  if (!v) return VT_ERR_UNSUPPORTED;

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");

  DecodeArgs args{};
  int grid = 0, per_sm = 0, min_units = 0;
  size_t ws_used = 0;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& ds = device_state(dev);
    vt_status st = prepare_device(dev, ds);
    if (st != VT_OK) return st;
    st = prepare_variant(ds, *v, &per_sm);
    if (st != VT_OK) return st;
    grid = g_override_grid > 0 ? g_override_grid : ds.num_sms * per_sm;
    min_units = g_override_min_units > 0 ? g_override_min_units : kDefaultMinUnits;
    const WsNeed need = ws_need(num_seqs, static_cast<int>(nvh), grid, gt, head_dim);
    st = ensure_workspace(ds, need, stream);
    if (st != VT_OK) return st;
    ws_used = ws_total(need);
    char* base = static_cast<char*>(ds.ws);
    args.status = reinterpret_cast<unsigned*>(base);
    args.counters = reinterpret_cast<int*>(base + 256);
    args.part = reinterpret_cast<float*>(base + 256 + ds.counters_cap);
    g_last_plan.num_sms = ds.num_sms;
  }

  CUtensorMap tk, tv;
  vt_status st = tensor_map(MapKey{k_cache, head_dim, num_kv_heads, num_blocks, dtype, dev}, &tk);
  if (st != VT_OK) return st;
  st = tensor_map(MapKey{v_cache, head_dim, num_kv_heads, num_blocks, dtype, dev}, &tv);
  if (st != VT_OK) return st;

  args.out = out;
  args.q = q;
  args.block_tables = block_tables;
  args.context_lens = context_lens;
  args.num_seqs = num_seqs;
  args.num_q_heads = num_q_heads;
  args.num_kv_heads = num_kv_heads;
  args.group = group;
  args.subgroups = subgroups;
  args.max_blocks = max_blocks_per_seq;
  args.num_blocks = num_blocks;
  args.window = window > 0 ? window : 0;
  args.scale_log2 = scale * 1.4426950408889634f;
  args.min_units = min_units;
  args.seg_cost = g_seg_cost < 0 ? kDefaultSegCost : g_seg_cost;

  e = v->launch(tk, tv, args, grid, stream, g_overlap);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  g_last_plan.launch_overlap = g_overlap ? 1 : 0;
  g_last_plan.segment_cost = args.seg_cost;

  g_last_plan.grid_ctas = grid;
  g_last_plan.ctas_per_sm = per_sm;
  g_last_plan.consumer_warps = v->consumer_warps;
  g_last_plan.tensor_cores = v->tensor_cores;
  g_last_plan.stages = v->stages;
  g_last_plan.group_tile = gt;
  g_last_plan.subgroups = subgroups;
  g_last_plan.min_units_per_cta = min_units;
  g_last_plan.head_dim = head_dim;
  g_last_plan.dtype = dtype;
  g_last_plan.smem_bytes = v->smem_bytes;
  g_last_plan.workspace_bytes = ws_used;
  g_have_plan = true;
  return VT_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant: the split scratch is a fixed, file-scope device
// array instead of the library's lazily allocated per-device workspace.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = VT_NOALLOC_SCRATCH_BYTES;  // held on every device that loads the library
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
std::vector<void*> g_noalloc_ptr;  // device address of the array, per device

// In host code the array's name is only a host-side stand-in: its device
// address must be looked up, once per device, with that device current.
vt_status noalloc_scratch(int dev, void** ptr) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (static_cast<int>(g_noalloc_ptr.size()) <= dev) g_noalloc_ptr.resize(dev + 1, nullptr);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return VT_OK;
}

}  // namespace

extern "C" {

vt_status vt_paged_attn_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                       float scale, int window, vt_stream_t stream_handle, int max_blocks_per_seq,
                                       int num_blocks, vt_dtype dtype) {
  if (num_seqs < 0) return VT_ERR_INVALID_ARG;
  if (num_seqs == 0) return VT_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return VT_ERR_INVALID_ARG;
  if (dtype != VT_BF16 && dtype != VT_F32) return VT_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return VT_ERR_INVALID_ARG;
  if (max_blocks_per_seq <= 0 || num_blocks <= 0 || block_size <= 0 || head_dim <= 0) return VT_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return VT_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return VT_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return VT_ERR_UNSUPPORTED;
  if (block_size != vt::kPageTokens) return VT_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * vt::kPageTokens > 0x7fffffffLL) return VT_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_blocks_per_seq) * vt::kPageTokens > 0x7fffffffLL) return VT_ERR_UNSUPPORTED;

  const int group = num_q_heads / num_kv_heads;
  const int gt = group_tile_for(group, dtype);
  const int subgroups = (group + gt - 1) / gt;
  const long long nvh = static_cast<long long>(num_kv_heads) * subgroups;
  if (nvh * num_seqs > 0x7fffffffLL) return VT_ERR_UNSUPPORTED;
  const VariantInfo* v = find_variant(head_dim, dtype, gt);
  if (!v) return VT_ERR_UNSUPPORTED;

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");

  int grid = 0, per_sm = 0, min_units = 0, num_sms = 0;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& ds = device_state(dev);
    vt_status st = prepare_device(dev, ds);
    if (st != VT_OK) return st;
    st = prepare_variant(ds, *v, &per_sm);
    if (st != VT_OK) return st;
    grid = g_override_grid > 0 ? g_override_grid : ds.num_sms * per_sm;
    min_units = g_override_min_units > 0 ? g_override_min_units : kDefaultMinUnits;
    num_sms = ds.num_sms;
  }
  // Layout inside the fixed array: [status 256 B | counters | partial records].
  const WsNeed need = ws_need(num_seqs, static_cast<int>(nvh), grid, gt, head_dim);
  const size_t counters_region = align_up(need.counters_bytes, 256);
  const size_t total = 256 + counters_region + need.part_bytes;
  if (total > kNoAllocScratchBytes) {
    g_last_cuda_error = "vt_paged_attn_decode_noalloc: this call needs " + std::to_string(total) +
                        " bytes of scratch; the static buffer holds " + std::to_string(kNoAllocScratchBytes);
    return VT_ERR_SCRATCH_LIMIT;
  }
  void* base_ptr = nullptr;
  vt_status st = noalloc_scratch(dev, &base_ptr);
  if (st != VT_OK) return st;
  char* base = static_cast<char*>(base_ptr);
  // The array keeps the previous call's contents: the status word and the
  // arrival counters must start at zero.
  e = cudaMemsetAsync(base, 0, 256 + counters_region, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");

  CUtensorMap tk, tv;
  st = tensor_map(MapKey{k_cache, head_dim, num_kv_heads, num_blocks, dtype, dev}, &tk);
  if (st != VT_OK) return st;
  st = tensor_map(MapKey{v_cache, head_dim, num_kv_heads, num_blocks, dtype, dev}, &tv);
  if (st != VT_OK) return st;

  DecodeArgs args{};
  args.status = reinterpret_cast<unsigned*>(base);
  args.counters = reinterpret_cast<int*>(base + 256);
  args.part = reinterpret_cast<float*>(base + 256 + counters_region);
  args.out = out;
  args.q = q;
  args.block_tables = block_tables;
  args.context_lens = context_lens;
  args.num_seqs = num_seqs;
  args.num_q_heads = num_q_heads;
  args.num_kv_heads = num_kv_heads;
  args.group = group;
  args.subgroups = subgroups;
  args.max_blocks = max_blocks_per_seq;
  args.num_blocks = num_blocks;
  args.window = window > 0 ? window : 0;
  args.scale_log2 = scale * 1.4426950408889634f;
  args.min_units = min_units;
  args.seg_cost = g_seg_cost < 0 ? kDefaultSegCost : g_seg_cost;

  e = v->launch(tk, tv, args, grid, stream, g_overlap);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  g_last_plan.launch_overlap = g_overlap ? 1 : 0;
  g_last_plan.segment_cost = args.seg_cost;

  g_last_plan.num_sms = num_sms;
  g_last_plan.grid_ctas = grid;
  g_last_plan.ctas_per_sm = per_sm;
  g_last_plan.consumer_warps = v->consumer_warps;
  g_last_plan.tensor_cores = v->tensor_cores;
  g_last_plan.stages = v->stages;
  g_last_plan.group_tile = gt;
  g_last_plan.subgroups = subgroups;
  g_last_plan.min_units_per_cta = min_units;
  g_last_plan.head_dim = head_dim;
  g_last_plan.dtype = dtype;
  g_last_plan.smem_bytes = v->smem_bytes;
  g_last_plan.workspace_bytes = total;
  g_have_plan = true;
  return VT_OK;
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
  DeviceState& ds = device_state(dev);
  if (!ds.ws) return VT_OK;
  unsigned word = 0;
  e = cudaMemcpy(&word, ds.ws, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy");
  *status = word;
  if (word == 0) return VT_OK;
  // A kernel gave up: clear the word and every arrival counter it may have left behind.
  e = cudaMemset(ds.ws, 0, 256 + ds.counters_cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
  return VT_ERR_DEVICE_TIMEOUT;
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
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& ds = device_state(dev);
  if (!ds.ws || n_words == 0) return VT_OK;
  e = cudaMemcpy(words, ds.ws, sizeof(unsigned) * n_words, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy");
  return VT_OK;
}

void vt_paged_attn_release(void) {
  std::lock_guard<std::mutex> lock(g_mutex);
  int cur = 0;
  cudaGetDevice(&cur);
  for (size_t d = 0; d < g_devices.size(); ++d) {
    DeviceState& ds = g_devices[d];
    if (ds.ws) {
      cudaSetDevice(static_cast<int>(d));
      cudaFree(ds.ws);
      ds.ws = nullptr;
      ds.ws_bytes = ds.counters_cap = ds.partial_cap = 0;
    }
  }
  cudaSetDevice(cur);
}

}  // extern "C"
