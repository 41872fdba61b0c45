// Paged decode attention kernel for sm_103a (GB300).
//
// One persistent kernel per call does the whole step:
//   S1  request lookup   each CTA reads context_lens on the device, forms the
//                        flattened work space of (sequence, kv head, page)
//                        tiles and takes an even, contiguous slice of it
//                        (stream-K style), so long and short sequences are
//                        balanced without any host-side knowledge of lengths;
//   S2  page gather      a producer warp streams each K and V page tile
//                        (32 tokens x head_dim, NHD, row stride Hkv*head_dim)
//                        with one 3-D TMA copy each into a ring of
//                        shared-memory stages guarded by mbarriers;
//   S3  QK^T (GQA)       consumer warps hold the g query rows that share the
//                        kv head in registers, so every K/V byte is read from
//                        HBM once per kv head;
//   S4  mask             tail slots past the context and tokens before the
//                        window are excluded; pages wholly outside the window
//                        are never loaded;
//   S5  online softmax   per query row, base-2 exponentials on pre-scaled
//                        scores, warp-shuffle reductions;
//   S6  PV               fp32 accumulation of p * v;
//   S7  split partials   a (sequence, kv head) whose tiles span several CTAs
//                        leaves one normalised partial (o, m, l) per CTA;
//   S8  LSE combine      the last CTA to finish such an item merges the
//                        partials (found through an arrival counter);
//   S9  finalize         out = acc / l, rounded once to the storage type.
//
// Operation defined by: issue "ROCm gfx1200: PagedAttnOnline is 8.1x slower
// per call than vLLM's paged-attention kernel", section "Where to look"
// (online softmax, NHD KV read through strides, device-side request lookup);
// PR "perf(cuda): head_dim-128 arm for the warp-split-KV decode kernel",
// commit message (32-token pages, head_dim 128/256, GQA-fused query heads,
// a sliding-window instantiation).
//
// Every wait on an mbarrier is bounded in wall time; on expiry the CTA sets a
// status bit in global memory, stops, lets its own copies in flight land
// (again with a bound) and exits.  No wait, trap or assert can hang the GPU.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace vt {

constexpr int kPageTokens = 32;  // tokens per KV page (block_size)
constexpr int kLaneElems = 8;    // head_dim elements each lane owns per row
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per wait
constexpr unsigned long long kDrainLimitNs = 200000000ull;  // 0.2 s per drained copy

// Stage flags written by the producer.
enum : int { kFirst = 1, kLast = 2, kSplit = 4, kBadPage = 8 };

// Status bits (global status word).
enum : unsigned { kStatusFull = 1u, kStatusEmpty = 2u, kStatusSync = 4u, kStatusDrain = 8u, kStatusWalk = 16u };

struct DecodeArgs {
  void* out;
  const void* q;
  const int* block_tables;
  const int* context_lens;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int group;        // num_q_heads / num_kv_heads
  int subgroups;    // ceil(group / group tile)
  int max_blocks;   // block-table row stride
  int num_blocks;   // pool size in pages
  int window;       // <= 0: none
  float scale_log2; // scale * log2(e)
  int min_units;    // lower bound on tiles per CTA
  int* counters;    // [num_seqs * num_kv_heads * subgroups] arrival counters, zero between calls
  float* part_ml;   // [2 * grid][G][2]  (m, l) of each partial, log2 domain
  float* part_o;    // [2 * grid][G][D]  normalised partial rows
  unsigned* status; // status word
};

struct StageHeader {
  int b;        // sequence
  int vh;       // virtual kv head = h * subgroups + sub
  int lo, hi;   // valid token slots [lo, hi) of this page
  int flags;
  int gq;       // live query rows of this virtual head (<= G)
  int nsplit;   // CTAs sharing this (sequence, virtual head)
  int slot;     // this CTA's partial slot for it
  long long item_u;  // first tile index of the (sequence, virtual head)
};

template <int D, typename T, int G, int NCW, int NSTAGE>
struct Smem {
  static constexpr int GS = D / kLaneElems;       // lanes per row group
  static constexpr int NG = NCW * 32 / GS;        // row groups per CTA
  static constexpr int TPG = kPageTokens / NG;    // tokens per group per page
  alignas(128) T k[NSTAGE][kPageTokens * D];
  alignas(128) T v[NSTAGE][kPageTokens * D];
  alignas(128) T q[NSTAGE][G * D];
  alignas(16) float red_acc[G][D];
  alignas(16) float pbuf[2][NG][G][TPG];
  float abuf[2][NG][G];
  float red_m[2][NG][G];  // double-buffered by segment parity
  float red_l[2][NG][G];
  StageHeader hdr[NSTAGE];
  alignas(8) unsigned long long full[NSTAGE];
  unsigned long long empty[NSTAGE];
  unsigned long long csync;
  long long scan[16];
  long long total_units, u0, u1, cum_start;
  int c_eff, b_start, flag_last;
  volatile int abort_flag;
};

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// 3-D tiled TMA load: box (D, 1, 32) at element coordinates (x, y, z).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// Plain bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Bounded wait on an mbarrier phase.  Returns false (and raises the CTA's
// abort flag plus a global status bit) once the wall-time limit is exceeded,
// or at once if the CTA has already aborted.
__device__ __forceinline__ bool wait_phase(unsigned long long* bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned* status, unsigned code,
                                           unsigned long long limit = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (*abort_flag) return false;
#pragma unroll 1
    for (int k = 0; k < 32; ++k)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit) {
      *abort_flag = 1;
      atomicOr(status, code);
      // first give-up in the grid: record where (status[1..4])
      if (atomicCAS(status + 1, 0u, 1u + blockIdx.x) == 0u) {
        status[2] = code | (threadIdx.x << 8);
        status[3] = static_cast<unsigned>(smem_addr(bar));
        status[4] = parity;
      }
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// Element access.  Lane c of a row group owns 8 elements of every row:
//   bf16: [8c, 8c+8)                  -> one 16-byte shared load
//   fp32: [4c, 4c+4) and [D/2+4c, +4) -> two 16-byte shared loads, each
//         contiguous across the group's lanes (no bank conflicts)
// ---------------------------------------------------------------------------
template <typename T, int D>
struct LaneMap;

template <int D>
struct LaneMap<__nv_bfloat16, D> {
  __device__ __forceinline__ static int col(int c, int e) { return c * 8 + e; }
  __device__ __forceinline__ static void load(const __nv_bfloat16* row, int c, float (&x)[8]) {
    const uint4 raw = *reinterpret_cast<const uint4*>(row + c * 8);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __uint_as_float(w[k] << 16);
      x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static void store(__nv_bfloat16* row, int d0, const float (&x)[8]) {
    // d0 is the first of 8 contiguous columns
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __nv_bfloat162 p = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
      w[k] = *reinterpret_cast<const uint32_t*>(&p);
    }
    *reinterpret_cast<uint4*>(row + d0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <int D>
struct LaneMap<float, D> {
  __device__ __forceinline__ static int col(int c, int e) { return (e < 4) ? c * 4 + e : D / 2 + c * 4 + (e - 4); }
  __device__ __forceinline__ static void load(const float* row, int c, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(row + c * 4);
    const float4 b = *reinterpret_cast<const float4*>(row + D / 2 + c * 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
  __device__ __forceinline__ static void store(float* row, int d0, const float (&x)[8]) {
    *reinterpret_cast<float4*>(row + d0) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(row + d0 + 4) = make_float4(x[4], x[5], x[6], x[7]);
  }
};

// Reduce-scatter of G per-lane partial sums across the GS lanes of a row
// group: afterwards lane c holds the full sum for query c / (GS / G).
template <int G, int GS>
__device__ __forceinline__ float group_reduce_scatter(float (&v)[G], int c) {
#pragma unroll
  for (int n = G, o = GS / 2; n > 1; n >>= 1, o >>= 1) {
    const bool upper = (c & o) != 0;
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
      const float send = upper ? v[k] : v[k + n / 2];
      const float keep = upper ? v[k + n / 2] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = GS / (2 * G); o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}

// ---------------------------------------------------------------------------
// Work partition (identical arithmetic in every CTA).
// ---------------------------------------------------------------------------
struct Partition {
  long long U;  // total tiles
  int C;        // CTAs sharing them
  __device__ __forceinline__ long long start(int c) const { return (static_cast<long long>(c) * U) / C; }
  // CTA whose slice holds tile x (0 <= x < U)
  __device__ __forceinline__ int owner(long long x) const {
    return static_cast<int>(((x + 1) * static_cast<long long>(C) - 1) / U);
  }
  // partial slot that CTA c uses for the item starting at tile item_u
  __device__ __forceinline__ int slot(int c, long long item_u) const { return 2 * c + (start(c) < item_u ? 1 : 0); }
};

struct SeqSpan {
  int p_lo;   // first page touched
  int np;     // pages touched (0: nothing to do)
  int t0;     // first token attended
  int L;      // context length
  bool bad;   // context length invalid
};

__device__ __forceinline__ SeqSpan seq_span(int L, int window, int max_blocks) {
  SeqSpan s;
  s.L = L;
  s.bad = (L < 0) || (static_cast<long long>(L) > static_cast<long long>(max_blocks) * kPageTokens);
  if (s.bad || L == 0) {
    s.p_lo = 0; s.np = 0; s.t0 = 0;
    return s;
  }
  s.t0 = (window > 0 && L > window) ? L - window : 0;
  s.p_lo = s.t0 / kPageTokens;
  s.np = (L + kPageTokens - 1) / kPageTokens - s.p_lo;
  return s;
}

template <int NT>
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long* scratch, long long& total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = (lane < NW) ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NW) scratch[lane] = w;
  }
  __syncthreads();
  const long long prefix = (warp > 0) ? scratch[warp - 1] : 0;
  total = scratch[NW - 1];
  __syncthreads();
  return prefix + x - v;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int D, typename T, int G, int NCW, int NSTAGE, int MINB>
__global__ void __launch_bounds__((NCW + 1) * 32, MINB)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                        const DecodeArgs a) {
  using S = Smem<D, T, G, NCW, NSTAGE>;
  using Map = LaneMap<T, D>;
  constexpr int NT = (NCW + 1) * 32;
  constexpr int NC = NCW * 32;  // consumer threads
  constexpr int GS = S::GS, NG = S::NG, TPG = S::TPG;
  constexpr uint32_t kTileBytes = kPageTokens * D * sizeof(T);
  static_assert(GS <= 32 && (32 % GS) == 0, "row group must tile a warp");
  static_assert(NG * TPG == kPageTokens, "groups must tile the page");
  static_assert(G <= GS && (GS % G) == 0, "group tile must divide the row group");

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // TMA destinations want 128-byte (here 1024-byte) aligned shared addresses;
  // the launch reserves 1 KB of slack for this round-up.
  const uint32_t raw_addr = smem_addr(smem_raw);
  S& s = *reinterpret_cast<S*>(smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nvh = a.num_kv_heads * a.subgroups;

  if (tid == 0) {
    for (int st = 0; st < NSTAGE; ++st) {
      mbar_init(&s.full[st], 1);
      mbar_init(&s.empty[st], NCW);
    }
    mbar_init(&s.csync, NC);
    s.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int e = tid; e < G * D; e += NT) (&s.red_acc[0][0])[e] = 0.f;

  // ---- S1: request lookup and balanced partition ---------------------------
  long long U = 0;
  for (int base = 0; base < a.num_seqs; base += NT) {
    const int b = base + tid;
    long long units = 0;
    if (b < a.num_seqs) {
      const SeqSpan sp = seq_span(__ldg(a.context_lens + b), a.window, a.max_blocks);
      units = static_cast<long long>(sp.np) * nvh;
      if (sp.np == 0 && (b % gridDim.x) == blockIdx.x) {
        // empty context -> zero rows; invalid context -> NaN rows
        const float fill = sp.bad ? __int_as_float(0x7fc00000) : 0.f;
        float vals[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) vals[e] = fill;
        T* row0 = static_cast<T*>(a.out) + static_cast<size_t>(b) * a.num_q_heads * D;
        for (int e = 0; e < a.num_q_heads * D; e += 8) Map::store(row0, e, vals);
      }
    }
    long long tot;
    block_exclusive_scan<NT>(units, s.scan, tot);
    U += tot;
  }
  if (U == 0) return;
  const long long cap = (U + a.min_units - 1) / a.min_units;
  const int C = static_cast<int>(cap < gridDim.x ? cap : gridDim.x);
  if (static_cast<int>(blockIdx.x) >= C) return;
  const Partition part{U, C};
  const long long u0 = part.start(blockIdx.x), u1 = part.start(blockIdx.x + 1);

  if (tid == 0) { s.b_start = -1; }
  {
    long long carry = 0;
    for (int base = 0; base < a.num_seqs; base += NT) {
      const int b = base + tid;
      long long units = 0;
      if (b < a.num_seqs) units = static_cast<long long>(seq_span(__ldg(a.context_lens + b), a.window, a.max_blocks).np) * nvh;
      long long tot;
      const long long excl = carry + block_exclusive_scan<NT>(units, s.scan, tot);
      if (units > 0 && excl <= u0 && u0 < excl + units) {
        s.b_start = b;
        s.cum_start = excl;
      }
      carry += tot;
      if (carry > u0) break;  // uniform: carry is the same in every thread
    }
  }
  __syncthreads();

  if (warp == NCW) {
    // =================== producer warp: TMA page gather (S2) ==================
    if (lane == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    int stage = 0;
    uint32_t phase = 0;
    long long issued = 0;
    long long u = u0, cum = s.cum_start;
    int b = s.b_start;
    // window of 32 context lengths cached across the warp
    int win_base = -(1 << 30), win_len = 0;  // nothing cached yet
    auto length_of = [&](int bb) -> int {
      if (bb < win_base || bb >= win_base + 32) {
        win_base = bb;
        const int idx = bb + lane;
        win_len = (idx < a.num_seqs) ? __ldg(a.context_lens + idx) : 0;
      }
      return __shfl_sync(0xffffffffu, win_len, bb - win_base);
    };
    bool ok = true;
    while (ok && u < u1) {
      const SeqSpan sp = seq_span(length_of(b), a.window, a.max_blocks);
      const long long ub = static_cast<long long>(sp.np) * nvh;
      long long off = u - cum;
      const long long off_end = (u1 - cum < ub) ? (u1 - cum) : ub;
      while (ok && off < off_end) {
        const int vh = static_cast<int>(off / sp.np);
        const int pa = static_cast<int>(off - static_cast<long long>(vh) * sp.np);
        const long long seg_end = off_end - static_cast<long long>(vh) * sp.np;
        const int pb = static_cast<int>(seg_end < sp.np ? seg_end : sp.np);
        const long long item_u = cum + static_cast<long long>(vh) * sp.np;
        const int nsplit = part.owner(item_u + sp.np - 1) - part.owner(item_u) + 1;
        const int h = vh / a.subgroups, sub = vh - h * a.subgroups;
        const int q_row0 = h * a.group + sub * G;
        const int gq = min(G, a.group - sub * G);
        const int* bt_row = a.block_tables + static_cast<size_t>(b) * a.max_blocks + sp.p_lo;
        for (int p0 = pa; ok && p0 < pb; p0 += 32) {
          const int my_p = p0 + lane;
          const int my_id = (my_p < pb) ? __ldg(bt_row + my_p) : 0;
          const int n = min(32, pb - p0);
          for (int jj = 0; jj < n; ++jj) {
            const int pid = __shfl_sync(0xffffffffu, my_id, jj);
            const int p = p0 + jj;
            ok = wait_phase(&s.empty[stage], phase ^ 1u, &s.abort_flag, a.status, kStatusEmpty);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (lane == 0) {
              const bool bad = pid < 0 || pid >= a.num_blocks;
              const int first_tok = (sp.p_lo + p) * kPageTokens;
              StageHeader& hd = s.hdr[stage];
              hd.b = b;
              hd.vh = vh;
              hd.lo = max(sp.t0 - first_tok, 0);
              hd.hi = min(sp.L - first_tok, kPageTokens);
              hd.flags = (p == pa ? kFirst : 0) | (p == pb - 1 ? kLast : 0) | (nsplit > 1 ? kSplit : 0) |
                         (bad ? kBadPage : 0);
              hd.gq = gq;
              hd.nsplit = nsplit;
              hd.slot = part.slot(blockIdx.x, item_u);
              hd.item_u = item_u;
              uint32_t bytes = bad ? 0u : 2u * kTileBytes;
              if (p == pa) bytes += static_cast<uint32_t>(gq) * D * sizeof(T);
              mbar_arrive_expect_tx(&s.full[stage], bytes);
              if (!bad) {
                tma_load_3d(s.k[stage], &tmap_k, 0, h, pid * kPageTokens, &s.full[stage]);
                tma_load_3d(s.v[stage], &tmap_v, 0, h, pid * kPageTokens, &s.full[stage]);
              }
              if (p == pa) {
                const T* qsrc = static_cast<const T*>(a.q) +
                                (static_cast<size_t>(b) * a.num_q_heads + q_row0) * D;
                bulk_load(s.q[stage], qsrc, static_cast<uint32_t>(gq) * D * sizeof(T), &s.full[stage]);
              }
            }
            __syncwarp();
            ++issued;
            if (++stage == NSTAGE) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        off = static_cast<long long>(vh) * sp.np + pb;
      }
      u = cum + off_end;
      cum += ub;
      // next sequence with work
      do {
        ++b;
      } while (ok && u < u1 && b < a.num_seqs && seq_span(length_of(b), a.window, a.max_blocks).np == 0);
      if (b >= a.num_seqs) break;
    }
    // Self-check: the walk must have produced exactly this CTA's tiles.
    if (ok && issued != u1 - u0 && lane == 0) {
      atomicOr(a.status, kStatusWalk);
      s.abort_flag = 1;
    }
    // Let every copy this warp issued land before the CTA can exit.
    if (lane == 0) {
      const long long n_drain = issued < NSTAGE ? issued : NSTAGE;
      for (long long k = 1; k <= n_drain; ++k) {
        const long long idx = issued - k;  // stage index of the k-th most recent copy
        const int st = static_cast<int>(idx % NSTAGE);
        const uint32_t ph = static_cast<uint32_t>((idx / NSTAGE) & 1);
        volatile int never = 0;
        if (!wait_phase(&s.full[st], ph, &never, a.status, kStatusDrain, kDrainLimitNs)) break;
      }
    }
    return;
  }

  // ===================== consumer warps (S3 - S9) =============================
  const int ct = tid;                 // 0 .. NC-1
  const int j = ct / GS;              // row group
  const int c = ct % GS;              // lane within row group
  constexpr int kSpread = GS / G;     // lanes holding the same query after the reduce
  const int iq = c / kSpread;         // query row this lane's scores belong to
  const bool owner = (c % kSpread) == 0;
  const float kNegInf = -__int_as_float(0x7f800000);

  float qf[G][8];
  float acc[G][8];
  float m_run = kNegInf, l_run = 0.f;
  bool poison = false;
  int stage = 0;
  uint32_t phase = 0, sync_phase = 0;
  int par = 0, seg_par = 0;

  auto cons_sync = [&]() -> bool {
    mbar_arrive(&s.csync);
    const bool r = wait_phase(&s.csync, sync_phase, &s.abort_flag, a.status, kStatusSync);
    sync_phase ^= 1u;
    return r;
  };

  const long long n_tiles = u1 - u0;
  for (long long it = 0; it < n_tiles; ++it) {
    bool ok = wait_phase(&s.full[stage], phase, &s.abort_flag, a.status, kStatusFull);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    const StageHeader hd = s.hdr[stage];

    if (hd.flags & kFirst) {
      const T* qs = s.q[stage];
#pragma unroll
      for (int i = 0; i < G; ++i) {
        float x[8];
        if (i < hd.gq) {
          Map::load(qs + i * D, c, x);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          qf[i][e] = x[e] * a.scale_log2;
          acc[i][e] = 0.f;
        }
      }
      m_run = kNegInf;
      l_run = 0.f;
      poison = false;
    }

    if (hd.flags & kBadPage) {
      poison = true;
    } else {
      const T* ks = s.k[stage];
      const T* vs = s.v[stage];
      // S3 + S4: scores of this group's tokens, for the lane's query row
      float sc[TPG];
#pragma unroll
      for (int tt = 0; tt < TPG; ++tt) {
        const int t = j + NG * tt;
        float kx[8];
        Map::load(ks + t * D, c, kx);
        float part_s[G];
#pragma unroll
        for (int i = 0; i < G; ++i) {
          float sum = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) sum = fmaf(qf[i][e], kx[e], sum);
          part_s[i] = sum;
        }
        const float r = group_reduce_scatter<G, GS>(part_s, c);
        sc[tt] = (t >= hd.lo && t < hd.hi) ? r : kNegInf;
      }
      // S5: online softmax update for query iq (base 2, scores pre-scaled)
      float mloc = sc[0];
#pragma unroll
      for (int tt = 1; tt < TPG; ++tt) mloc = fmaxf(mloc, sc[tt]);
      const float m_new = fmaxf(m_run, mloc);
      const float m_use = (m_new == kNegInf) ? 0.f : m_new;
      const float alpha = exp2f(m_run - m_use);
      float p[TPG];
      float psum = 0.f;
#pragma unroll
      for (int tt = 0; tt < TPG; ++tt) {
        p[tt] = exp2f(sc[tt] - m_use);
        psum += p[tt];
      }
      l_run = l_run * alpha + psum;
      m_run = m_new;
      if (owner) {
#pragma unroll
        for (int tt = 0; tt < TPG; ++tt) s.pbuf[par][j][iq][tt] = p[tt];
        s.abuf[par][j][iq] = alpha;
      }
      __syncwarp();
      // rescale the accumulators if any row's maximum moved
      const bool moved = __any_sync(0xffffffffu, alpha != 1.f);
      if (moved) {
#pragma unroll
        for (int i = 0; i < G; ++i) {
          const float ai = s.abuf[par][j][i];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[i][e] *= ai;
        }
      }
      // S6: acc += p * v over this group's valid tokens
#pragma unroll
      for (int tt = 0; tt < TPG; ++tt) {
        const int t = j + NG * tt;
        if (t >= hd.lo && t < hd.hi) {
          float vx[8];
          Map::load(vs + t * D, c, vx);
#pragma unroll
          for (int i = 0; i < G; ++i) {
            const float pi = s.pbuf[par][j][i][tt];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(pi, vx[e], acc[i][e]);
          }
        }
      }
      par ^= 1;
    }
    // release the stage to the producer
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[stage]);
    if (++stage == NSTAGE) {
      stage = 0;
      phase ^= 1u;
    }

    if (!(hd.flags & kLast)) continue;

    // ---- end of a (sequence, virtual head) segment: merge the row groups ----
    // red_m/red_l are double-buffered: a thread can only reach the next
    // segment's first rendezvous after every thread finished reading these.
    float (*rm)[G] = s.red_m[seg_par];
    float (*rl)[G] = s.red_l[seg_par];
    seg_par ^= 1;
    if (owner) {
      rm[j][iq] = m_run;
      rl[j][iq] = poison ? __int_as_float(0x7fc00000) : l_run;
    }
    if (!cons_sync()) break;
#pragma unroll
    for (int i = 0; i < G; ++i) {
      float M = kNegInf;
#pragma unroll
      for (int g2 = 0; g2 < NG; ++g2) M = fmaxf(M, rm[g2][i]);
      const float f = exp2f(rm[j][i] - ((M == kNegInf) ? 0.f : M));
#pragma unroll
      for (int e = 0; e < 8; ++e) atomicAdd(&s.red_acc[i][Map::col(c, e)], acc[i][e] * f);
    }
    if (!cons_sync()) break;

    const int h = hd.vh / a.subgroups, sub = hd.vh - h * a.subgroups;
    const int q_row0 = h * a.group + sub * G;
    const bool split = (hd.flags & kSplit) != 0;
    for (int e0 = ct * 8; e0 < G * D; e0 += NC * 8) {
      const int i = e0 / D, d0 = e0 - i * D;
      float M = kNegInf;
#pragma unroll
      for (int g2 = 0; g2 < NG; ++g2) M = fmaxf(M, rm[g2][i]);
      M = (M == kNegInf) ? 0.f : M;
      float L = 0.f;
#pragma unroll
      for (int g2 = 0; g2 < NG; ++g2) L += rl[g2][i] * exp2f(rm[g2][i] - M);
      float val[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        val[e] = s.red_acc[i][d0 + e] / L;
        s.red_acc[i][d0 + e] = 0.f;
      }
      if (i >= hd.gq) continue;
      if (!split) {
        // S9: final row, one rounding to the storage type
        T* row = static_cast<T*>(a.out) + (static_cast<size_t>(hd.b) * a.num_q_heads + q_row0 + i) * D;
        // columns d0..d0+7 are contiguous here (not the lane map)
        if constexpr (sizeof(T) == 2) {
          LaneMap<__nv_bfloat16, D>::store(reinterpret_cast<__nv_bfloat16*>(row), d0, val);
        } else {
          LaneMap<float, D>::store(reinterpret_cast<float*>(row), d0, val);
        }
      } else {
        // S7: normalised partial row plus its (m, l)
        float* po = a.part_o + (static_cast<size_t>(hd.slot) * G + i) * D + d0;
        *reinterpret_cast<float4*>(po) = make_float4(val[0], val[1], val[2], val[3]);
        *reinterpret_cast<float4*>(po + 4) = make_float4(val[4], val[5], val[6], val[7]);
        if (d0 == 0) {
          float* pm = a.part_ml + (static_cast<size_t>(hd.slot) * G + i) * 2;
          pm[0] = M;
          pm[1] = L;
        }
      }
    }
    if (!split) continue;

    // ---- S8: the last CTA to finish this item merges all partials ----------
    __threadfence();
    if (!cons_sync()) break;
    const int item = hd.b * nvh + hd.vh;
    if (ct == 0) {
      const int prev = atomicAdd(a.counters + item, 1);
      const int last = (prev == hd.nsplit - 1) ? 1 : 0;
      if (last) atomicExch(a.counters + item, 0);
      s.flag_last = last;
    }
    if (!cons_sync()) break;
    if (!s.flag_last) continue;
    __threadfence();
    const int c_first = part.owner(hd.item_u);
    for (int e0 = ct * 8; e0 < G * D; e0 += NC * 8) {
      const int i = e0 / D, d0 = e0 - i * D;
      if (i >= hd.gq) continue;
      float M = kNegInf;
      for (int k = 0; k < hd.nsplit; ++k) {
        const int sl = part.slot(c_first + k, hd.item_u);
        M = fmaxf(M, __ldcg(a.part_ml + (static_cast<size_t>(sl) * G + i) * 2));
      }
      float L = 0.f, o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = 0.f;
      for (int k = 0; k < hd.nsplit; ++k) {
        const int sl = part.slot(c_first + k, hd.item_u);
        const float* pm = a.part_ml + (static_cast<size_t>(sl) * G + i) * 2;
        const float w = __ldcg(pm + 1) * exp2f(__ldcg(pm) - M);
        L += w;
        const float* po = a.part_o + (static_cast<size_t>(sl) * G + i) * D + d0;
        const float4 x0 = __ldcg(reinterpret_cast<const float4*>(po));
        const float4 x1 = __ldcg(reinterpret_cast<const float4*>(po + 4));
        o[0] = fmaf(w, x0.x, o[0]); o[1] = fmaf(w, x0.y, o[1]);
        o[2] = fmaf(w, x0.z, o[2]); o[3] = fmaf(w, x0.w, o[3]);
        o[4] = fmaf(w, x1.x, o[4]); o[5] = fmaf(w, x1.y, o[5]);
        o[6] = fmaf(w, x1.z, o[6]); o[7] = fmaf(w, x1.w, o[7]);
      }
      float val[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) val[e] = o[e] / L;
      T* row = static_cast<T*>(a.out) + (static_cast<size_t>(hd.b) * a.num_q_heads + q_row0 + i) * D;
      if constexpr (sizeof(T) == 2) {
        LaneMap<__nv_bfloat16, D>::store(reinterpret_cast<__nv_bfloat16*>(row), d0, val);
      } else {
        LaneMap<float, D>::store(reinterpret_cast<float*>(row), d0, val);
      }
    }
  }
}

}  // namespace vt
