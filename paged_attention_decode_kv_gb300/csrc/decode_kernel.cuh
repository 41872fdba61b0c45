// Paged decode attention kernel for sm_103a (GB300).
//
// One persistent kernel per call does the whole step:
//   S1  request lookup   each CTA reads context_lens on the device, forms the
//                        flattened work space of (sequence, kv head, page)
//                        tiles and takes an even, contiguous slice of it
//                        (stream-K style; each (sequence, kv head) also
//                        weighs a little for its segment overhead), so long
//                        and short sequences are balanced without any
//                        host-side knowledge of lengths;
//   S2  page gather      a producer warp streams each K and V page tile
//                        (32 tokens x head_dim, NHD, row stride Hkv*head_dim)
//                        with one TMA copy each into a ring of shared-memory
//                        stages guarded by mbarriers;
//   S3  QK^T (GQA)       the g query rows that share a kv head are computed
//                        together, so every K/V byte is read from HBM once
//                        per kv head.  bf16 storage: tensor cores
//                        (mma.sync m16n8k16, the page's tokens as M and the
//                        query group as N); FP8 E4M3 codes: the same on f16
//                        after exact widening; fp32 storage: CUDA-core FMAs;
//   S4  mask             tail slots past the context and tokens before the
//                        window are excluded; pages wholly outside the window
//                        are never loaded;
//   S5  online softmax   per query row, base-2 exponentials on pre-scaled
//                        scores, warp-shuffle reductions;
//   S6  PV               fp32 accumulation of p * v (tensor cores for bf16,
//                        with p split into two bf16 terms, hi + lo, so the
//                        weights keep ~16 significant bits; f16 weights for
//                        FP8 codes);
//   S7  split partials   a (sequence, kv head) whose tiles span several CTAs
//                        leaves one normalised partial (o, m, l) per CTA;
//   S8  LSE combine      the last CTA to finish such an item (found through
//                        an arrival counter) stages the partials with bulk
//                        copies and merges them;
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
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace vt {

constexpr int kPageTokens = 32;  // tokens per KV page (block_size)
constexpr int kSwizzleCols = 64; // bf16 columns per 128-byte swizzled sub-tile row
// Wait limits in SM clock cycles (clock64 is a cheap per-SM counter; at the
// GB300's 2.07 GHz maximum, 2^31 cycles is about 1 s and 2^28 about 0.13 s).
constexpr long long kWaitLimitCycles = 1ll << 31;
constexpr long long kDrainLimitCycles = 1ll << 28;

// Page tiles of its slice a CTA prefetches into L2 before its dependency wait.
constexpr int kPrefetchTiles = 8;

// Stage flags written by the producer.
// kEnd: no more tiles; kPad: a stage without tiles that only closes a segment
// for a warp pair (see Smem::NPAR).
enum : int { kFirst = 1, kLast = 2, kSplit = 4, kBadPage = 8, kEnd = 16, kPad = 32 };

// Status bits (global status word).
enum : unsigned {
  kStatusFull = 1u,
  kStatusEmpty = 2u,
  kStatusSync = 4u,
  kStatusDrain = 8u,
  kStatusWalk = 16u,
  kStatusCombine = 32u
};

struct DecodeArgs {
  void* out;
  const void* q;
  const int* block_tables;
  const int* context_lens;
  int num_seqs;
  int num_q_heads;
  int q_len;        // new tokens per sequence (1: single-token decode)
  int rows;         // query rows per kv head: q_len * group
  int num_kv_heads;
  int group;        // num_q_heads / num_kv_heads
  int subgroups;    // ceil(rows / group tile)
  int max_blocks;   // block-table row stride
  int num_blocks;   // pool size in pages
  int window;       // <= 0: none
  float scale_log2; // scale * log2(e)
  int min_units;    // lower bound on tiles per CTA
  int seg_cost;     // tiles' worth of time a segment boundary costs (partition weight)
  int* counters;    // [num_seqs * num_kv_heads * subgroups] arrival counters, zero between calls
  // Split partials: one record per slot, G * 4 + min(G, group) * D floats,
  // holding (m, l, 0, 0) per row in the log2 domain, then the normalised
  // rows.  Slots [0, grid) hold each CTA's first segment (an item that
  // started before its slice), slots [grid, 2 grid) its last (an item that
  // starts inside its slice): the partials of one item then sit in one run
  // of consecutive records, plus at most one record of the second half.
  float* part;
  unsigned* status; // status words
  // Bounded waits give up after wait_limit clock cycles (kWaitLimitCycles
  // unless a test shortens it).  Test hook: CTA withhold_cta stops feeding
  // its consumers before its withhold_tile-th tile (-1: never), so their
  // wait for that tile runs out and reports through the status word.
  long long wait_limit;
  int withhold_cta;
  int withhold_tile;
  // FP8 E4M3 K/V storage only: per-kv-head dequantisation scales [num_kv_heads]
  // (a code of kv head h stands for its E4M3 value times k_scale[h] or v_scale[h]).
  const float* k_scale;
  const float* v_scale;
};

struct StageHeader {
  int b;        // sequence
  int vh;       // virtual kv head = h * subgroups + sub
  int lo, hi;   // token slots [lo, hi) of this page attended by some query row
  int rel_end;  // context length minus the page's first token (may exceed 32)
  int flags;
  int gq;       // live query rows of this virtual head (<= G)
  int nsplit;   // CTAs sharing this (sequence, virtual head)
  int slot;     // this CTA's partial slot for it
  int c_first;  // first CTA sharing it
  long long item_u;  // work unit of the item's first page
};

// Consumer kinds: CUDA cores (fp32 storage); tensor cores on bf16 K/V
// (mma.sync bf16); tensor cores on FP8 E4M3 K/V codes (widened exactly to f16
// in registers for mma.sync f16, with f16 queries and weights; bf16 queries
// and output in memory).  An e4m3 mma.sync is no cheaper here: on this GPU it
// issues two f16 MMAs plus the operand widening for every k32 step.
enum class Math { kSimt, kMma, kMma8 };

// Element type of the K/V page tiles for a consumer kind.
template <typename T, Math M>
using KvElem = std::conditional_t<M == Math::kMma8, uint8_t, T>;

// A combine the CTA owes: it was the last to finish a split item.
struct PendingCombine {
  int b, vh, nsplit, gq, c_first;
  long long item_u;
};

// Shared memory of a CTA.  The stage ring (k, v) sits last, followed by EXT
// spare bytes: once the tiles are done, k, v and ext form one contiguous
// buffer the split-KV combine stages partial records into.
template <int D, typename T, int G, int NCW, int NSTAGE, Math M, int EXT = 0>
struct Smem {
  // CUDA-core layout: lane c of a row group owns 8 elements of every row.
  static constexpr int GS = D / 8;
  static constexpr int NG = (M == Math::kSimt) ? NCW * 32 / GS : 1;
  static constexpr int TPG = kPageTokens / NG;
  // mma layout: warps split the page into (token half tg) x (head_dim part
  // dp).  With NPAR = 2 the warps also form two pairs of alternate pages:
  // pair par takes the ring stages s with s mod 2 = par, so two pages are in
  // flight per CTA and no head_dim part repeats another's QK^T and softmax:
  // for the 8 KB tiles of FP8 K/V at head_dim 128 and 256 and of bf16 at
  // head_dim 64, whose per-tile work, not the bytes, bounds them (bf16 at
  // head_dim 128 and 256 measured no faster).  The producer gives every
  // segment an even number of stages (closing odd ones with a kPad stage),
  // so segments start on even stages.
  static constexpr int NPAR =
      ((M == Math::kMma8 || (M == Math::kMma && D == 64)) && G <= 8 && NCW == 4) ? 2 : 1;
  static constexpr int NDP = (M != Math::kSimt) ? NCW / (2 * NPAR) : 1;
  static constexpr int kRedRows = (M == Math::kSimt) ? NG : 2 * NPAR;
  alignas(128) T q[NSTAGE][G * D];
  // head_dim 512 (bf16 tensor cores): the Q^T fragments of 32 k-steps do not
  // fit in registers, so the segment's query rows are copied into this
  // buffer ([head_dim / 64][G][64 columns], 128-byte swizzle) and read with
  // ldmatrix per k-step pair.
  static constexpr bool QS = (M == Math::kMma) && D >= 512;
  alignas(1024) T qs[QS ? G * D : 8];
  // Tensor-core epilogue: warps of token half 1 hand their O^T accumulator
  // fragments to the warps of token half 0 ([segment parity][dp][slot][m-tile]
  // [lane]); token half 0 then reuses the slice to stage rows for coalesced
  // stores.  With NPAR = 2 the second pair first hands its fragments to the
  // first (slot tg), then token half 1 of the first pair uses slot 1.
  static constexpr int XV = (G > 8) ? 8 : 4;  // accumulator values per lane and m-tile
  static constexpr int XP = (M != Math::kSimt) ? 2 : 1;
  static constexpr int XN = (M != Math::kSimt) ? D / NDP / 16 : 1;
  alignas(16) float xbuf[XP][NDP][NPAR][XN][32][XV];
  // bf16 at head_dim 512: the four head_dim parts split QK^T (SQK) and sum
  // their partial scores through this buffer ([tile parity][tg][dp][lane],
  // a float4 per query n-tile), one mbarrier per (tile parity, tg).  (With
  // the two parts of head_dim 256 the exchange costs more than it saves.)
  static constexpr bool SQK = (M == Math::kMma) && D >= 512 && NDP > 1;
  static constexpr int QXN = (G > 8) ? 2 : 1;
  alignas(16) float4 qx[SQK ? 2 : 1][SQK ? 2 : 1][SQK ? NDP : 1][SQK ? 32 : 1][SQK ? QXN : 1];
  unsigned long long qx_bar[2][2];
  // CUDA-core consumer only: per-group broadcast of p and the rescale factor.
  static constexpr int PG = (M == Math::kSimt) ? G : 1;
  static constexpr int PT = (M == Math::kSimt) ? TPG : 1;
  alignas(16) float pbuf[2][NG][PG][PT];
  float abuf[2][NG][PG];
  float red_m[2][kRedRows][G];  // double-buffered by segment parity
  float red_l[2][kRedRows][G];
  float fin_m[G];
  float fin_l[G];
  StageHeader hdr[NSTAGE];
  alignas(8) unsigned long long full[NSTAGE];
  unsigned long long empty[NSTAGE];
  unsigned long long csync;
  unsigned long long comb;  // partials staged for a combine
  long long scan[16];
  int b_start_s;
  long long cum_start_s;
  PendingCombine pend[2];
  int pend_n;
  volatile int abort_flag;
  alignas(1024) KvElem<T, M> k[NSTAGE][kPageTokens * D];
  alignas(1024) KvElem<T, M> v[NSTAGE][kPageTokens * D];
  alignas(16) unsigned char ext[EXT > 0 ? EXT : 16];
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

// 3-D tiled TMA load at element coordinates (x, y, z).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar))
      : "memory");
}

// L2 prefetch of a tensor box (no shared-memory destination, no barrier).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int x, int y, int z, int w) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w)
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

// Programmatic dependent launch.  launch_dependents lets the next kernel on
// the stream (if it was launched as a programmatic dependent) start its CTAs
// once every CTA of this grid has issued it; wait blocks until the grids this
// one depends on have completed and their memory is visible.  Both are no-ops
// for an ordinary launch.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Orders this thread's generic-proxy accesses to global memory with its
// async-proxy (bulk copy) accesses: partials are written with plain stores
// and read back by bulk copies of another CTA.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// The same for this thread's shared-memory accesses (a stage's tiles that
// consumers wrote before the producer's next copy into them).
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrival counter increment with acquire-release semantics at GPU scope: the
// release orders every store the CTA made before the preceding rendezvous,
// the acquire lets the last arriver see the other CTAs' partials.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void st_relaxed_gpu(int* p, int v) {
  asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D = A * B + D, bf16 inputs, fp32 accumulators, m16n8k16.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A * B + D, f16 inputs, fp32 accumulators, m16n8k16.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four E4M3 codes (byte i: element i) widened exactly to two f16 pairs,
// lo = (e0, e1) and hi = (e2, e3) (every E4M3 value is an f16 normal number
// or zero; the NaN codes give NaN).
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t codes, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(codes));
}

// 2^e as a float, e in [-126, 127].
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// 2^x with the hardware approximation (ex2.approx.ftz: relative error about
// 2^-22; results below 2^-126 flush to 0, 2^-inf = 0): the softmax weights,
// which enter the sums against weights of at least 1.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Transpose of an 8x8 b16 matrix held one 32-bit pair per lane (row lane/4,
// columns 2(lane%4), +1): afterwards each lane holds the same positions of
// the transposed matrix.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

__device__ __forceinline__ float bf16_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Bounded wait on an mbarrier phase.  Returns false (and raises the CTA's
// abort flag plus a global status bit) once the clock-cycle limit is
// exceeded, or at once if the CTA has already aborted.  The limit is checked
// with clock64 every 32 probes: a %globaltimer read costs far more than a
// probe and would sit on the critical path of every wait that does not
// complete at once.
__device__ __forceinline__ bool wait_phase(unsigned long long* bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned* status, unsigned code, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (*abort_flag) return false;
#pragma unroll 1
    for (int k = 0; k < 32; ++k)
      if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit) {
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
// Element access for the CUDA-core consumer.  Lane c of a row group owns 8
// elements of every row:
//   bf16: [8c, 8c+8)                  -> one 16-byte shared load
//   fp32: [4c, 4c+4) and [D/2+4c, +4) -> two 16-byte shared loads, each
//         contiguous across the group's lanes (no bank conflicts)
// store(row, d0, x) writes 8 contiguous columns d0..d0+7 of a global row.
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
      x[2 * k] = bf16_lo_f(w[k]);
      x[2 * k + 1] = bf16_hi_f(w[k]);
    }
  }
  __device__ __forceinline__ static void store(__nv_bfloat16* row, int d0, const float (&x)[8]) {
    *reinterpret_cast<uint4*>(row + d0) = make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]),
                                                     pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
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
};

// Row of q / out (in rows of head_dim elements) for query row r of kv head h
// of sequence b: r = j * group + i is head h * group + i of new token j.
__device__ __forceinline__ size_t q_row(const DecodeArgs& a, int b, int h, int r) {
  const int j = r / a.group, i = r - j * a.group;
  return (static_cast<size_t>(b) * a.q_len + j) * a.num_q_heads + h * a.group + i;
}

struct SeqSpan {
  int p_lo;   // first page touched
  int np;     // pages touched (0: nothing to do)
  int t0;     // first token attended
  int L;      // context length
  bool bad;   // context length invalid
};

// Pages a sequence's query rows attend: with q_len new tokens (the last
// q_len of the context), token j sees the first L - q_len + 1 + j tokens and
// the window counts back from there, so the union starts at the first
// token's window.  A context shorter than q_len > 1 is invalid.
__device__ __forceinline__ SeqSpan seq_span(int L, int window, int max_blocks, int q_len) {
  SeqSpan s;
  s.L = L;
  s.bad = (L < 0) || (static_cast<long long>(L) > static_cast<long long>(max_blocks) * kPageTokens) ||
          (q_len > 1 && L < q_len);
  if (s.bad || L == 0) {
    s.p_lo = 0; s.np = 0; s.t0 = 0;
    return s;
  }
  const int first_end = L - q_len + 1;  // context of the first new token
  s.t0 = (window > 0 && first_end > window) ? first_end - window : 0;
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
template <int D, typename T, int G, int NCW, int NSTAGE, int MINB, Math MATH, int EXT>
__global__ void __launch_bounds__((NCW + 1) * 32, MINB)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                        const DecodeArgs a) {
  using S = Smem<D, T, G, NCW, NSTAGE, MATH, EXT>;
  constexpr int NT = (NCW + 1) * 32;
  constexpr int NC = NCW * 32;  // consumer threads
  using KV = KvElem<T, MATH>;
  constexpr uint32_t kTileBytes = kPageTokens * D * sizeof(KV);
  const int prec = G * 4 + min(G, a.rows) * D;  // floats of a partial record
  constexpr bool kMma = MATH != Math::kSimt;
  constexpr bool kFp8 = MATH == Math::kMma8;
  constexpr bool kQSmem = S::QS;
  // Independent QK^T accumulator chains per query n-tile: k-step i feeds
  // chain i mod kQAcc (each MMA waits on the one before it in its chain).
  constexpr int kQAcc = (kMma && G <= 8) ? 4 : 2;
  constexpr int NPAR = S::NPAR;
  static_assert(!kMma || (sizeof(T) == 2 && (NCW == 4 || NCW == 8) && G <= 16 && (D / S::NDP) % 16 == 0),
                "mma consumer shape");
  static_assert(!kFp8 || ((D % 128 == 0 || D == 64) && (D / S::NDP) % 32 == 0), "fp8 consumer shape");
  // FP8 tiles in shared memory: rows of kF8Row code bytes per column block,
  // swizzled as the tensor map writes them (128-byte rows: 16-byte chunk
  // XOR row mod 8; the 64-byte rows of head_dim 64: chunk XOR (row / 2) mod 4).
  constexpr int kF8Row = (D >= 128) ? 128 : 64;
  auto f8_off = [&](int t, int byte) -> uint32_t {
    const int sb = byte / kF8Row, chunk = (byte % kF8Row) >> 4;
    const int sw = (kF8Row == 128) ? (chunk ^ (t & 7)) : (chunk ^ ((t >> 1) & 3));
    return static_cast<uint32_t>(sb * (kPageTokens * kF8Row) + t * kF8Row + (sw << 4));
  };
  static_assert(NSTAGE % NPAR == 0, "alternate-page pairs need an even ring");
  static_assert(kMma || (S::GS <= 32 && (32 % S::GS) == 0 && S::NG * S::TPG == kPageTokens &&
                         G <= S::GS && (S::GS % G) == 0), "CUDA-core consumer shape");

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // TMA destinations (128-byte swizzle atoms) want 1024-byte aligned shared
  // addresses; the launch reserves 1 KB of slack for this round-up.
  const uint32_t raw_addr = smem_addr(smem_raw);
  S& s = *reinterpret_cast<S*>(smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nvh = a.num_kv_heads * a.subgroups;
  // The next decode on the stream may start its CTAs as SMs free up; it reads
  // nothing this grid writes before its own grid_dependency_wait.
  grid_launch_dependents();
  // Sequences without tiles (empty context: zero rows; invalid length: NaN
  // rows) are filled by CTA b mod grid, after the dependency wait: the
  // previous kernel on the stream may still read or write `out`.
  auto fill_empty_rows = [&](int nthreads, int t) {
    for (int b = blockIdx.x; b < a.num_seqs; b += gridDim.x) {
      const SeqSpan sp = seq_span(__ldg(a.context_lens + b), a.window, a.max_blocks, a.q_len);
      if (sp.np != 0) continue;
      const float fill = sp.bad ? __int_as_float(0x7fc00000) : 0.f;
      float vals[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) vals[e] = fill;
      T* row0 = static_cast<T*>(a.out) + static_cast<size_t>(b) * a.q_len * a.num_q_heads * D;
      for (int e = t * 8; e < a.q_len * a.num_q_heads * D; e += nthreads * 8) LaneMap<T, D>::store(row0, e, vals);
    }
  };

  if (tid == 0) {
    for (int st = 0; st < NSTAGE; ++st) {
      mbar_init(&s.full[st], 1);
      mbar_init(&s.empty[st], NCW / NPAR);  // the warps of the stage's pair
    }
    mbar_init(&s.csync, NCW);  // one arrival per consumer warp
    for (int p2 = 0; p2 < 4; ++p2) mbar_init(&s.qx_bar[p2 >> 1][p2 & 1], S::NDP);  // the warps of one tg
    mbar_init(&s.comb, 1);
    s.abort_flag = 0;
    s.b_start_s = -1;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  // ---- S1: request lookup and balanced partition ---------------------------
  // The split balances work units: every page of a (sequence, virtual head)
  // item is one, and every item also weighs seg_cost units for the time a
  // segment boundary costs -- when CTAs have pages enough for that to matter
  // (at least kWeightMinTiles each).  One scan sums pages and items together
  // (packed: pages << 24 | items); when the whole batch fits one pass of the
  // block, it also locates this CTA's first sequence.
  constexpr int kItemBits = 24;
  constexpr long long kItemMask = (1ll << kItemBits) - 1;
  constexpr int kWeightMinTiles = 4;
  const bool weighable = static_cast<long long>(a.num_seqs) * nvh <= kItemMask;
  auto packed_units = [&](int b) -> long long {
    const int np = seq_span(__ldg(a.context_lens + b), a.window, a.max_blocks, a.q_len).np;
    if (np <= 0) return 0;
    return (static_cast<long long>(np) * nvh << kItemBits) + (weighable ? nvh : 0);
  };
  long long P = 0, my_pexcl = 0, my_punits = 0;  // packed
  for (int base = 0; base < a.num_seqs; base += NT) {
    const int b = base + tid;
    const long long pu = b < a.num_seqs ? packed_units(b) : 0;
    long long tot;
    const long long excl = block_exclusive_scan<NT>(pu, s.scan, tot);
    my_pexcl = P + excl;
    my_punits = pu;
    P += tot;
  }
  const long long U_pages = P >> kItemBits;
  const int X = weighable && U_pages >= static_cast<long long>(kWeightMinTiles) * gridDim.x ? a.seg_cost : 0;
  auto unpack = [&](long long v) { return (v >> kItemBits) + X * (v & kItemMask); };
  const long long U = unpack(P), my_excl = unpack(my_pexcl), my_units = unpack(my_punits);
  if (U == 0) {
    grid_dependency_wait();
    fill_empty_rows(NT, tid);
    return;
  }
  const long long cap = (U + a.min_units - 1) / a.min_units;
  const int C = static_cast<int>(cap < gridDim.x ? cap : gridDim.x);
  if (static_cast<int>(blockIdx.x) >= C) {
    grid_dependency_wait();
    fill_empty_rows(NT, tid);
    return;
  }
  const Partition part{U, C};
  const long long u0 = part.start(blockIdx.x), u1 = part.start(blockIdx.x + 1);

  if (a.num_seqs <= NT) {
    if (my_units > 0 && my_excl <= u0 && u0 < my_excl + my_units) {
      s.b_start_s = tid;
      s.cum_start_s = my_excl;
    }
  } else {
    long long carry = 0;
    for (int base = 0; base < a.num_seqs; base += NT) {
      const int b = base + tid;
      const long long units = b < a.num_seqs ? unpack(packed_units(b)) : 0;
      long long tot;
      const long long excl = carry + block_exclusive_scan<NT>(units, s.scan, tot);
      if (units > 0 && excl <= u0 && u0 < excl + units) {
        s.b_start_s = b;
        s.cum_start_s = excl;
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
    long long u = u0, cum = s.cum_start_s;
    int b = s.b_start_s;
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
    bool ok = b >= 0;
    bool withheld = false;
    long long covered = 0;  // units walked, for the self-check
    while (ok && u < u1) {
      const SeqSpan sp = seq_span(length_of(b), a.window, a.max_blocks, a.q_len);
      const int w = sp.np + X;  // units of one (sequence, virtual head) item
      const long long ub = static_cast<long long>(w) * nvh;
      long long off = u - cum;
      const long long off_end = (u1 - cum < ub) ? (u1 - cum) : ub;
      for (int vh = static_cast<int>(off / w); ok && off < off_end; ++vh) {
        // An item's first seg_cost units stand for the time a segment boundary
        // costs and hold no tile; its pages are the units after them.
        const long long ibase = static_cast<long long>(vh) * w;
        const int r0 = static_cast<int>(off - ibase);
        const int r1 = static_cast<int>(off_end - ibase < w ? off_end - ibase : w);
        covered += r1 - r0;
        off = ibase + r1;
        const int pa = max(r0 - X, 0), pb = r1 - X;
        if (pb <= pa) continue;  // only the item's weight falls in this slice
        const long long item_u = cum + ibase + X;  // the item's first page unit
        const int c_first = part.owner(item_u);
        const int nsplit = part.owner(item_u + sp.np - 1) - c_first + 1;
        // first-segment slots, then last-segment slots (the item starts inside our slice)
        const int slot = static_cast<int>(blockIdx.x) + (u0 < item_u ? static_cast<int>(gridDim.x) : 0);
        const int h = vh / a.subgroups, sub = vh - h * a.subgroups;
        const int qr0 = sub * G;  // first query row of this subgroup
        const int gq = min(G, a.rows - qr0);
        const int* bt_row = a.block_tables + static_cast<size_t>(b) * a.max_blocks + sp.p_lo;
        // Segment stages: the item's pages, plus a kPad stage when NPAR = 2
        // and the count is odd.  The first NPAR stages carry the query rows
        // (kFirst) and the last NPAR close the segment (kLast), one of each
        // per warp pair.
        const int nst = (pb - pa + NPAR - 1) / NPAR * NPAR;
        auto put = [&](int pid, int p, bool pad) -> bool {
          if (static_cast<int>(blockIdx.x) == a.withhold_cta && issued == a.withhold_tile) {
            withheld = true;  // test hook: this tile never arrives
            return false;
          }
          bool live = wait_phase(&s.empty[stage], phase ^ 1u, &s.abort_flag, a.status, kStatusEmpty, a.wait_limit);
          live = __all_sync(0xffffffffu, live);
          if (!live) return false;
          const int i = p - pa;  // stage of the segment
          const bool first = i < NPAR;
          const bool bad = !pad && (pid < 0 || pid >= a.num_blocks);
          if (lane == 0) {
            const int first_tok = (sp.p_lo + p) * kPageTokens;
            StageHeader& hd = s.hdr[stage];
            hd.b = b;
            hd.vh = vh;
            hd.lo = pad ? 0 : max(sp.t0 - first_tok, 0);
            hd.hi = pad ? 0 : min(sp.L - first_tok, kPageTokens);
            hd.rel_end = pad ? 0 : sp.L - first_tok;
            hd.flags = (first ? kFirst : 0) | (i >= nst - NPAR ? kLast : 0) | (nsplit > 1 ? kSplit : 0) |
                       (bad ? kBadPage : 0) | (pad ? kPad : 0);
            hd.gq = gq;
            hd.nsplit = nsplit;
            hd.slot = slot;
            hd.c_first = c_first;
            hd.item_u = item_u;
            uint32_t bytes = (bad || pad) ? 0u : 2u * kTileBytes;
            if (first) bytes += static_cast<uint32_t>(gq) * D * sizeof(T);
            mbar_arrive_expect_tx(&s.full[stage], bytes);
          }
          __syncwarp();
          // One tensor copy per K (or V) tile, each issued by its own lane.
          // bf16 boxes cover (64 columns, 32 tokens, D/64 column blocks) of one
          // head, landing as D/64 swizzled [token][64] sub-tiles; fp8 boxes
          // the same with 128-code column blocks.
          if (!bad && !pad && lane < 2) {
            const bool is_v = lane == 1;
            KV* dst = is_v ? s.v[stage] : s.k[stage];
            if constexpr (kMma)
              tma_load_4d(dst, is_v ? &tmap_v : &tmap_k, 0, pid * kPageTokens, 0, h, &s.full[stage]);
            else
              tma_load_3d(dst, is_v ? &tmap_v : &tmap_k, 0, h, pid * kPageTokens, &s.full[stage]);
          }
          if (first && lane >= 16) {
            // The subgroup's rows, one bulk copy per new token they cover
            // (one copy in all for single-token decode).
            const int j = qr0 / a.group + (lane - 16);
            const int lo = max(j * a.group, qr0), hi = min(j * a.group + a.group, qr0 + gq);
            if (hi > lo) {
              const T* qsrc = static_cast<const T*>(a.q) + q_row(a, b, h, lo) * D;
              bulk_load(s.q[stage] + (lo - qr0) * D, qsrc, static_cast<uint32_t>(hi - lo) * D * sizeof(T),
                        &s.full[stage]);
            }
          }
          __syncwarp();
          ++issued;
          if (++stage == NSTAGE) {
            stage = 0;
            phase ^= 1u;
          }
          return true;
        };
        for (int p0 = pa; ok && p0 < pb; p0 += 32) {
          const int my_p = p0 + lane;
          const int my_id = (my_p < pb) ? __ldg(bt_row + my_p) : 0;
          // q, K and V may be written by the previous kernel on the stream;
          // the first copies wait for it (context lengths and block tables
          // were read before: the caller keeps them unchanged across it).
          // Before waiting, the first pages of the slice are prefetched into
          // L2, so their HBM latency overlaps that kernel's tail.  L2 is the
          // point of coherence: the copies after the wait still see every
          // write the previous kernel made.
          if (issued == 0) {
            const int n_pf = min(min(pb - p0, kPrefetchTiles), 32);
            if (lane < n_pf && my_id >= 0 && my_id < a.num_blocks) {
              if constexpr (kMma) {
                tma_prefetch_4d(&tmap_k, 0, my_id * kPageTokens, 0, h);
                tma_prefetch_4d(&tmap_v, 0, my_id * kPageTokens, 0, h);
              } else {
                tma_prefetch_3d(&tmap_k, 0, h, my_id * kPageTokens);
                tma_prefetch_3d(&tmap_v, 0, h, my_id * kPageTokens);
              }
            }
            grid_dependency_wait();
          }
          const int n = min(32, pb - p0);
          for (int jj = 0; jj < n; ++jj) {
            const int pid = __shfl_sync(0xffffffffu, my_id, jj);
            ok = put(pid, p0 + jj, false);
            if (!ok) break;
          }
        }
        // An odd segment gets one more stage, without tiles, for the second pair.
        if (NPAR == 2 && ok && ((pb - pa) & 1)) ok = put(0, pb, true);
      }
      u = cum + off_end;
      cum += ub;
      // next sequence with work
      do {
        ++b;
      } while (ok && u < u1 && b < a.num_seqs && seq_span(length_of(b), a.window, a.max_blocks, a.q_len).np == 0);
      if (b >= a.num_seqs) break;
    }
    // Self-check: the walk must have covered exactly this CTA's slice.
    if (covered != u1 - u0 && !withheld && !s.abort_flag && lane == 0) {
      atomicOr(a.status, kStatusWalk);
      s.abort_flag = 1;
    }
    // The consumers learn that the work is over from one more stage that
    // carries no tiles (how many pages the slice holds depends on the items
    // it crosses).
    int n_end = 0;  // end stages sent, one per warp pair
    if (ok && __all_sync(0xffffffffu, !s.abort_flag)) {
      for (int e = 0; e < NPAR; ++e) {
        ok = wait_phase(&s.empty[stage], phase ^ 1u, &s.abort_flag, a.status, kStatusEmpty, a.wait_limit);
        if (!__all_sync(0xffffffffu, ok)) break;
        if (lane == 0) {
          s.hdr[stage].flags = kEnd;
          mbar_arrive(&s.full[stage]);
        }
        ++n_end;
        if (++stage == NSTAGE) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // Let every copy this warp issued land before the CTA can exit.  Once an
    // end stage went out, its own stage's last tile had been released, and
    // its full barrier has moved on a phase: drain only the others.
    if (lane == 0) {
      const long long cap = NSTAGE - n_end;
      const long long n_drain = issued < cap ? issued : cap;
      for (long long k = 1; k <= n_drain; ++k) {
        const long long idx = issued - k;  // stage index of the k-th most recent copy
        const int st = static_cast<int>(idx % NSTAGE);
        const uint32_t ph = static_cast<uint32_t>((idx / NSTAGE) & 1);
        volatile int never = 0;
        if (!wait_phase(&s.full[st], ph, &never, a.status, kStatusDrain, kDrainLimitCycles)) break;
      }
    }
    return;
  }

  // ===================== consumer warps (S3 - S9) =============================
  const int ct = tid;  // 0 .. NC-1
  const float kNegInf = -__int_as_float(0x7f800000);
  const float kNaN = __int_as_float(0x7fc00000);
  uint32_t sync_phase = 0;
  // Rendezvous of the consumer warps.  One elected lane per warp arrives
  // (after __syncwarp has ordered the warp's shared-memory writes): 128
  // arrivals on one mbarrier word serialise and cost microseconds.
  auto cons_sync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.csync);
    bool r = wait_phase(&s.csync, sync_phase, &s.abort_flag, a.status, kStatusSync, a.wait_limit);
    r = __all_sync(0xffffffffu, r);
    sync_phase ^= 1u;
    return r;
  };
  if (ct == 0) s.pend_n = 0;  // only thread 0 touches it until the final rendezvous
  // Global memory this grid shares with the previous kernel on the stream
  // (out, the workspace) is touched only after this point.
  grid_dependency_wait();
  fill_empty_rows(NC, ct);

  // ---- per-consumer constants ----------------------------------------------
  // CUDA-core consumer (fp32): row group j (GS lanes), lane c owns 8 columns.
  constexpr int GS = S::GS, NG = S::NG, TPG = S::TPG;
  const int j = ct / GS;
  const int c = ct % GS;
  constexpr int kSpread = (GS / G) > 0 ? GS / G : 1;
  const int iq = c / kSpread;
  const bool owner = (c % kSpread) == 0;
  // mma consumer (bf16, FP8): warp = (token half tg, page pair par, head_dim
  // part dp); par is 0 unless the pairs take alternate stages (NPAR = 2).
  // The products are taken transposed, with the warp's 16 tokens as the M
  // dimension and the query group as N (8 or 16): S^T = K Q^T over the full
  // head_dim (repeated by the dp warps, or at head_dim 512 split over them
  // and summed), O^T = V^T P^T for the warp's D / NDP output rows of O^T.
  // No M padding for groups of up to 8.
  constexpr int NDP = S::NDP;
  constexpr int kDPart = D / NDP;        // O^T rows (head_dim columns of O) per warp
  constexpr int kKSteps = D / 16;        // k-steps of S^T over head_dim
  constexpr int kMt = kDPart / 16;       // 16-row m-tiles of O^T per warp
  constexpr int NQT = (G > 8) ? 2 : 1;   // 8-query n-tiles
  constexpr bool kSplitQK = S::SQK;
  constexpr int kQKS = kSplitQK ? kKSteps / NDP : kKSteps;  // k-steps of this warp's share of S^T
  static_assert(!kSplitQK || (kQKS % 2 == 0 && NQT == S::QXN), "split QK^T shape");
  const int tg = warp & 1, par = (warp >> 1) % NPAR, dp = warp / (2 * NPAR);
  const int kq0 = kSplitQK ? dp * kQKS : 0;  // first k-step of the share
  const int gid = lane >> 2, tig = lane & 3;

  int stage = kMma ? par : 0;  // a warp pair walks its own stages of the ring
  uint32_t phase = 0;
  int qx_t = 0;          // split QK^T: tiles exchanged so far (buffer parity)
  uint32_t qx_ph = 0u;   // and the phase bit of each parity's barrier
  int pbuf_par = 0, seg_par = 0;
  bool alive = true, more = true;
  // One iteration per (sequence, virtual head) segment: the query fragments
  // and accumulators are scoped to it, so they are dead in the epilogue.
  while (alive && more) {
  float qf[kMma ? 1 : G][8];
  float acc[kMma ? 1 : G][8];
  uint32_t qb[kMma && !kQSmem ? kQKS : 1][NQT][2];  // Q^T as the B operand of S^T = K Q^T
  float oacc[kMma ? kMt : 1][NQT][4];       // O^T accumulators
  float m_run = kNegInf, l_run = 0.f;       // simt: the lane's query
  float sl2 = a.scale_log2;                 // score factor into the log2 domain
  float sq[kFp8 ? NQT : 1][2];              // fp8: the factor of the lane's query columns
  float vsc = 1.f;                          // value factor (fp8: v_scale[h])
  // Causal offset of a query row's new token: q_len - 1 - j (0 for
  // single-token decode); its keys end that many tokens before the context's.
  int qoff[kMma ? NQT : 1][2];              // mma: queries 8n + 2tig + {0,1}; simt: [0][0] is the lane's
  float mq[NQT][2], lq[NQT][2];             // mma: queries 8n + 2tig + {0,1}
  bool poison = false;
  int hold_stage = 0;
  StageHeader hd;
  do {
    bool ok = wait_phase(&s.full[stage], phase, &s.abort_flag, a.status, kStatusFull, a.wait_limit);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      alive = false;
      break;
    }
    hd = s.hdr[stage];
    if (hd.flags & kEnd) {
      more = false;
      break;
    }

    if constexpr (!kMma) {
      // ====================== CUDA-core consumer ==============================
      using Map = LaneMap<T, D>;
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
        qoff[0][0] = a.q_len - 1 - ((hd.vh % a.subgroups) * G + iq) / a.group;
      }
      if (hd.flags & kBadPage) {
        poison = true;
      } else if (!(hd.flags & kPad)) {
        const int end_q = hd.rel_end - qoff[0][0];                      // keys t < end_q
        const int beg_q = a.window > 0 ? end_q - a.window : -(1 << 30);  // and t >= beg_q
        const T* ks = s.k[stage];
        const T* vs = s.v[stage];
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
          sc[tt] = (t >= hd.lo && t < hd.hi && t >= beg_q && t < end_q) ? r : kNegInf;
        }
        float mloc = sc[0];
#pragma unroll
        for (int tt = 1; tt < TPG; ++tt) mloc = fmaxf(mloc, sc[tt]);
        const float m_new = fmaxf(m_run, mloc);
        const float m_use = (m_new == kNegInf) ? 0.f : m_new;
        const float alpha = ex2(m_run - m_use);
        float p[TPG];
        float psum = 0.f;
#pragma unroll
        for (int tt = 0; tt < TPG; ++tt) {
          p[tt] = ex2(sc[tt] - m_use);
          psum += p[tt];
        }
        l_run = l_run * alpha + psum;
        m_run = m_new;
        if (owner) {
#pragma unroll
          for (int tt = 0; tt < TPG; ++tt) s.pbuf[pbuf_par][j][iq][tt] = p[tt];
          s.abuf[pbuf_par][j][iq] = alpha;
        }
        __syncwarp();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int i = 0; i < G; ++i) {
            const float ai = s.abuf[pbuf_par][j][i];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][e] *= ai;
          }
        }
#pragma unroll
        for (int tt = 0; tt < TPG; ++tt) {
          const int t = j + NG * tt;
          if (t >= hd.lo && t < hd.hi) {
            float vx[8];
            Map::load(vs + t * D, c, vx);
#pragma unroll
            for (int i = 0; i < G; ++i) {
              const float pi = s.pbuf[pbuf_par][j][i][tt];
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(pi, vx[e], acc[i][e]);
            }
          }
        }
        pbuf_par ^= 1;
      }
    } else {
      // ======================== tensor-core consumer ==========================
      if (hd.flags & kFirst) {
        // Q^T as the B operand (k = head_dim, n = query): lane holds query
        // 8n + gid, columns 16ks + 2tig (+1) and +8; queries past the live
        // group are zero.
        const uint32_t* q32 = reinterpret_cast<const uint32_t*>(s.q[stage]);
        if constexpr (kFp8) {
          // f16 operands of mma.sync m16n8k16 (the codes are widened to f16
          // exactly): the lane holds query 8n + gid, columns 16ks + 4tig,
          // +1 (b0) and 16ks + 4tig + 2, +3 (b1) of k-step ks -- the columns
          // its K codes sit in (S3).  Each query row is scaled by a power of
          // two 2^e that puts its largest magnitude in [2^14, 2^15), so f16
          // holds the bf16 values exactly down to 2^-28 of the largest (rows
          // below 2^-100 count as zero); the score of a query column is
          // scaled back by 2^-e with the softmax factor.
          const int h = hd.vh / a.subgroups;
          const float sk = a.scale_log2 * __ldg(a.k_scale + h);
          vsc = __ldg(a.v_scale + h);
#pragma unroll
          for (int n = 0; n < NQT; ++n) {
            const int qr = 8 * n + gid;
            const bool ok = qr < hd.gq;
            uint2 w[kKSteps];
            float mx = 0.f;
#pragma unroll
            for (int ks = 0; ks < kKSteps; ++ks) {
              w[ks] = ok ? *reinterpret_cast<const uint2*>(q32 + ((qr * D + ks * 16 + 4 * tig) >> 1))
                         : make_uint2(0u, 0u);
              mx = fmaxf(mx, fmaxf(fmaxf(fabsf(bf16_lo_f(w[ks].x)), fabsf(bf16_hi_f(w[ks].x))),
                                   fmaxf(fabsf(bf16_lo_f(w[ks].y)), fabsf(bf16_hi_f(w[ks].y)))));
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 127;  // floor(log2 mx)
            const int e = (mx >= 0x1p-100f && mx <= 0x1p+100f) ? 14 - ex : 0;
            const float sc = pow2f(e);
#pragma unroll
            for (int ks = 0; ks < kKSteps; ++ks) {
              qb[ks][n][0] = pack_f16(bf16_lo_f(w[ks].x) * sc, bf16_hi_f(w[ks].x) * sc);
              qb[ks][n][1] = pack_f16(bf16_lo_f(w[ks].y) * sc, bf16_hi_f(w[ks].y) * sc);
            }
            // the factor of this lane's score columns, queries 8n + 2tig (+1),
            // whose exponents sit with the lanes of gid 2tig (+1)
#pragma unroll
            for (int jq = 0; jq < 2; ++jq) {
              const int eq = __shfl_sync(0xffffffffu, e, (2 * tig + jq) * 4);
              sq[n][jq] = sk * pow2f(-eq);
            }
          }
        } else if constexpr (kQSmem) {
          // Every consumer warp is past the previous segment's epilogue
          // rendezvous, so nobody reads the buffer any more: copy the rows in
          // 16-byte chunks (rows past the live group are zero), then meet.
          char* qs = reinterpret_cast<char*>(s.qs);
          const T* src = s.q[stage];
          for (int e = ct; e < G * (D / 8); e += NC) {
            const int row = e / (D / 8), c8 = e - row * (D / 8);
            const uint4 val = row < hd.gq ? *reinterpret_cast<const uint4*>(src + row * D + c8 * 8)
                                          : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(qs + (c8 >> 3) * (G * 128) + row * 128 + (((c8 & 7) ^ (row & 7)) << 4)) = val;
          }
          if (!cons_sync()) {
            alive = false;
            break;
          }
        } else {
#pragma unroll
          for (int n = 0; n < NQT; ++n) {
            const int qr = 8 * n + gid;
            const bool ok = qr < hd.gq;
#pragma unroll
            for (int ks = 0; ks < kQKS; ++ks) {
              const int col = (kq0 + ks) * 16 + 2 * tig;
              qb[ks][n][0] = ok ? q32[(qr * D + col) >> 1] : 0u;
              qb[ks][n][1] = ok ? q32[(qr * D + col + 8) >> 1] : 0u;
            }
          }
        }
#pragma unroll
        for (int mt = 0; mt < kMt; ++mt)
#pragma unroll
          for (int n = 0; n < NQT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[mt][n][e] = 0.f;
#pragma unroll
        for (int n = 0; n < NQT; ++n) {
          mq[n][0] = mq[n][1] = kNegInf;
          lq[n][0] = lq[n][1] = 0.f;
#pragma unroll
          for (int jq = 0; jq < 2; ++jq)
            qoff[n][jq] = a.q_len - 1 - ((hd.vh % a.subgroups) * G + 8 * n + 2 * tig + jq) / a.group;
        }
        poison = false;
      }
      if (hd.flags & kBadPage) {
        poison = true;
      } else if (!(hd.flags & kPad)) {
        // S3: S^T = K Q^T for this warp's 16 tokens of the page; even and odd
        // k-steps accumulate separately (two short MMA chains instead of one).
        auto qk = [&](const uint32_t kbase, float (&sc)[NQT][kQAcc][4]) {
#pragma unroll
          for (int n = 0; n < NQT; ++n)
#pragma unroll
            for (int hh = 0; hh < kQAcc; ++hh)
#pragma unroll
              for (int e = 0; e < 4; ++e) sc[n][hh][e] = 0.f;
        if constexpr (kFp8) {
          // K codes, [token][head_dim] bytes in 128-byte swizzled rows: one
          // ldmatrix.x4 gives, for the warp's 16 tokens, the codes of columns
          // 4tig .. +3 of two 16-column chunks (tokens gid and gid + 8); each
          // register widens to the f16 pairs of k-slots 2tig, +1 (columns
          // 4tig, +1) and 2tig + 8, +9 (columns 4tig + 2, +3).
          const int mi = lane >> 3, r = lane & 7;
          const int t = 16 * tg + ((mi & 1) << 3) + r;
#pragma unroll
          for (int kp = 0; kp < kKSteps / 2; ++kp) {
            uint32_t ak[4];
            ldmatrix_x4(kbase + f8_off(t, kp * 32 + ((mi >> 1) << 4)), ak);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              uint32_t af[4];
              e4m3x4_to_f16(ak[2 * hf], af[0], af[2]);
              e4m3x4_to_f16(ak[2 * hf + 1], af[1], af[3]);
              const int ks = 2 * kp + hf;
#pragma unroll
              for (int n = 0; n < NQT; ++n) mma_f16(sc[n][ks % kQAcc], af, qb[ks][n][0], qb[ks][n][1]);
            }
          }
        } else if constexpr (kQSmem) {
          // Q^T B fragments by ldmatrix from the swizzled copy: matrices
          // (queries 8n..+7) x (columns 16ks, 16ks + 8, 16ks + 16, 16ks + 24)
          // give b0b1 / b2b3 of k-steps ks and ks + 1.
          const int mi = lane >> 3, r = lane & 7;
          const int t = 16 * tg + ((mi & 1) << 3) + r;
          const uint32_t qbase = smem_addr(s.qs);
#pragma unroll 4
          for (int kk = 0; kk < kQKS; kk += 2) {
            const int ks = kq0 + kk;
            uint32_t qf[NQT][4];
#pragma unroll
            for (int n = 0; n < NQT; ++n) {
              const int row = 8 * n + r;
              const int d = ks * 16 + ((mi & 1) << 3) + ((mi >> 1) << 4);
              ldmatrix_x4(qbase + (d / kSwizzleCols) * (G * 128) + row * 128 + ((((d % kSwizzleCols) >> 3) ^ (row & 7)) << 4),
                          qf[n]);
            }
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int d = (ks + h2) * 16 + ((mi >> 1) << 3);
              const int sb = d / kSwizzleCols, chunk = (d % kSwizzleCols) >> 3;
              uint32_t ak[4];
              ldmatrix_x4(kbase + sb * (kPageTokens * 128) + t * 128 + ((chunk ^ (t & 7)) << 4), ak);
#pragma unroll
              for (int n = 0; n < NQT; ++n) mma_bf16(sc[n][(kk + h2) % kQAcc], ak, qf[n][2 * h2], qf[n][2 * h2 + 1]);
            }
          }
        } else {
          const int mi = lane >> 3, r = lane & 7;
          const int t = 16 * tg + ((mi & 1) << 3) + r;  // token row this lane addresses
#pragma unroll
          for (int ks = 0; ks < kQKS; ++ks) {
            const int d = (kq0 + ks) * 16 + ((mi >> 1) << 3);
            const int sb = d / kSwizzleCols, chunk = (d % kSwizzleCols) >> 3;
            uint32_t ak[4];
            ldmatrix_x4(kbase + sb * (kPageTokens * 128) + t * 128 + ((chunk ^ (t & 7)) << 4), ak);
#pragma unroll
            for (int n = 0; n < NQT; ++n) mma_bf16(sc[n][ks % kQAcc], ak, qb[ks][n][0], qb[ks][n][1]);
          }
        }
        };
        float sacc[NQT][kQAcc][4];
        qk(smem_addr(s.k[stage]), sacc);
        if constexpr (kSplitQK) {
          // The dp warps of this token half add their partial scores in dp
          // order, so each gets the same bits.  A warp is at most one tile
          // ahead of the others (it cannot pass the next tile's barrier
          // before they reach it), hence two buffers.
          const int xq = qx_t & 1;
#pragma unroll
          for (int n = 0; n < NQT; ++n) {
            float v4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float x = sacc[n][0][e];
#pragma unroll
              for (int c2 = 1; c2 < kQAcc; ++c2) x += sacc[n][c2][e];
              v4[e] = x;
            }
            s.qx[xq][tg][dp][lane][n] = make_float4(v4[0], v4[1], v4[2], v4[3]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.qx_bar[xq][tg]);
          const bool xok = wait_phase(&s.qx_bar[xq][tg], (qx_ph >> xq) & 1u, &s.abort_flag, a.status, kStatusSync,
                                      a.wait_limit);
          if (!__all_sync(0xffffffffu, xok)) {
            alive = false;
            break;
          }
          qx_ph ^= 1u << xq;
          ++qx_t;
#pragma unroll
          for (int n = 0; n < NQT; ++n) {
            float4 tot = s.qx[xq][tg][0][lane][n];
#pragma unroll
            for (int d2 = 1; d2 < NDP; ++d2) {
              const float4 x = s.qx[xq][tg][d2][lane][n];
              tot.x += x.x;
              tot.y += x.y;
              tot.z += x.z;
              tot.w += x.w;
            }
            sacc[n][0][0] = tot.x;
            sacc[n][0][1] = tot.y;
            sacc[n][0][2] = tot.z;
            sacc[n][0][3] = tot.w;
          }
        }
        // S4 + S5: mask and scale; online softmax per query column.  Lane
        // holds tokens 16tg + gid (values 0, 1) and + 8 (values 2, 3) of
        // queries 8n + 2tig (values 0, 2) and + 1 (values 1, 3).  Query row q
        // of new token j sees the page's tokens t with beg <= t < end,
        // end = rel_end - (q_len - 1 - j), beg = end - window (for
        // single-token decode exactly [lo, hi)).
        const int t_lo = 16 * tg + gid, t_hi = t_lo + 8;
        const int wlim = a.window > 0 ? a.window : (1 << 30);
        // Interior page: every token is live for every query row (rows past
        // the live group have zero queries, so finite scores that no output
        // reads), and the masks are skipped.
        const bool interior = hd.rel_end - (a.q_len - 1) >= kPageTokens && hd.rel_end <= wlim;
        float sv[NQT][2][2];
        bool up = false;  // some score above its column's running maximum
#pragma unroll
        for (int n = 0; n < NQT; ++n) {
#pragma unroll
          for (int jq = 0; jq < 2; ++jq) {
            const int q = 8 * n + 2 * tig + jq;
            const bool qok = q < hd.gq;
            const int end = hd.rel_end - qoff[n][jq], beg = end - wlim;
            const float f = kFp8 ? sq[kFp8 ? n : 0][jq] : sl2;
            float s0 = sacc[n][0][jq], s1 = sacc[n][0][jq + 2];
#pragma unroll
            for (int c = 1; c < (kSplitQK ? 1 : kQAcc); ++c) {
              s0 += sacc[n][c][jq];
              s1 += sacc[n][c][jq + 2];
            }
            if (interior) {
              sv[n][jq][0] = s0 * f;
              sv[n][jq][1] = s1 * f;
            } else {
              sv[n][jq][0] = (qok && t_lo >= beg && t_lo < end) ? s0 * f : kNegInf;
              sv[n][jq][1] = (qok && t_hi >= beg && t_hi < end) ? s1 * f : kNegInf;
            }
            up |= fmaxf(sv[n][jq][0], sv[n][jq][1]) > mq[n][jq];
          }
        }
        float pr[NQT][4];
        if (__any_sync(0xffffffffu, up)) {
          // A column maximum moves: reduce it over the 16 tokens (three
          // shuffles), rescale l and O by 2^(m_old - m_new).
          float al[NQT][2];
#pragma unroll
          for (int n = 0; n < NQT; ++n) {
#pragma unroll
            for (int jq = 0; jq < 2; ++jq) {
              float mx = fmaxf(sv[n][jq][0], sv[n][jq][1]);
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
              const float mn = fmaxf(mq[n][jq], mx);
              const float mu = (mn == kNegInf) ? 0.f : mn;
              al[n][jq] = ex2(mq[n][jq] - mu);
              pr[n][jq] = ex2(sv[n][jq][0] - mu);
              pr[n][jq + 2] = ex2(sv[n][jq][1] - mu);
              lq[n][jq] = lq[n][jq] * al[n][jq] + pr[n][jq] + pr[n][jq + 2];
              mq[n][jq] = mn;
            }
          }
#pragma unroll
          for (int mt = 0; mt < kMt; ++mt)
#pragma unroll
            for (int n = 0; n < NQT; ++n) {
              oacc[mt][n][0] *= al[n][0];
              oacc[mt][n][1] *= al[n][1];
              oacc[mt][n][2] *= al[n][0];
              oacc[mt][n][3] *= al[n][1];
            }
        } else {
          // No maximum moves (the usual case once a segment is under way):
          // the weights are taken against the running maxima as they stand.
#pragma unroll
          for (int n = 0; n < NQT; ++n) {
#pragma unroll
            for (int jq = 0; jq < 2; ++jq) {
              const float mu = (mq[n][jq] == kNegInf) ? 0.f : mq[n][jq];
              pr[n][jq] = ex2(sv[n][jq][0] - mu);
              pr[n][jq + 2] = ex2(sv[n][jq][1] - mu);
              lq[n][jq] += pr[n][jq] + pr[n][jq + 2];
            }
          }
        }
        // S6: O^T[this warp's rows] += V^T P^T over the page's 16 tokens of
        // this warp.  V rows of masked tokens may hold anything (NaN in unused
        // slots) and 0 * NaN is NaN inside the MMA: clear those tokens in the
        // V^T fragments.  This lane's fragments carry tokens 16tg + 2tig (+1)
        // and (+8, +9).
        const int tl = 16 * tg + 2 * tig;
        auto pv = [&](const int st, const StageHeader& h, const float (&p)[NQT][4]) {
          const uint32_t mlo = ((tl >= h.lo && tl < h.hi) ? 0x0000ffffu : 0u) |
                               ((tl + 1 >= h.lo && tl + 1 < h.hi) ? 0xffff0000u : 0u);
          const uint32_t mhi = ((tl + 8 >= h.lo && tl + 8 < h.hi) ? 0x0000ffffu : 0u) |
                               ((tl + 9 >= h.lo && tl + 9 < h.hi) ? 0xffff0000u : 0u);
          const bool full_page = h.lo == 0 && h.hi == kPageTokens;  // no token to clear
        if constexpr (kFp8) {
          // P^T as f16 B fragments (11 significant bits of the weights): the
          // S^T accumulator layout transposed per 8x8 block with movmatrix, so a
          // lane holds, for query gid, tokens 2tig, 2tig + 1 and 2tig + 8, +9.
          uint32_t pb[NQT][2];
#pragma unroll
          for (int n = 0; n < NQT; ++n) {
            pb[n][0] = movmatrix_trans(pack_f16(p[n][0], p[n][1]));
            pb[n][1] = movmatrix_trans(pack_f16(p[n][2], p[n][3]));
          }
          // V^T A fragments by ldmatrix.trans over byte pairs: an 8x8 matrix of
          // 16-bit elements is 8 tokens x 16 codes, and transposed a lane gets
          // codes 2gid, 2gid + 1 (bytes 0, 1) of token 2tig and the same of
          // token 2tig + 1 (bytes 2, 3).  A byte permute pairs the two tokens
          // per code, and widening gives f16 pairs (tokens 2tig, +1) of
          // columns 2gid and 2gid + 1: rows gid and gid + 8 of m-tile mt are
          // columns 16mt + 2gid and 16mt + 2gid + 1 of the warp's part.  Codes
          // of tokens outside the page's range are cleared (they may be NaN).
          const int mi = lane >> 3, r = lane & 7;
          const int t = 16 * tg + ((mi & 1) << 3) + r;  // token row this lane addresses
          const uint32_t vbase = smem_addr(s.v[st]);
#pragma unroll
          for (int mp = 0; mp < kMt / 2; ++mp) {  // two 16-code blocks per ldmatrix.x4
            uint32_t w[4];  // (tokens 0-7, 8-15) of block 2mp, then of block 2mp + 1
            ldmatrix_x4_trans(vbase + f8_off(t, dp * kDPart + mp * 32 + ((mi >> 1) << 4)), w);
            if (!full_page) {
              w[0] &= mlo;
              w[1] &= mhi;
              w[2] &= mlo;
              w[3] &= mhi;
            }
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              uint32_t av[4];
              e4m3x4_to_f16(__byte_perm(w[2 * hb], 0u, 0x3120u), av[0], av[1]);
              e4m3x4_to_f16(__byte_perm(w[2 * hb + 1], 0u, 0x3120u), av[2], av[3]);
#pragma unroll
              for (int n = 0; n < NQT; ++n) mma_f16(oacc[2 * mp + hb][n], av, pb[n][0], pb[n][1]);
            }
          }
        } else {
          // P^T as the B operand (k = token, n = query): the S^T accumulator
          // layout transposed per 8x8 block with movmatrix, split bf16 hi + lo so
          // hi + lo carries ~16 significant bits of p.
          uint32_t pbh[NQT][2], pbl[NQT][2];
#pragma unroll
          for (int n = 0; n < NQT; ++n) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {  // tokens 0-7 then 8-15 of the warp
              const float p0 = p[n][2 * hh], p1 = p[n][2 * hh + 1];
              const uint32_t h = pack_bf16(p0, p1);
              const uint32_t l = pack_bf16(p0 - bf16_lo_f(h), p1 - bf16_hi_f(h));
              pbh[n][hh] = movmatrix_trans(h);
              pbl[n][hh] = movmatrix_trans(l);
            }
          }
          // S6: O^T[this warp's rows] += V^T P^T over the 16 tokens.
          const int mi = lane >> 3, r = lane & 7;
          const int t = 16 * tg + ((mi >> 1) << 3) + r;
#pragma unroll
          for (int mt = 0; mt < kMt; ++mt) {
            const int d = dp * kDPart + mt * 16 + ((mi & 1) << 3);
            const int sb = d / kSwizzleCols, chunk = (d % kSwizzleCols) >> 3;
            uint32_t av[4];
            ldmatrix_x4_trans(smem_addr(s.v[st]) + sb * (kPageTokens * 128) + t * 128 + ((chunk ^ (t & 7)) << 4), av);
            if (!full_page) {
              av[0] &= mlo;
              av[1] &= mlo;
              av[2] &= mhi;
              av[3] &= mhi;
            }
#pragma unroll
            for (int n = 0; n < NQT; ++n) {
              mma_bf16(oacc[mt][n], av, pbh[n][0], pbh[n][1]);
              mma_bf16(oacc[mt][n], av, pbl[n][0], pbl[n][1]);
            }
          }
        }
        };
        pv(stage, hd, pr);
      }
    }

    // release the stage to the producer (the CUDA-core consumer keeps a
    // segment's last stage: its tiles hold the row-group merge, after which
    // the stage is released)
    __syncwarp();
    if (!kMma && (hd.flags & kLast))
      hold_stage = stage;
    else if (lane == 0)
      mbar_arrive(&s.empty[stage]);
    stage += NPAR;
    if (stage >= NSTAGE) {
      stage -= NSTAGE;
      phase ^= 1u;
    }
  } while (!(hd.flags & kLast));
  if (!alive || !more) break;

  // ---- end of a (sequence, virtual head) segment ----------------------------
  const int h = hd.vh / a.subgroups, sub = hd.vh - h * a.subgroups;
  const int r0 = sub * G;  // first query row of this subgroup
  const bool split = (hd.flags & kSplit) != 0;
  // red_m / red_l / xbuf are double-buffered: a thread can only reach the next
  // segment but one after every thread finished reading this segment's copy.
  float (*rm)[G] = s.red_m[seg_par];
  float (*rl)[G] = s.red_l[seg_par];
  const int xp = seg_par;
  seg_par ^= 1;
  if constexpr (!kMma) {
    // ---- merge the row groups in a fixed order ----
    // The row groups of a warp are summed with shuffles; each warp leaves its
    // [G][D] sum in the held stage's K (then V) tile, and every output adds
    // the warps' sums in warp order, so the bits are the same on every run.
    if (owner) {
      rm[j][iq] = m_run;
      rl[j][iq] = poison ? kNaN : l_run;
    }
    if (!cons_sync()) break;
    constexpr int kRegions = kPageTokens * static_cast<int>(sizeof(T)) / (4 * G);  // [G][D] sums per tile
    static_assert(2 * kRegions >= NCW, "a stage's K and V tiles must hold every warp's sum");
    auto region = [&](int w) -> float* {
      return (w < kRegions) ? reinterpret_cast<float*>(s.k[hold_stage]) + w * G * D
                            : reinterpret_cast<float*>(s.v[hold_stage]) + (w - kRegions) * G * D;
    };
    float* wsum = region(warp);
#pragma unroll
    for (int i = 0; i < G; ++i) {
      float Mx = kNegInf;
#pragma unroll
      for (int g2 = 0; g2 < NG; ++g2) Mx = fmaxf(Mx, rm[g2][i]);
      const float Ms = (Mx == kNegInf) ? 0.f : Mx;
      const float f = exp2f(rm[j][i] - Ms);
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = acc[i][e] * f;
#pragma unroll
      for (int o = GS; o < 32; o <<= 1)
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] += __shfl_xor_sync(0xffffffffu, x[e], o);
      if (lane < GS) {
        *reinterpret_cast<float4*>(wsum + i * D + LaneMap<T, D>::col(c, 0)) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4*>(wsum + i * D + LaneMap<T, D>::col(c, 4)) = make_float4(x[4], x[5], x[6], x[7]);
      }
      if (ct == i) {
        float L = 0.f;
#pragma unroll
        for (int g2 = 0; g2 < NG; ++g2) L += rl[g2][i] * exp2f(rm[g2][i] - Ms);
        s.fin_m[i] = Mx;  // -inf for a row with no key in this share
        s.fin_l[i] = L;
      }
    }
    if (!cons_sync()) break;
    // ---- S9 / S7: final rows, or this CTA's normalised partial ----
    for (int e0 = ct * 8; e0 < G * D; e0 += NC * 8) {
      const int i = e0 / D, d0 = e0 - i * D;
      const float L = s.fin_l[i];
      float val[8];
      {
        const float4 a4 = *reinterpret_cast<const float4*>(region(0) + e0);
        const float4 b4 = *reinterpret_cast<const float4*>(region(0) + e0 + 4);
        val[0] = a4.x; val[1] = a4.y; val[2] = a4.z; val[3] = a4.w;
        val[4] = b4.x; val[5] = b4.y; val[6] = b4.z; val[7] = b4.w;
      }
#pragma unroll
      for (int w = 1; w < NCW; ++w) {
        const float4 a4 = *reinterpret_cast<const float4*>(region(w) + e0);
        const float4 b4 = *reinterpret_cast<const float4*>(region(w) + e0 + 4);
        val[0] += a4.x; val[1] += a4.y; val[2] += a4.z; val[3] += a4.w;
        val[4] += b4.x; val[5] += b4.y; val[6] += b4.z; val[7] += b4.w;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) val[e] = (L == 0.f) ? 0.f : val[e] / L;  // l = 0: a row with no key here
      if (i >= hd.gq) continue;
      if (!split) {
        T* row = static_cast<T*>(a.out) + q_row(a, hd.b, h, r0 + i) * D;
        LaneMap<T, D>::store(row, d0, val);
      } else {
        float* po = a.part + static_cast<size_t>(hd.slot) * prec + G * 4 + i * D + d0;
        *reinterpret_cast<float4*>(po) = make_float4(val[0], val[1], val[2], val[3]);
        *reinterpret_cast<float4*>(po + 4) = make_float4(val[4], val[5], val[6], val[7]);
        if (d0 == 0)
          *reinterpret_cast<float4*>(a.part + static_cast<size_t>(hd.slot) * prec + i * 4) =
              make_float4(s.fin_m[i], L, 0.f, 0.f);
      }
    }
    // The held stage goes back to the producer, whose next copy into it is
    // an async-proxy write after these generic ones.
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[hold_stage]);
  } else {
    // ---- token-half 1 hands its O^T fragments to token-half 0 ----
    // l: each lane summed its two tokens; the column sums run over the 8
    // lanes that share tig.
    float lfull[NQT][2];
#pragma unroll
    for (int n = 0; n < NQT; ++n)
#pragma unroll
      for (int jq = 0; jq < 2; ++jq) {
        float l = lq[n][jq];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        lfull[n][jq] = l;
      }
    if constexpr (NPAR == 2) {
      // ---- the second warp pair hands its partial to the first ----
      float* xa = &s.xbuf[xp][dp][tg][0][0][0];
      if (par == 1) {
        if (dp == 0 && gid == 0) {
#pragma unroll
          for (int n = 0; n < NQT; ++n)
#pragma unroll
            for (int jq = 0; jq < 2; ++jq) {
              const int q = 8 * n + 2 * tig + jq;
              rm[2 + tg][q] = mq[n][jq];
              rl[2 + tg][q] = poison ? kNaN : lfull[n][jq];
            }
        }
#pragma unroll
        for (int mt = 0; mt < kMt; ++mt)
#pragma unroll
          for (int n = 0; n < NQT; ++n)
            *reinterpret_cast<float4*>(xa + (mt * 32 + lane) * S::XV + 4 * n) =
                make_float4(oacc[mt][n][0], oacc[mt][n][1], oacc[mt][n][2], oacc[mt][n][3]);
      }
      if (!cons_sync()) break;
      if (par == 0) {
        // (m, l, O) of both pairs against their larger maximum; a pair that
        // saw no key of a row (m = -inf) weighs nothing
        float f0[NQT][2], f1[NQT][2];
#pragma unroll
        for (int n = 0; n < NQT; ++n)
#pragma unroll
          for (int jq = 0; jq < 2; ++jq) {
            const int q = 8 * n + 2 * tig + jq;
            const float m1 = rm[2 + tg][q];
            const float Mx = fmaxf(mq[n][jq], m1);
            const float Ms = (Mx == kNegInf) ? 0.f : Mx;
            f0[n][jq] = exp2f(mq[n][jq] - Ms);
            f1[n][jq] = exp2f(m1 - Ms);
            lfull[n][jq] = lfull[n][jq] * f0[n][jq] + rl[2 + tg][q] * f1[n][jq];
            mq[n][jq] = Mx;
          }
#pragma unroll
        for (int mt = 0; mt < kMt; ++mt)
#pragma unroll
          for (int n = 0; n < NQT; ++n) {
            const float4 x = *reinterpret_cast<const float4*>(xa + (mt * 32 + lane) * S::XV + 4 * n);
            oacc[mt][n][0] = oacc[mt][n][0] * f0[n][0] + x.x * f1[n][0];
            oacc[mt][n][1] = oacc[mt][n][1] * f0[n][1] + x.y * f1[n][1];
            oacc[mt][n][2] = oacc[mt][n][2] * f0[n][0] + x.z * f1[n][0];
            oacc[mt][n][3] = oacc[mt][n][3] * f0[n][1] + x.w * f1[n][1];
          }
      }
    }
    if (par == 0 && dp == 0 && gid == 0) {
#pragma unroll
      for (int n = 0; n < NQT; ++n)
#pragma unroll
        for (int jq = 0; jq < 2; ++jq) {
          const int q = 8 * n + 2 * tig + jq;
          if (q < G) {
            rm[tg][q] = mq[n][jq];
            rl[tg][q] = poison ? kNaN : lfull[n][jq];
          }
        }
    }
    // this dp's slice (kMt * 32 * XV floats); with two pairs, slot 1, which
    // only token half 1 of the first pair touched since the last rendezvous
    float* xb = &s.xbuf[xp][dp][NPAR - 1][0][0][0];
    if (par == 0 && tg == 1) {
#pragma unroll
      for (int mt = 0; mt < kMt; ++mt)
#pragma unroll
        for (int n = 0; n < NQT; ++n)
          *reinterpret_cast<float4*>(xb + (mt * 32 + lane) * S::XV + 4 * n) =
              make_float4(oacc[mt][n][0], oacc[mt][n][1], oacc[mt][n][2], oacc[mt][n][3]);
    }
    if (!cons_sync()) break;
    if (par == 0 && tg == 0) {
      // merge the two token halves for this warp's queries and O^T rows
      float f0[NQT][2], f1[NQT][2], inv[NQT][2];
#pragma unroll
      for (int n = 0; n < NQT; ++n)
#pragma unroll
        for (int jq = 0; jq < 2; ++jq) {
          const int q = 8 * n + 2 * tig + jq;
          f0[n][jq] = f1[n][jq] = inv[n][jq] = 0.f;
          if (q < hd.gq) {
            const float m0 = rm[0][q], m1 = rm[1][q];
            const float Mx = fmaxf(m0, m1);
            const float Ms = (Mx == kNegInf) ? 0.f : Mx;
            f0[n][jq] = exp2f(m0 - Ms);
            f1[n][jq] = exp2f(m1 - Ms);
            const float L = rl[0][q] * f0[n][jq] + rl[1][q] * f1[n][jq];
            // With several new tokens a CTA's share of an item can hold no key
            // of a row (l = 0): its partial is zero and weighs nothing.  A
            // poisoned row (l NaN) stays NaN.
            inv[n][jq] = (L == 0.f) ? 0.f : vsc / L;
            if (split && dp == 0 && gid == 0)
              *reinterpret_cast<float4*>(a.part + static_cast<size_t>(hd.slot) * prec + q * 4) =
                  make_float4(Mx, L, 0.f, 0.f);  // m = -inf for a row with no key here
          }
        }
      float o[kMt][NQT][4];
#pragma unroll
      for (int mt = 0; mt < kMt; ++mt)
#pragma unroll
        for (int n = 0; n < NQT; ++n) {
          const float4 x = *reinterpret_cast<const float4*>(xb + (mt * 32 + lane) * S::XV + 4 * n);
          o[mt][n][0] = (oacc[mt][n][0] * f0[n][0] + x.x * f1[n][0]) * inv[n][0];
          o[mt][n][1] = (oacc[mt][n][1] * f0[n][1] + x.y * f1[n][1]) * inv[n][1];
          o[mt][n][2] = (oacc[mt][n][2] * f0[n][0] + x.z * f1[n][0]) * inv[n][0];
          o[mt][n][3] = (oacc[mt][n][3] * f0[n][1] + x.w * f1[n][1]) * inv[n][1];
        }
      // Stage the rows [query][this warp's head_dim columns] in the slice the
      // partner warp just handed over, then store them 16 bytes per lane.
      __syncwarp();
#pragma unroll
      for (int mt = 0; mt < kMt; ++mt)
#pragma unroll
        for (int n = 0; n < NQT; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int q = 8 * n + 2 * tig + (e & 1);
            // bf16: m-tile rows are 16 consecutive head_dim columns; fp8: rows
            // gid and gid + 8 are neighbouring columns (see S6)
            const int dl = kFp8 ? mt * 16 + 2 * gid + (e >> 1) : mt * 16 + gid + ((e >> 1) << 3);
            xb[q * kDPart + dl] = o[mt][n][e];
          }
      __syncwarp();
      constexpr int kChunk = 16 / static_cast<int>(sizeof(T));  // elements per 16-byte store
      for (int idx = lane; idx < hd.gq * (kDPart / 4); idx += 32) {
        const int q = idx / (kDPart / 4), c4 = idx - q * (kDPart / 4);
        const float4 v4 = *reinterpret_cast<const float4*>(xb + q * kDPart + 4 * c4);
        const int d = dp * kDPart + 4 * c4;
        if (split) {
          *reinterpret_cast<float4*>(a.part + static_cast<size_t>(hd.slot) * prec + G * 4 + q * D + d) = v4;
        } else if constexpr (kChunk == 8) {
          // bf16: two neighbouring float4 chunks make one 16-byte store
          if ((c4 & 1) == 0) {
            const float4 w4 = *reinterpret_cast<const float4*>(xb + q * kDPart + 4 * c4 + 4);
            T* row = static_cast<T*>(a.out) + q_row(a, hd.b, h, r0 + q) * D + d;
            *reinterpret_cast<uint4*>(row) = make_uint4(pack_bf16(v4.x, v4.y), pack_bf16(v4.z, v4.w),
                                                        pack_bf16(w4.x, w4.y), pack_bf16(w4.z, w4.w));
          }
        }
      }
    }
  }
  if (!split) continue;

  // ---- S8 bookkeeping: the last CTA to finish this item owes its combine --
  // The rendezvous orders every consumer's partial stores before thread 0's
  // release-acquire increment (one GPU-scope round trip instead of a fence
  // in every thread plus an atomic plus another fence).  The proxy fence
  // lets the combining CTA's bulk copies observe those stores.
  fence_proxy_async_global();
  if (!cons_sync()) break;
  if (ct == 0) {
    const int item = hd.b * nvh + hd.vh;
    const int prev = atom_add_acq_rel_gpu(a.counters + item, 1);
    if (prev == hd.nsplit - 1) {
      st_relaxed_gpu(a.counters + item, 0);  // every other CTA has arrived: reset for the next call
      // Only a CTA's first and last segments can be split, so at most two.
      if (s.pend_n < 2) s.pend[s.pend_n++] = PendingCombine{hd.b, hd.vh, hd.nsplit, hd.gq, hd.c_first, hd.item_u};
    }
  }
  }  // segment loop

  // ===================== S8: deferred LSE combines ============================
  // Run after this CTA consumed all its tiles, so the stage ring is free.  An
  // item's partials are one run of records (see DecodeArgs::part): one or two
  // bulk copies stage a round of them.  Each thread then merges its 4-column
  // chunks, weighting every partial by l * 2^(m - M).
  if (!alive) return;
  if (!cons_sync()) return;  // pend_n was written by thread 0
  const int n_pend = s.pend_n;
  float* const ring = reinterpret_cast<float*>(&s.k[0][0]);
  constexpr size_t kRingBytes = 2ull * NSTAGE * kPageTokens * D * sizeof(KV) + EXT;  // k, v and ext
  constexpr int kRowChunks = D / 4;  // float4 chunks of a row
  constexpr int kOwn = (G * kRowChunks + NC - 1) / NC;
  static_assert(kRingBytes >= static_cast<size_t>(G) * (4 + D) * 4, "the ring must hold a partial record");
  uint32_t comb_phase = 0;
  for (int pi = 0; pi < n_pend; ++pi) {
    const PendingCombine pc = s.pend[pi];
    const int h = pc.vh / a.subgroups, sub = pc.vh - h * a.subgroups;
    const int r0 = sub * G;  // first query row of this subgroup
    const int gq = pc.gq;
    const int c_first = pc.c_first;
    // The k-th CTA sharing the item left its partial in first-segment slot
    // c_first + k, except the first CTA when the item starts inside its slice
    // (last-segment slot grid + c_first).
    const bool first_last = part.start(c_first) < pc.item_u;
    const int rec = prec;
    const uint32_t rec_bytes = static_cast<uint32_t>(rec) * 4;
    const int per_round = static_cast<int>(kRingBytes / rec_bytes);
    float Mrun[kOwn], Lrun[kOwn], acc[kOwn][4];
#pragma unroll
    for (int q = 0; q < kOwn; ++q) {
      Mrun[q] = kNegInf;
      Lrun[q] = 0.f;
      acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
    }
    for (int k0 = 0; k0 < pc.nsplit; k0 += per_round) {
      const int nk = min(per_round, pc.nsplit - k0);
      if (k0 > 0 || pi > 0) {
        if (!cons_sync()) return;  // everyone is done reading the ring
      }
      if (warp == 0) {
        // records k0 .. k0 + nk - 1 are one run of first-segment slots, but
        // for record 0 when it sits in the last-segment half: two copies at most
        const bool split0 = k0 == 0 && first_last;
        if (lane == 0) mbar_arrive_expect_tx(&s.comb, static_cast<uint32_t>(nk) * rec_bytes);
        __syncwarp();
        if (lane < 2) {
          fence_proxy_async_global();
          const size_t g = gridDim.x;
          if (lane == 0 && split0) bulk_load(ring, a.part + (g + c_first) * rec, rec_bytes, &s.comb);
          const int k_run = split0 ? 1 : 0;  // first record of the run in this round
          if (lane == (split0 ? 1 : 0) && nk > k_run)
            bulk_load(ring + static_cast<size_t>(k_run) * rec,
                      a.part + static_cast<size_t>(c_first + k0 + k_run) * rec,
                      static_cast<uint32_t>(nk - k_run) * rec_bytes, &s.comb);
        }
      }
      bool ok = wait_phase(&s.comb, comb_phase, &s.abort_flag, a.status, kStatusCombine, a.wait_limit);
      comb_phase ^= 1u;
      if (!__all_sync(0xffffffffu, ok)) return;
#pragma unroll
      for (int q = 0; q < kOwn; ++q) {
        const int oc = ct + q * NC;
        const int i = oc / kRowChunks, cc = oc - i * kRowChunks;
        if (i >= gq) continue;
        const float* mlp = ring + i * 4;                  // (m, l) of row i, record stride rec
        const float* src = ring + G * 4 + i * D + 4 * cc;  // this thread's chunk, record stride rec
        // One pass in batches of kB partials, all loads of a batch in flight:
        // the batch's largest m rescales what is accumulated so far.
        constexpr int kB = 8;
        float M = Mrun[q], l = Lrun[q], a0 = acc[q][0], a1 = acc[q][1], a2 = acc[q][2], a3 = acc[q][3];
        for (int k = 0; k < nk; k += kB) {
          float2 ml[kB];
          float4 ov[kB];
#pragma unroll
          for (int u = 0; u < kB; ++u) {
            if (k + u < nk) {
              ml[u] = *reinterpret_cast<const float2*>(mlp + static_cast<size_t>(k + u) * rec);
              ov[u] = *reinterpret_cast<const float4*>(src + static_cast<size_t>(k + u) * rec);
            } else {
              ml[u] = make_float2(kNegInf, 0.f);
              ov[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
          float Mb = M;
#pragma unroll
          for (int u = 0; u < kB; ++u) Mb = fmaxf(Mb, ml[u].x);
          // Mu: the batch maximum, or 0 while every partial so far is empty
          // (m = -inf, l = 0: a multi-token row with no key in that share)
          const float Mu = (Mb == kNegInf) ? 0.f : Mb;
          const float sc = exp2f(M - Mu);  // 0 before the first partial (M = -inf)
          M = Mb;
          l *= sc;
          a0 *= sc;
          a1 *= sc;
          a2 *= sc;
          a3 *= sc;
#pragma unroll
          for (int u = 0; u < kB; ++u) {
            const float w = ml[u].y * exp2f(ml[u].x - Mu);  // 0 for the padding and the empty entries
            l += w;
            a0 = fmaf(w, ov[u].x, a0);
            a1 = fmaf(w, ov[u].y, a1);
            a2 = fmaf(w, ov[u].z, a2);
            a3 = fmaf(w, ov[u].w, a3);
          }
        }
        Mrun[q] = M;
        Lrun[q] = l;
        acc[q][0] = a0;
        acc[q][1] = a1;
        acc[q][2] = a2;
        acc[q][3] = a3;
      }
    }
#pragma unroll
    for (int q = 0; q < kOwn; ++q) {
      const int oc = ct + q * NC;
      const int i = oc / kRowChunks, cc = oc - i * kRowChunks;
      if (i >= gq) continue;
      const float inv = 1.f / Lrun[q];
      T* row = static_cast<T*>(a.out) + q_row(a, pc.b, h, r0 + i) * D + 4 * cc;
      if constexpr (sizeof(T) == 2) {
        *reinterpret_cast<uint2*>(row) = make_uint2(pack_bf16(acc[q][0] * inv, acc[q][1] * inv),
                                                    pack_bf16(acc[q][2] * inv, acc[q][3] * inv));
      } else {
        *reinterpret_cast<float4*>(row) =
            make_float4(acc[q][0] * inv, acc[q][1] * inv, acc[q][2] * inv, acc[q][3] * inv);
      }
    }
  }
}

}  // namespace vt
