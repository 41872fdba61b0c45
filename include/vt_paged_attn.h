/*
 * vt_paged_attn -- single-token decode attention over a paged KV cache,
 * hand-written for NVIDIA GB300 (sm_103a).
 *
 * The operation (issue "ROCm gfx1200: PagedAttnOnline is 8.1x slower per call
 * than vLLM's paged-attention kernel", section "Where to look"; PR
 * "perf(cuda): head_dim-128 arm for the warp-split-KV decode kernel", commit
 * message): every sequence b has one query row per query head; query head i
 * attends, with a numerically stable softmax, over the keys and values of kv
 * head h = i / (num_q_heads / num_kv_heads) for the tokens of its context,
 * which live in 32-token pages named by the sequence's block-table row:
 *
 *   L = context_lens[b]; t0 = window > 0 ? max(0, L - window) : 0
 *   s_t = scale * <q[b][i], k_cache[bt[b][t/32]][t%32][h]>      t0 <= t < L
 *   out[b][i] = sum_t softmax(s)_t * v_cache[bt[b][t/32]][t%32][h]
 *
 * Storage is bf16 (or fp32); all arithmetic accumulates in fp32.  A context
 * of 0 tokens produces a zero row.
 *
 * Threading / ordering: every call only enqueues work on `stream` and
 * returns; it never synchronises the device.  The library keeps one
 * split-KV workspace per device (its own, or one the caller hands it with
 * vt_paged_attn_set_workspace); calls that share a device must be ordered on
 * the GPU (same stream, or streams ordered by events), otherwise they race on
 * that workspace.
 */
#ifndef VT_PAGED_ATTN_H
#define VT_PAGED_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define VT_API __attribute__((visibility("default")))
#else
#define VT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as CUDA's cudaStream_t / CUstream (NULL = legacy default stream). */
typedef struct CUstream_st* vt_stream_t;

typedef enum {
  VT_OK = 0,
  VT_ERR_INVALID_ARG = 1,   /* an argument is out of range, NULL or misaligned */
  VT_ERR_UNSUPPORTED = 2,   /* well-formed but not implemented (head_dim, block_size, group) */
  VT_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed; see vt_last_cuda_error() */
  VT_ERR_OOM = 4,           /* the split workspace could not be allocated */
  VT_ERR_DEVICE_TIMEOUT = 5, /* a kernel gave up a bounded wait (see vt_paged_attn_device_status) */
  VT_ERR_SCRATCH_LIMIT = 6   /* the call needs more scratch than a fixed buffer holds (the static array
                                of vt_paged_attn_decode_noalloc, or the caller's vt_paged_attn_set_workspace) */
} vt_status;

/* Storage types.  VT_E4M3 is an FP8 K/V cache (with bf16 q and out) and is
 * taken only by vt_paged_attn_decode_fp8 and vt_paged_attn_decode_multi_fp8. */
typedef enum { VT_BF16 = 0, VT_F32 = 1, VT_E4M3 = 2 } vt_dtype;

/*
 * vt_paged_attn_decode -- the decode step.
 *
 * Device pointers (all caller-owned; nothing is retained after the call):
 *   out          [num_seqs][num_q_heads][head_dim] dtype, written.  16-byte aligned.
 *   q            [num_seqs][num_q_heads][head_dim] dtype.  16-byte aligned.
 *   k_cache      [num_blocks][block_size][num_kv_heads][head_dim] dtype ("NHD"
 *                pages, head_dim contiguous).  16-byte aligned.
 *   v_cache      same layout as k_cache.  16-byte aligned.
 *   block_tables [num_seqs][max_blocks_per_seq] int32 physical page ids; only
 *                the first ceil(L_b / block_size) entries of row b are read,
 *                and of those only pages that overlap the window.
 *   context_lens [num_seqs] int32, 0 <= L_b <= max_blocks_per_seq * block_size.
 * Sizes:
 *   num_seqs >= 0 (0 is a no-op), num_q_heads % num_kv_heads == 0,
 *   head_dim in {64, 128, 256} (and 512 for bf16 storage; the pages' widest
 *   arm), block_size == 32, scale finite (1/sqrt(head_dim)
 *   is usual), window <= 0 for full context else the number of most recent
 *   tokens attended (query token included).
 * Forced additions to the classic signature:
 *   max_blocks_per_seq  block-table row stride (entries) and per-row bound;
 *   num_blocks          pool size in pages: extent of the cache tensors, and
 *                       the bound every page id read is checked against;
 *   dtype               storage type of q, k_cache, v_cache and out.
 *
 * Invalid data found on the device never faults: a context length outside
 * [0, max_blocks_per_seq*block_size] or a page id outside [0, num_blocks)
 * turns that sequence's (or that kv head's) output rows into NaN.
 *
 * Returns VT_OK once the work is enqueued; argument errors return before any
 * launch; VT_ERR_CUDA reports a launch or runtime failure.
 */
VT_API vt_status vt_paged_attn_decode(void* out, const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               const int32_t* context_lens, int num_seqs,
                               int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, float scale, int window,
                               vt_stream_t stream, int max_blocks_per_seq,
                               int num_blocks, vt_dtype dtype);

/*
 * vt_paged_attn_decode_noalloc -- the same decode, for callers that cannot
 * allocate device memory.  The pages this library follows have no
 * counterpart to it; it exists for the caller's sake.
 *
 * vt_paged_attn_decode allocates its split scratch (partial results and
 * arrival counters) itself, on first use and whenever a call needs more,
 * with cudaMallocAsync.  Some callers cannot let a library do that: serving
 * engines that hand nearly all device memory to their KV-cache pool up front,
 * programs whose device memory belongs to one external allocator or arena
 * that no library may bypass, and latency-critical decode loops where a
 * library may not enter the CUDA allocator after start-up.  This entry point
 * never allocates: it takes its scratch from one file-scope device array of
 * VT_NOALLOC_SCRATCH_BYTES (8 MiB), which every GPU that loads the library
 * holds until the process exits.  The caller still passes q, the caches, the
 * tables and out, exactly as for vt_paged_attn_decode; arguments, layouts,
 * results and error codes are the same.
 *
 * - The first call on each device looks up the array's device address with
 *   that device current (a one-time set-up); make that first call before
 *   any stream capture.
 * - A call whose scratch would exceed the array (very large batches, or a
 *   very large forced grid) returns VT_ERR_SCRATCH_LIMIT before launching
 *   anything; vt_last_cuda_error() names the sizes.
 * - All calls share the one array and it keeps the previous call's contents;
 *   each call clears the parts that must start at zero (status word and
 *   arrival counters) on its stream first.  Calls that overlap on the GPU
 *   (concurrent streams, or several host threads) race on the array and
 *   produce wrong results: order them.
 * - The status words of bounded waits live in the array; the next call
 *   clears them.  vt_paged_attn_device_status and
 *   vt_paged_attn_device_status_detail read them (with the other scratch
 *   areas of the device), so a give-up on this path is reported like any
 *   other.
 * - Nothing here calls cudaMalloc, cudaFree or any allocating routine.
 */
#define VT_NOALLOC_SCRATCH_BYTES (8u << 20)
VT_API vt_status vt_paged_attn_decode_noalloc(void* out, const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_tables,
                                              const int32_t* context_lens, int num_seqs,
                                              int num_q_heads, int num_kv_heads, int head_dim,
                                              int block_size, float scale, int window,
                                              vt_stream_t stream, int max_blocks_per_seq,
                                              int num_blocks, vt_dtype dtype);

/*
 * vt_paged_attn_decode_fp8 -- the decode step over an FP8 (E4M3) KV cache
 * with one dequantisation scale per kv head, for keys and for values.
 *
 * A storage extension beyond the pages, whose kernels keep the cache in
 * bf16: the path reads K/V bytes from HBM, so one-byte codes halve the bytes
 * of every step.  The operation is the decode of vt_paged_attn_decode with
 *   k_cache[page][slot][h][d] standing for  e4m3(code) * k_scale[h]
 *   v_cache[page][slot][h][d] standing for  e4m3(code) * v_scale[h]
 * where e4m3() is the OCP 8-bit floating-point value of the code (4 exponent
 * bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN).
 *
 * Arguments as for vt_paged_attn_decode, except:
 *   q, out            bf16 [num_seqs][num_q_heads][head_dim].
 *   k_cache, v_cache  uint8 E4M3 codes, [num_blocks][block_size][num_kv_heads]
 *                     [head_dim] (NHD), 16-byte aligned.
 *   k_scale, v_scale  device float32 [num_kv_heads], 4-byte aligned; NULL is
 *                     VT_ERR_INVALID_ARG.
 *   head_dim          64, 128 or 256 (512 is VT_ERR_UNSUPPORTED).
 * Arithmetic: the K and V codes are widened exactly to f16 and enter f16
 * tensor-core MMAs with fp32 accumulation.  Each query row is scaled by a
 * power of two that puts its largest magnitude in [2^14, 2^15) and rounded
 * to f16, which holds the bf16 values exactly down to 2^-28 of that largest
 * (rows below 2^-100 in magnitude count as zero); the softmax weights enter
 * PV as f16 (11 significant bits).  k_scale folds into the score scale and
 * v_scale into the final normalisation.
 * Workspace, plan, status and errors are those of vt_paged_attn_decode.
 */
VT_API vt_status vt_paged_attn_decode_fp8(void* out, const void* q, const void* k_cache,
                                          const void* v_cache, const float* k_scale,
                                          const float* v_scale, const int32_t* block_tables,
                                          const int32_t* context_lens, int num_seqs,
                                          int num_q_heads, int num_kv_heads, int head_dim,
                                          int block_size, float scale, int window,
                                          vt_stream_t stream, int max_blocks_per_seq,
                                          int num_blocks);

/*
 * vt_paged_attn_decode_multi -- several new tokens per sequence over the same
 * paged cache: a chunk of a prefill, or draft tokens to verify.
 *
 * The pages list a head_dim-128 prefill as owed (PR "perf(rocm): head_dim=128
 * decode arm", section "Not claimed"); the reading taken: every sequence b
 * carries q_len new tokens whose keys and values are already in its pages as
 * the last q_len of its L = context_lens[b] tokens.  New token j
 * (0 <= j < q_len), at position L - q_len + j, attends with the decode's
 * arithmetic to the tokens t with
 *   t0_j <= t <= L - q_len + j,   t0_j = window > 0 ? max(0, L - q_len + 1 + j - window) : 0
 * (causal within the chunk), i.e. it is the single-token decode over a
 * context of L - q_len + 1 + j tokens.
 *
 * Arguments as for vt_paged_attn_decode, except:
 *   q, out   [num_seqs][q_len][num_q_heads][head_dim] (bf16 or fp32).
 *   q_len    >= 1 (1 is vt_paged_attn_decode); q_len * group <= 4096.
 * The query rows of one kv head (q_len tokens x its group of query heads)
 * share every page the head's kv tile is read for, so the cache is read once
 * per kv head for the whole chunk.  A sequence with L < q_len gets NaN rows
 * for all its new tokens.  dtype VT_E4M3 is VT_ERR_INVALID_ARG (an FP8 cache
 * takes vt_paged_attn_decode_multi_fp8).
 */
VT_API vt_status vt_paged_attn_decode_multi(void* out, const void* q, const void* k_cache,
                                            const void* v_cache, const int32_t* block_tables,
                                            const int32_t* context_lens, int num_seqs, int q_len,
                                            int num_q_heads, int num_kv_heads, int head_dim,
                                            int block_size, float scale, int window,
                                            vt_stream_t stream, int max_blocks_per_seq,
                                            int num_blocks, vt_dtype dtype);

/*
 * vt_paged_attn_decode_multi_fp8 -- several new tokens per sequence over an
 * FP8 (E4M3) cache: the operation of vt_paged_attn_decode_multi on the cache
 * that vt_paged_attn_decode_fp8 reads (codes times per-kv-head scales).
 *
 * Arguments as for vt_paged_attn_decode_fp8, plus q_len after num_seqs:
 *   q, out   bf16 [num_seqs][q_len][num_q_heads][head_dim].
 *   q_len    >= 1 (1 is vt_paged_attn_decode_fp8); q_len * group <= 4096.
 * Arithmetic as for vt_paged_attn_decode_fp8; causal limits, windows and the
 * NaN rows of L < q_len as for vt_paged_attn_decode_multi.  NULL scales are
 * VT_ERR_INVALID_ARG.
 */
VT_API vt_status vt_paged_attn_decode_multi_fp8(void* out, const void* q, const void* k_cache,
                                                const void* v_cache, const float* k_scale,
                                                const float* v_scale, const int32_t* block_tables,
                                                const int32_t* context_lens, int num_seqs, int q_len,
                                                int num_q_heads, int num_kv_heads, int head_dim,
                                                int block_size, float scale, int window,
                                                vt_stream_t stream, int max_blocks_per_seq,
                                                int num_blocks);

/* What the last successful decode call on this host thread launched. */
typedef struct {
  int grid_ctas;          /* CTAs launched (persistent, balanced split of the work) */
  int ctas_per_sm;        /* resident CTAs per SM for this kernel variant */
  int num_sms;            /* SMs of the device */
  int consumer_warps;     /* compute warps per CTA (plus one TMA producer warp) */
  int tensor_cores;       /* 1: QK^T and PV on tensor cores (bf16, fp8), 0: CUDA cores (fp32) */
  int stages;             /* K/V page tiles in flight per CTA */
  int group_tile;         /* query heads computed per kv head and CTA (padded) */
  int subgroups;          /* ceil(group / group_tile) */
  int min_units_per_cta;  /* lower bound on work units per CTA (page tiles plus item weights) */
  int head_dim;
  int dtype;              /* vt_dtype of the K/V cache */
  size_t smem_bytes;      /* dynamic shared memory per CTA */
  size_t workspace_bytes; /* split-KV workspace used (partials + arrival counters) */
  int launch_overlap;     /* 1: launched as a programmatic dependent (vt_paged_attn_set_overlap) */
  int segment_cost;       /* partition weight of a segment boundary, in tiles (vt_paged_attn_set_segment_cost) */
  int scratch_source;     /* split scratch used: 0 library-owned, 1 the caller's (vt_paged_attn_set_workspace),
                             2 the static array (vt_paged_attn_decode_noalloc) */
  int q_len;              /* new tokens per sequence (1 except for vt_paged_attn_decode_multi) */
} vt_plan;

VT_API vt_status vt_paged_attn_last_plan(vt_plan* plan);

/*
 * Test / benchmark override of the launch plan for this host thread, read on
 * every call.  grid_ctas > 0 forces the number of CTAs (so tests can force
 * every sequence to be split, or never split); min_units_per_cta > 0 replaces
 * the default lower bound on work per CTA.  0 restores the automatic choice.
 */
VT_API vt_status vt_paged_attn_set_override(int grid_ctas, int min_units_per_cta);

/*
 * Launch overlap for this host thread, read on every call (default 0).  Not
 * an operation of the pages: a launch choice of this library.
 *
 * enabled = 1 launches each decode as a programmatic dependent of the kernel
 * before it on the same stream (CUDA programmatic dependent launch; it also
 * applies inside stream capture).  The decode's CTAs may then start while
 * that kernel finishes: they read context_lens and block_tables and plan the
 * split at once, and wait for it to complete before they read q, k_cache or
 * v_cache, or touch out and the workspace.  The decode itself lets the next
 * kernel start the same way.  Back-to-back decode steps (CUDA graphs of
 * layers or steps) overlap one call's start-up with the previous call's
 * tail.
 *
 * Contract: with enabled = 1, the kernel launched immediately before the
 * decode on its stream must not write context_lens or block_tables (step
 * metadata usually comes from host copies, which do not overlap).  Results
 * are identical either way.  Returns VT_ERR_INVALID_ARG unless enabled is 0
 * or 1.
 */
VT_API vt_status vt_paged_attn_set_overlap(int enabled);

/*
 * Partition weight of a segment boundary for this host thread, read on every
 * call.  Not an operation of the pages: a scheduling choice of this library.
 *
 * The kernel splits the (sequence, kv head, page) tiles evenly over its CTAs.
 * Every (sequence, kv head) a CTA starts costs it time beyond its pages (an
 * epilogue, a new query tile, a block-table row), so each one also weighs
 * `tiles` tiles in the split: CTAs whose share crosses many short sequences
 * get fewer pages.  The weight applies when the batch gives every CTA at
 * least 4 pages (below that the split is latency-bound and weights only add
 * partial results).  tiles < 0 restores the default: 2 for bf16 and fp32
 * K/V, 6 for an FP8 cache or several new tokens per sequence (their tiles
 * take less time per segment boundary); 0 balances pages alone.  Results are the same within rounding (split points move, and with
 * them the order of the log-sum-exp merge).  Returns VT_ERR_INVALID_ARG for
 * tiles > 64.
 */
VT_API vt_status vt_paged_attn_set_segment_cost(int tiles);

/*
 * Reads and clears the device status word that kernels set when a bounded
 * wait gives up (bit 0: page tile never arrived, bit 1: stage never released,
 * bit 2: consumer-warp rendezvous, bit 3: drain of copies in flight, bit 5:
 * partials staged for a split-KV combine) or a
 * self-check fails (bit 4: a CTA's tile walk did not match its share).
 * Synchronises `stream` first.  *status is 0 when all is well; the call
 * returns VT_ERR_DEVICE_TIMEOUT if it was not.  Clearing also resets the
 * split workspace's arrival counters.
 */
VT_API vt_status vt_paged_attn_device_status(vt_stream_t stream, unsigned* status);

/*
 * Copies the first n_words (<= 8) words of the device status area without
 * clearing them: [0] status bits as above; [1] 1 + index of the CTA whose
 * wait gave up first (0: none); [2] its status bit | (thread index << 8);
 * [3] shared-memory address of the barrier it waited on; [4] the phase
 * parity it waited for.  Synchronises `stream` first.
 */
VT_API vt_status vt_paged_attn_device_status_detail(vt_stream_t stream, unsigned* words, int n_words);

/*
 * vt_paged_attn_set_workspace -- hand the library a caller-owned split-KV
 * workspace for the current device (the boundary's optional workspace; the
 * operation itself is unchanged).
 *
 * vt_paged_attn_decode needs device scratch for split-KV partial results and
 * arrival counters.  By default the library allocates it lazily with
 * cudaMallocAsync on the call's stream and grows it when a call needs more.
 * After this call, decodes on the current device use [dev_ptr, dev_ptr +
 * bytes) instead and never allocate:
 *   dev_ptr  device memory, 256-byte aligned, owned by the caller; it must
 *            stay allocated and be touched by nothing else while it is set.
 *            NULL returns the device to the library-owned workspace.
 *   bytes    >= VT_MIN_WORKSPACE_BYTES.  The arrival counters must stay
 *            zeroed between calls, so their region only grows: a call needs
 *            256 bytes, plus the largest counter region any call on this
 *            workspace used, plus its own partial records.  For one model
 *            shape (heads, head_dim, dtype) the partials do not depend on the
 *            batch, so vt_paged_attn_workspace_bytes() of the largest
 *            num_seqs in use is enough for every call; for several shapes,
 *            the sum of their largest needs is.
 *   stream   the first 256 bytes (status words) are zeroed on it; later
 *            calls zero newly used counter space on their own streams.
 * A decode that needs more than `bytes` returns VT_ERR_SCRATCH_LIMIT before
 * launching anything.  Calls that share the workspace must be ordered on
 * the GPU.  vt_paged_attn_device_status reads its status words.
 * Returns VT_ERR_INVALID_ARG for a misaligned pointer or a too-small size.
 */
#define VT_MIN_WORKSPACE_BYTES 4096u
VT_API vt_status vt_paged_attn_set_workspace(void* dev_ptr, size_t bytes, vt_stream_t stream);

/*
 * Test hook for the failure path of bounded waits (this host thread, read on
 * every call; not an operation of the pages).  Every wait on an mbarrier in
 * the kernel gives up after a limit of about one second of SM clock cycles,
 * sets a status bit and lets the CTA exit; this hook shortens the limit to
 * wait_limit_cycles (<= 0: the default) and, when withhold_tile >= 0, makes
 * CTA withhold_cta stop feeding its consumers before its withhold_tile-th
 * ring stage (counting from 0; stages that only close a segment count too).
 * The consumers' wait for that stage then runs out, the kernel returns
 * without faulting, and vt_paged_attn_device_status reports
 * VT_ERR_DEVICE_TIMEOUT (bit 0); the output of that call is incomplete.
 * vt_paged_attn_set_test_wait(0, -1, -1) restores normal operation.
 * Returns VT_ERR_INVALID_ARG when withhold_tile >= 0 and withhold_cta < 0.
 */
VT_API vt_status vt_paged_attn_set_test_wait(long long wait_limit_cycles, int withhold_cta, int withhold_tile);

/* Bytes of split-KV workspace a call with these sizes uses on the current device. */
VT_API size_t vt_paged_attn_workspace_bytes(int num_seqs, int num_q_heads,
                                     int num_kv_heads, int head_dim,
                                     vt_dtype dtype);

/* Frees the library's per-device workspaces.  No call may be in flight. */
VT_API void vt_paged_attn_release(void);

VT_API const char* vt_status_string(vt_status status);

/* Text of the last CUDA error seen by this host thread ("" if none). */
VT_API const char* vt_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
VT_API int vt_paged_attn_version(void);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* VT_PAGED_ATTN_H */
