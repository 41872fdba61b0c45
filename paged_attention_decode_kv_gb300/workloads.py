"""Seeded synthetic decode workloads (inputs only; no attention arithmetic).

Both the CUDA path and the CPU oracle take their inputs from here, and this
module holds none of the method's arithmetic: it draws queries, paged K/V
contents, context lengths and block tables, and lays them out.

The shapes follow the decode workloads the pages measure (Qwen3-family decode
with 32-token pages, GQA groups of 2 to 8, head_dim 128 and 256), as five
named configurations plus a batch-1 long-context case, plus batches for the
library's other arms: head_dim 512 and 64, and FP8 (E4M3) K/V storage.  Recipe, per case:

* one ``torch.Generator`` seeded with ``seed`` draws, in this order: the
  context lengths, a random permutation of the page pool, Q, K (all used
  pages), V (all used pages), then any per-case extra (the peaked head);
* Q/K/V are drawn as float32 N(0, sigma); bf16 storage is their
  round-to-nearest-even image, fp32 storage keeps them as drawn; FP8 (E4M3)
  K/V storage divides each kv head's draws by one scale per head (the
  head's largest magnitude over 448, the largest E4M3 value) and keeps the
  nearest E4M3 codes, with bf16 queries;
* sequence b takes the next ceil(L_b / 32) pages of the permutation; its
  block-table slots past those point at pool pages no sequence uses;
* every pool page no sequence uses, and every in-page slot at or past L_b
  in a sequence's last page, holds NaN, so any read the method must not make
  shows up in the output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

BLOCK_SIZE = 32


@dataclass(frozen=True)
class Workload:
    name: str
    description: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    pool_blocks: int
    contexts: str  # "fixed:33", "list:1,31,...", "forced_uniform:1,1152:1,31,...", "uniform:a,b",
    #                 "loguniform:a,b", "skewed"
    max_blocks_per_seq: int
    sigma: float = 1.0
    dtype: str = "bf16"  # K/V storage: "bf16" | "f32" | "e4m3" (bf16 q and out)
    window: int = 0
    peaked_head: bool = False
    table_is_permutation: bool = False
    block_size: int = BLOCK_SIZE
    q_len: int = 1  # new tokens per sequence (> 1: multi-token decode, q is [B][q_len][Hq][D])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def elem_bytes(self) -> int:
        """Bytes of one stored K/V element."""
        return {"bf16": 2, "f32": 4, "e4m3": 1}[self.dtype]

    @property
    def qo_elem_bytes(self) -> int:
        """Bytes of one query or output element."""
        return 4 if self.dtype == "f32" else 2

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS: dict[str, Workload] = {}


def _register(w: Workload) -> Workload:
    WORKLOADS[w.name] = w
    return w


TINY = _register(Workload(
    name="tiny_b1_gqa2_d128_ctx33",
    description="1 seq, 16 q / 8 kv heads, head_dim 128, context 33; block table is a "
                "seeded permutation of a 4-page pool",
    num_seqs=1, num_q_heads=16, num_kv_heads=8, head_dim=128, pool_blocks=4,
    contexts="fixed:33", max_blocks_per_seq=4, table_is_permutation=True))

QWEN3_1P7B = _register(Workload(
    name="qwen3_1p7b_b8_gqa2_d128",
    description="Qwen3-1.7B-shaped decode batch: 8 seqs, 16 q / 8 kv heads, head_dim 128; "
                "contexts U[1,1152] with 1,31,32,33,100,685,1000 forced; K x4 on one seeded "
                "kv head; 512-page pool",
    num_seqs=8, num_q_heads=16, num_kv_heads=8, head_dim=128, pool_blocks=512,
    contexts="forced_uniform:1,1152:1,31,32,33,100,685,1000", max_blocks_per_seq=36,
    peaked_head=True))

D256_GQA4 = _register(Workload(
    name="d256_gqa4_b16",
    description="head_dim 256 GQA-4 decode: 16 seqs, 8 q / 2 kv heads, contexts U[512,4096]; "
                "4096-page pool",
    num_seqs=16, num_q_heads=8, num_kv_heads=2, head_dim=256, pool_blocks=4096,
    contexts="uniform:512,4096", max_blocks_per_seq=128))

D256_GQA4_W1024 = _register(D256_GQA4.with_(
    name="d256_gqa4_b16_w1024", window=1024,
    description=D256_GQA4.description + "; sliding window 1024"))

D256_GQA4_F32 = _register(D256_GQA4.with_(
    name="d256_gqa4_b16_f32", dtype="f32",
    description=D256_GQA4.description + "; fp32 storage"))

D256_GQA4_F32_W1024 = _register(D256_GQA4.with_(
    name="d256_gqa4_b16_f32_w1024", dtype="f32", window=1024,
    description=D256_GQA4.description + "; fp32 storage; sliding window 1024"))

# head_dim 512 arm (the pages' kernels cover head_dim 512): the d256 batch's
# sequences and GQA-4 grouping at the wider head; 4096-page pool.
D512_GQA4 = _register(Workload(
    name="d512_gqa4_b16",
    description="head_dim 512 GQA-4 decode: 16 seqs, 8 q / 2 kv heads, contexts U[512,4096]; "
                "4096-page pool",
    num_seqs=16, num_q_heads=8, num_kv_heads=2, head_dim=512, pool_blocks=4096,
    contexts="uniform:512,4096", max_blocks_per_seq=128))

D512_GQA4_W1024 = _register(D512_GQA4.with_(
    name="d512_gqa4_b16_w1024", window=1024,
    description=D512_GQA4.description + "; sliding window 1024"))

# head_dim 64 arm: not a configuration of the pages (their kernels cover
# head_dim 128, 256 and 512); the d256 batch's lengths at a Qwen-like
# 16 q / 4 kv heads, so every (sequence, kv head) page tile is 4 KB.
D64_GQA4 = _register(Workload(
    name="d64_gqa4_b32",
    description="head_dim 64 GQA-4 decode: 32 seqs, 16 q / 4 kv heads, contexts U[512,4096]; "
                "8192-page pool",
    num_seqs=32, num_q_heads=16, num_kv_heads=4, head_dim=64, pool_blocks=8192,
    contexts="uniform:512,4096", max_blocks_per_seq=128))

D64_GQA4_F32 = _register(D64_GQA4.with_(
    name="d64_gqa4_b32_f32", dtype="f32",
    description=D64_GQA4.description + "; fp32 storage"))

LARGE_GQA = _register(Workload(
    name="large_gqa8_b64_d128",
    description="Large-GQA server batch: 64 seqs, 64 q / 8 kv heads, head_dim 128, contexts "
                "log-uniform [256,8192], N(0,0.5); 20000-page pool",
    num_seqs=64, num_q_heads=64, num_kv_heads=8, head_dim=128, pool_blocks=20000,
    contexts="loguniform:256,8192", max_blocks_per_seq=256, sigma=0.5))

SKEWED = _register(Workload(
    name="skewed_b128_gqa4_d128",
    description="Long-context skewed batch: 128 seqs, 32 q / 8 kv heads, head_dim 128; 120 seqs "
                "U[64,2048] and 8 seqs at 32768; 65536-page pool",
    num_seqs=128, num_q_heads=32, num_kv_heads=8, head_dim=128, pool_blocks=65536,
    contexts="skewed", max_blocks_per_seq=1024))

BATCH1_LONG = _register(Workload(
    name="batch1_ctx32768_gqa4_d128",
    description="batch 1 at context 32768, 32 q / 8 kv heads, head_dim 128; 65536-page pool",
    num_seqs=1, num_q_heads=32, num_kv_heads=8, head_dim=128, pool_blocks=65536,
    contexts="fixed:32768", max_blocks_per_seq=1024))

# FP8 (E4M3) K/V storage with per-kv-head scales: the same batches with one
# byte per cached element (not configurations of the pages, whose caches are
# bf16; the storage extension's own test and sweep cases).
_FP8 = "; FP8 E4M3 K/V codes with per-kv-head scales, bf16 queries"
QWEN3_1P7B_FP8 = _register(QWEN3_1P7B.with_(name="qwen3_1p7b_b8_gqa2_d128_fp8", dtype="e4m3",
                                           description=QWEN3_1P7B.description + _FP8))
D256_GQA4_FP8 = _register(D256_GQA4.with_(name="d256_gqa4_b16_fp8", dtype="e4m3",
                                         description=D256_GQA4.description + _FP8))
D256_GQA4_W1024_FP8 = _register(D256_GQA4.with_(name="d256_gqa4_b16_w1024_fp8", dtype="e4m3", window=1024,
                                               description=D256_GQA4.description + "; sliding window 1024" + _FP8))
LARGE_GQA_FP8 = _register(LARGE_GQA.with_(name="large_gqa8_b64_d128_fp8", dtype="e4m3",
                                         description=LARGE_GQA.description + _FP8))
SKEWED_FP8 = _register(SKEWED.with_(name="skewed_b128_gqa4_d128_fp8", dtype="e4m3",
                                   description=SKEWED.description + _FP8))
# Multi-token decode (several new tokens per sequence: draft tokens to verify,
# or a chunk of a prefill), attending causally within the chunk: the large
# batch's shape at GQA 4 with 4 new tokens, so one kv head's 16 query rows
# fill one tensor-core tile.  Not a configuration of the pages (which list a
# head_dim-128 prefill as owed); the multi-token arm's own case.
MULTI_Q4 = _register(Workload(
    name="multi_q4_b64_gqa4_d128",
    description="multi-token decode: 64 seqs x 4 new tokens, 32 q / 8 kv heads, head_dim 128, contexts "
                "U[512,8192] (the new tokens are the last 4); 20000-page pool",
    num_seqs=64, num_q_heads=32, num_kv_heads=8, head_dim=128, pool_blocks=20000,
    contexts="uniform:512,8192", max_blocks_per_seq=256, q_len=4))

BATCH1_LONG_FP8 = _register(BATCH1_LONG.with_(name="batch1_ctx32768_gqa4_d128_fp8", dtype="e4m3",
                                             description=BATCH1_LONG.description + _FP8))
MULTI_Q4_FP8 = _register(MULTI_Q4.with_(name="multi_q4_b64_gqa4_d128_fp8", dtype="e4m3",
                                       description=MULTI_Q4.description + _FP8))
D64_GQA4_FP8 = _register(D64_GQA4.with_(name="d64_gqa4_b32_fp8", dtype="e4m3",
                                       description=D64_GQA4.description + _FP8))


def custom(name: str, contexts, num_q_heads: int, num_kv_heads: int, head_dim: int,
           dtype: str = "bf16", window: int = 0, sigma: float = 1.0, spare_pages: int = 3,
           q_len: int = 1) -> Workload:
    """A workload with an explicit list of context lengths (edge-case tests)."""
    contexts = [int(x) for x in contexts]
    pages = sum((L + BLOCK_SIZE - 1) // BLOCK_SIZE for L in contexts)
    maxb = max(1, max((L + BLOCK_SIZE - 1) // BLOCK_SIZE for L in contexts))
    return Workload(name=name, description=f"explicit contexts {contexts}", num_seqs=len(contexts),
                    num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                    pool_blocks=pages + spare_pages, contexts="list:" + ",".join(map(str, contexts)),
                    max_blocks_per_seq=maxb, sigma=sigma, dtype=dtype, window=window, q_len=q_len)


def _draw_contexts(w: Workload, g: torch.Generator) -> torch.Tensor:
    kind, _, arg = w.contexts.partition(":")
    B = w.num_seqs
    if kind == "fixed":
        return torch.full((B,), int(arg), dtype=torch.int32)
    if kind == "list":
        L = [int(x) for x in arg.split(",")]
        if len(L) != B:
            raise ValueError("context list length must equal num_seqs")
        return torch.tensor(L, dtype=torch.int32)
    if kind == "uniform":
        lo, hi = (int(x) for x in arg.split(","))
        return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    if kind == "loguniform":
        lo, hi = (int(x) for x in arg.split(","))
        u = torch.rand((B,), generator=g, dtype=torch.float64)
        L = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
        return L.round().clamp(lo, hi).to(torch.int32)
    if kind == "forced_uniform":
        rng, _, forced = arg.partition(":")
        lo, hi = (int(x) for x in rng.split(","))
        forced_l = [int(x) for x in forced.split(",")]
        rest = torch.randint(lo, hi + 1, (B - len(forced_l),), generator=g, dtype=torch.int64)
        L = torch.cat([torch.tensor(forced_l, dtype=torch.int64), rest])
        return L[torch.randperm(B, generator=g)].to(torch.int32)
    if kind == "skewed":
        short = torch.randint(64, 2048 + 1, (B - 8,), generator=g, dtype=torch.int64)
        L = torch.cat([short, torch.full((8,), 32768, dtype=torch.int64)])
        return L[torch.randperm(B, generator=g)].to(torch.int32)
    raise ValueError(f"unknown context recipe {w.contexts!r}")


@dataclass
class PagedCase:
    """One seeded decode problem.  All tensors live on CPU.

    ``k_pages`` / ``v_pages`` hold only the pages sequences use, in the order
    ``used_pages`` lists their physical ids; ``device_pool`` and ``host_pool``
    scatter them into full NaN-filled pools of ``num_blocks`` pages.
    """
    workload: Workload
    seed: int
    q: torch.Tensor             # [B][Hq][D], bf16 or fp32
    k_pages: torch.Tensor       # [n_used][P][Hkv][D]
    v_pages: torch.Tensor       # [n_used][P][Hkv][D]
    used_pages: torch.Tensor    # [n_used] int64 physical page ids
    block_tables: torch.Tensor  # [B][max_blocks_per_seq] int32
    context_lens: torch.Tensor  # [B] int32
    peaked_kv_head: int = -1
    extra: dict = field(default_factory=dict)

    @property
    def num_blocks(self) -> int:
        return self.workload.pool_blocks

    @property
    def dtype(self) -> torch.dtype:
        """Storage type of q and out."""
        return self.q.dtype

    @property
    def kv_dtype(self) -> torch.dtype:
        """Storage type of the K/V pages (uint8 E4M3 codes for FP8)."""
        return self.k_pages.dtype

    @property
    def fp8(self) -> bool:
        return self.workload.dtype == "e4m3"

    def _nan_fill(self, shape, device):
        if self.fp8:
            return torch.full(shape, E4M3_NAN, dtype=torch.uint8, device=device)
        return torch.full(shape, float("nan"), dtype=self.kv_dtype, device=device)

    def pool(self, device="cpu"):
        """Full (k_cache, v_cache) pools [num_blocks][P][Hkv][D] on ``device``."""
        w = self.workload
        shape = (self.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
        idx = self.used_pages.to(device)
        out = []
        for pages in (self.k_pages, self.v_pages):
            cache = self._nan_fill(shape, device)
            cache.index_copy_(0, idx, pages.to(device))
            out.append(cache)
        return tuple(out)

    def scales(self, device="cpu"):
        """FP8 storage: the per-kv-head (k_scale, v_scale), float32 [Hkv]."""
        return self.extra["k_scale"].to(device), self.extra["v_scale"].to(device)

    def compact(self):
        """(k, v, block_tables) with only the used pages, renumbered 0..n_used-1,
        plus one NaN page (id n_used) that every unused table slot points at.
        Same logical KV as ``pool()`` for every token a sequence owns."""
        w = self.workload
        n = self.used_pages.numel()
        remap = torch.full((self.num_blocks,), n, dtype=torch.int64)
        remap[self.used_pages] = torch.arange(n)
        nan_page = self._nan_fill((1, w.block_size, w.num_kv_heads, w.head_dim), "cpu")
        k = torch.cat([self.k_pages, nan_page])
        v = torch.cat([self.v_pages, nan_page])
        bt = remap[self.block_tables.long()].to(torch.int32)
        return k, v, bt

    def kv_bytes(self) -> int:
        """Exact K+V bytes the method must read: tokens inside the window."""
        w = self.workload
        L = self.context_lens.long()
        if w.window > 0:
            L = torch.clamp(L, max=w.window)
        return int(L.sum()) * w.num_kv_heads * w.head_dim * 2 * w.elem_bytes

    def qo_bytes(self) -> int:
        w = self.workload
        return 2 * w.num_seqs * w.q_len * w.num_q_heads * w.head_dim * w.qo_elem_bytes


def make_case(w: Workload, seed: int = 0) -> PagedCase:
    g = torch.Generator().manual_seed(int(seed))
    B, Hq, Hkv, D, P = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
    ctx = _draw_contexts(w, g)
    if int(ctx.max()) > w.max_blocks_per_seq * P:
        raise ValueError("context longer than a block-table row")
    perm = torch.randperm(w.pool_blocks, generator=g)
    pages_per_seq = [(int(L) + P - 1) // P for L in ctx]
    n_used = sum(pages_per_seq)
    if n_used >= w.pool_blocks and not w.table_is_permutation:
        raise ValueError("pool too small for the drawn contexts")
    used = perm[:n_used]
    spare = perm[n_used:]
    bt = torch.empty((B, w.max_blocks_per_seq), dtype=torch.int64)
    pos, spare_pos = 0, 0
    for b, n in enumerate(pages_per_seq):
        bt[b, :n] = used[pos:pos + n]
        pos += n
        for s in range(n, w.max_blocks_per_seq):
            bt[b, s] = spare[spare_pos % spare.numel()]
            spare_pos += 1

    fp8 = w.dtype == "e4m3"
    store = torch.float32 if w.dtype == "f32" else torch.bfloat16
    q = (torch.randn((B, Hq, D), generator=g) * w.sigma).to(store)
    k = torch.randn((n_used, P, Hkv, D), generator=g) * w.sigma
    v = torch.randn((n_used, P, Hkv, D), generator=g) * w.sigma
    if not fp8:
        k, v = k.to(store), v.to(store)
    peaked = -1
    if w.peaked_head:
        peaked = int(torch.randint(0, Hkv, (1,), generator=g))
        k[:, :, peaked, :] *= 4  # power of two: exact in bf16 and fp32
    extra = {}
    if fp8:
        k, ks = _e4m3_per_head(k)
        v, vs = _e4m3_per_head(v)
        extra = {"k_scale": ks, "v_scale": vs}
    if w.q_len > 1:
        # multi-token decode: the queries of the q_len new tokens, drawn last
        # so every other draw matches the single-token case of the same seed
        q = (torch.randn((B, w.q_len, Hq, D), generator=g) * w.sigma).to(store)
    # Poison the in-page tail of every sequence's last page.
    poison = E4M3_NAN if fp8 else float("nan")
    pos = 0
    for b, n in enumerate(pages_per_seq):
        L = int(ctx[b])
        if n and L % P:
            k[pos + n - 1, L % P:] = poison
            v[pos + n - 1, L % P:] = poison
        pos += n
    return PagedCase(workload=w, seed=int(seed), q=q, k_pages=k, v_pages=v, used_pages=used,
                     block_tables=bt.to(torch.int32), context_lens=ctx, peaked_kv_head=peaked, extra=extra)


E4M3_MAX = 448.0
E4M3_NAN = 0x7F  # the positive NaN code of E4M3


def _e4m3_per_head(x: torch.Tensor):
    """float32 [..][Hkv][D] draws -> (uint8 E4M3 codes, float32 scale per kv
    head): each head is divided by its largest magnitude over 448 and rounded
    to the nearest code by torch's float8_e4m3fn conversion."""
    amax = x.abs().amax(dim=tuple(i for i in range(x.dim()) if i != x.dim() - 2))
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).to(torch.float32)
    codes = (x / scale[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a bf16 tensor's bit patterns (what the oracle reads)."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def to_oracle_array(t: torch.Tensor):
    """Storage-exact numpy array for the oracle: bf16 -> uint16 bits, fp32 ->
    float32, E4M3 codes (uint8) -> uint8."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    if t.dtype in (torch.float32, torch.float64, torch.uint8):
        return t.contiguous().numpy()
    raise TypeError(t.dtype)
