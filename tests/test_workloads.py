"""The seeded input generator: determinism and the layout promises the
parity tests rely on (CPU only)."""
import math

import numpy as np
import pytest
import torch

from paged_attention_decode_kv_gb300 import workloads as W


def test_registry_has_every_workload():
    names = set(W.WORKLOADS)
    for w in (W.TINY, W.QWEN3_1P7B, W.D256_GQA4, W.D256_GQA4_W1024, W.D256_GQA4_F32,
              W.D256_GQA4_F32_W1024, W.LARGE_GQA, W.SKEWED, W.BATCH1_LONG):
        assert w.name in names


@pytest.mark.parametrize("w", [W.TINY, W.QWEN3_1P7B, W.D256_GQA4, W.D256_GQA4_F32])
def test_same_seed_same_case(w):
    a, b = W.make_case(w, 5), W.make_case(w, 5)
    for x, y in ((a.q, b.q), (a.k_pages, b.k_pages), (a.v_pages, b.v_pages)):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32),
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32))
    assert torch.equal(a.block_tables, b.block_tables) and torch.equal(a.context_lens, b.context_lens)
    c = W.make_case(w, 6)
    assert not torch.equal(a.q.float(), c.q.float())


def test_tiny_table_is_a_permutation_of_four_pages():
    c = W.make_case(W.TINY, 0)
    assert sorted(c.block_tables[0].tolist()) == [0, 1, 2, 3]
    assert c.context_lens.tolist() == [33]


def test_qwen_forced_contexts_and_peaked_head():
    c = W.make_case(W.QWEN3_1P7B, 0)
    L = sorted(c.context_lens.tolist())
    for forced in (1, 31, 32, 33, 100, 685, 1000):
        assert forced in L
    assert all(1 <= x <= 1152 for x in L)
    assert 0 <= c.peaked_kv_head < 8
    # the peaked head's keys are 4x bf16 values: the spread is visibly larger
    kf = c.k_pages.float()
    kf = torch.nan_to_num(kf)
    s_peak = kf[:, :, c.peaked_kv_head].abs().mean()
    s_other = kf[:, :, (c.peaked_kv_head + 1) % 8].abs().mean()
    assert s_peak > 3 * s_other


def test_fp32_variant_rounds_to_bf16_variant():
    a, b = W.make_case(W.D256_GQA4, 3), W.make_case(W.D256_GQA4_F32, 3)
    assert torch.equal(a.context_lens, b.context_lens)
    assert torch.equal(b.q.to(torch.bfloat16).view(torch.int16), a.q.view(torch.int16))


def test_pages_disjoint_tails_poisoned_unused_slots_unreferenced():
    c = W.make_case(W.QWEN3_1P7B, 1)
    P = c.workload.block_size
    used = set(c.used_pages.tolist())
    assert len(used) == c.used_pages.numel()
    seen = set()
    pos = 0
    for b, L in enumerate(c.context_lens.tolist()):
        n = math.ceil(L / P)
        row = c.block_tables[b].tolist()
        assert set(row[:n]) <= used and not (set(row[:n]) & seen)
        seen |= set(row[:n])
        assert not (set(row[n:]) & used)  # unused slots point at pages no sequence owns
        if L % P:
            tail = c.k_pages[pos + n - 1, L % P:].float()
            assert torch.isnan(tail).all()
        assert not torch.isnan(c.k_pages[pos:pos + n].float().reshape(-1, *c.k_pages.shape[2:])[:L]).any()
        pos += n


def test_compact_view_has_same_tokens():
    c = W.make_case(W.QWEN3_1P7B, 2)
    k_full, v_full = c.pool("cpu")
    k_c, v_c, bt_c = c.compact()
    P = c.workload.block_size
    for b, L in enumerate(c.context_lens.tolist()):
        for t in (0, L // 2, L - 1):
            full = k_full[c.block_tables[b, t // P], t % P]
            comp = k_c[bt_c[b, t // P], t % P]
            assert torch.equal(full.view(torch.int16), comp.view(torch.int16))


def test_loguniform_and_skewed_ranges():
    c = W.make_case(W.LARGE_GQA.with_(num_seqs=256, pool_blocks=200000), 0)
    L = c.context_lens.numpy()
    assert L.min() >= 256 and L.max() <= 8192
    # log-uniform: about half the mass below the geometric midpoint 1448
    assert 0.35 < np.mean(L < 1448) < 0.65
    s = W._draw_contexts(W.SKEWED, torch.Generator().manual_seed(0))
    assert (s == 32768).sum() == 8 and ((s >= 64) & (s <= 2048)).sum() == 120


def test_kv_bytes_counts_window():
    c = W.make_case(W.D256_GQA4_W1024, 0)
    L = torch.clamp(c.context_lens.long(), max=1024)
    assert c.kv_bytes() == int(L.sum()) * 2 * 256 * 2 * 2
