"""CUDA path vs the fp64 oracle, element by element, through the C-ABI.

Tolerances (fixed by the decode PR's CPU-oracle gate and the workload spec):
bf16 output (bf16 storage, and the FP8 E4M3 K/V cache against the oracle
on the dequantised cache): NMSE <= 5e-4 over the call's outputs and
max |err| <= 2e-2; fp32 storage: max |err| <= 1e-5.
NMSE = sum (gpu - ref)^2 / sum ref^2.

These tests fail (never skip) when no GPU or no library is present: a GPU
job that cannot run them must not look green.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import paged_attention_decode_kv_gb300 as vt
from paged_attention_decode_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

BF16_NMSE, BF16_MAXABS, F32_MAXABS = 5e-4, 2e-2, 1e-5
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from paged_attention_decode_kv_gb300 import build_lib
    build_lib.build()
    vt.library()
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _reset_override():
    yield
    if vt._lib is not None:
        vt.vt_paged_attn_set_override(0, 0)
        vt.vt_paged_attn_set_overlap(False)
        vt.vt_paged_attn_set_segment_cost(-1)
        vt.vt_paged_attn_set_test_wait(0, -1, -1)
        vt.vt_paged_attn_set_workspace(0, 0)


def run_decode(case, q, k, v, bt, cl, window=None, out=None, stream=None, scale=None):
    """One decode through the entry point for the case's storage type."""
    w = case.workload
    scale = w.scale if scale is None else scale
    window = w.window if window is None else window
    if case.fp8:
        ks, vs = case.scales(q.device)
        return vt.decode_fp8(q, k, v, ks, vs, bt, cl, scale, window, out=out, stream=stream)
    if w.q_len > 1:
        return vt.decode_multi(q, k, v, bt, cl, scale, window, out=out, stream=stream)
    return vt.decode(q, k, v, bt, cl, scale, window, out=out, stream=stream)


def gpu_run(case, dev, grid=0, min_units=0, window=None, tables=None, lens=None, stream=None):
    k, v = case.pool(dev)
    q = case.q.to(dev)
    bt = (case.block_tables if tables is None else tables).to(dev)
    cl = (case.context_lens if lens is None else lens).to(dev)
    vt.vt_paged_attn_set_override(grid, min_units)
    out = run_decode(case, q, k, v, bt, cl, window=window, stream=stream)
    plan = vt.vt_paged_attn_last_plan()
    vt.vt_paged_attn_set_override(0, 0)
    torch.cuda.synchronize()
    assert vt.vt_paged_attn_device_status() == 0
    return out.cpu(), plan


def oracle_rows(case, rows=None, window=None, lens=None):
    import oracle
    o = oracle.default_oracle()
    w = case.workload
    k, v, bt = case.compact()
    cl = case.context_lens if lens is None else lens
    args = (W.to_oracle_array(case.q), W.to_oracle_array(k), W.to_oracle_array(v), bt.numpy(), cl.numpy(),
            w.scale, w.window if window is None else window)
    if rows is None:
        rows = [(b, i) for b in range(w.num_seqs) for i in range(w.num_q_heads)]
    if case.fp8:
        ks, vs = case.scales()
        return np.asarray(rows), o.decode_rows_e4m3(rows, args[0], args[1], args[2], ks.numpy(), vs.numpy(),
                                                    *args[3:], threads=THREADS)
    return np.asarray(rows), o.decode_rows(rows, *args, threads=THREADS)


def compare(got, ref, dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = got - ref
    maxabs = float(np.abs(err).max()) if err.size else 0.0
    if dtype == torch.float32:
        assert maxabs <= F32_MAXABS, f"{what}: fp32 max|err| {maxabs:.3e}"
        return maxabs, 0.0
    nmse = float((err ** 2).sum() / max((ref ** 2).sum(), 1e-300))
    assert nmse <= BF16_NMSE and maxabs <= BF16_MAXABS, f"{what}: nmse {nmse:.3e} max|err| {maxabs:.3e}"
    return maxabs, nmse


def check_case(case, dev, rows=None, **kw):
    out, plan = gpu_run(case, dev, **kw)
    # the intended variant ran: head_dim, storage type and consumer kind
    w = case.workload
    code = {"bf16": vt.VT_BF16, "f32": vt.VT_F32, "e4m3": vt.VT_E4M3}[w.dtype]
    assert plan["head_dim"] == w.head_dim and plan["dtype"] == code
    assert plan["tensor_cores"] == (0 if w.dtype == "f32" else 1)
    assert plan["group_tile"] * plan["subgroups"] >= w.num_q_heads // w.num_kv_heads
    idx, ref = oracle_rows(case, rows, window=kw.get("window"))
    got = out[idx[:, 0], idx[:, 1]].to(torch.float64).numpy()
    return compare(got, ref, case.q.dtype, case.workload.name), plan


# ---------------------------------------------------------------------------
SMALL = [W.TINY, W.QWEN3_1P7B, W.D256_GQA4, W.D256_GQA4_W1024, W.D256_GQA4_F32, W.D256_GQA4_F32_W1024,
         W.D64_GQA4, W.D64_GQA4_F32, W.QWEN3_1P7B_FP8, W.D256_GQA4_FP8, W.D256_GQA4_W1024_FP8,
         W.D512_GQA4, W.D512_GQA4_W1024, W.D64_GQA4_FP8]


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_workload_all_rows(dev, w, seed):
    """Every output row of the small and medium workloads, default launch plan."""
    check_case(W.make_case(w, seed), dev)


def _sample_rows(case, n_seqs=6):
    """All heads of the longest, the shortest and a few other sequences."""
    L = case.context_lens.numpy()
    order = np.argsort(L)
    pick = {int(order[0]), int(order[-1]), int(order[len(order) // 2])}
    rng = np.random.default_rng(case.seed)
    pick |= set(int(x) for x in rng.choice(len(L), size=min(n_seqs, len(L)), replace=False))
    return [(b, i) for b in sorted(pick) for i in range(case.workload.num_q_heads)]


@pytest.mark.parametrize("w", [W.LARGE_GQA, W.SKEWED, W.BATCH1_LONG, W.LARGE_GQA_FP8, W.SKEWED_FP8,
                               W.BATCH1_LONG_FP8], ids=lambda w: w.name)
def test_workload_full_size_sampled(dev, w):
    """Full-size workloads in the benchmark's launch plan; the oracle checks all
    heads of sampled sequences (always the longest and the shortest)."""
    case = W.make_case(w, 0)
    check_case(case, dev, rows=_sample_rows(case))


@pytest.mark.parametrize("grid", [1, 2, 3, 7, 64, 152, 500, 1500])
@pytest.mark.parametrize("w", [W.QWEN3_1P7B, W.D256_GQA4_W1024, W.D256_GQA4_F32, W.D64_GQA4, W.QWEN3_1P7B_FP8,
                               W.D256_GQA4_W1024_FP8, W.D512_GQA4_W1024], ids=lambda w: w.name)
def test_forced_partitions(dev, w, grid):
    """The split/no-split paths and the combine: any CTA count (with at least
    one tile per CTA) gives the oracle's result."""
    (_, _), plan = check_case(W.make_case(w, 4), dev, grid=grid, min_units=1)
    assert plan["grid_ctas"] == grid


STRADDLE = (1, 31, 32, 33, 64, 100, 685, 1000)


@pytest.mark.parametrize("ctx", STRADDLE)
def test_page_boundary_contexts(dev, ctx):
    """Contexts straddling the 32-token page, at the Qwen3 geometry (16 q / 8 kv
    heads, head_dim 128: 2048 outputs), split and unsplit."""
    case = W.make_case(W.custom(f"straddle{ctx}", [ctx], 16, 8, 128), 7)
    check_case(case, dev)
    check_case(case, dev, grid=max(2, ctx // 16), min_units=1)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (12, 4), (16, 4), (20, 4), (32, 4), (48, 4), (64, 4), (6, 2)])
@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (256, "bf16"), (128, "f32"), (64, "bf16"), (64, "f32"),
                                     (64, "e4m3"), (128, "e4m3"), (256, "e4m3"), (512, "bf16")])
def test_group_sizes(dev, hq, hkv, d, dtype):
    """GQA groups 1..16 including ones that pad the group tile (3, 5) or need
    several query subgroups per kv head (12, 16)."""
    case = W.make_case(W.custom(f"g{hq // hkv}", [1, 40, 97, 300], hq, hkv, d, dtype=dtype), 8)
    check_case(case, dev)
    check_case(case, dev, grid=5, min_units=1)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("window", [1, 2, 31, 32, 33, 64, 299, 300, 301, 5000])
def test_windows(dev, window, dtype):
    case = W.make_case(W.custom("win", [1, 33, 300, 1000], 16, 4, 128, dtype=dtype), 9)
    check_case(case, dev, window=window)
    check_case(case, dev, window=window, grid=11, min_units=1)


@pytest.mark.parametrize("d", [512])
def test_head_dim_512_page_boundary_contexts(dev, d):
    """The head_dim 512 arm on the contexts straddling the 32-token page, with
    and without a window, split and unsplit."""
    case = W.make_case(W.custom(f"d{d}_straddle", list(STRADDLE), 16, 4, d), 29)
    for window in (0, 33, 300):
        check_case(case, dev, window=window)
        check_case(case, dev, window=window, grid=13, min_units=1)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp8_page_boundary_contexts(dev, d):
    """The FP8 arm on the contexts straddling the 32-token page, with and
    without a window, split and unsplit."""
    case = W.make_case(W.custom(f"fp8_straddle_d{d}", list(STRADDLE), 16, 4, d, dtype="e4m3"), 26)
    for window in (0, 33, 300):
        check_case(case, dev, window=window)
        check_case(case, dev, window=window, grid=13, min_units=1)


def test_fp8_scales_per_head(dev):
    """Scaling one kv head's key or value scale acts on exactly that head's
    query rows: the value scale multiplies them, the key scale sharpens their
    softmax (checked against the oracle with the same scales)."""
    case = W.make_case(W.custom("fp8_scales", [40, 300, 77], 16, 4, 128, dtype="e4m3"), 27)
    base, _ = gpu_run(case, dev)
    ks, vs = case.extra["k_scale"].clone(), case.extra["v_scale"].clone()
    case.extra["v_scale"][2] *= 4
    case.extra["k_scale"][1] *= 3
    try:
        check_case(case, dev)
        got, _ = gpu_run(case, dev)
    finally:
        case.extra["k_scale"], case.extra["v_scale"] = ks, vs
    g = case.workload.group
    for i in range(16):
        h = i // g
        if h == 2:
            assert torch.equal(got[:, i].float(), (base[:, i].float() * 4).bfloat16().float())
        elif h == 1:
            assert not torch.equal(got[:, i], base[:, i])
        else:
            assert torch.equal(got[:, i], base[:, i])


def test_fp8_invalid_device_data_and_empty(dev):
    """FP8 arm: an empty context gives a zero row, a page id outside the pool
    NaN rows for that sequence only."""
    case = W.make_case(W.custom("fp8_bad", [0, 40, 70, 33], 8, 2, 128, dtype="e4m3"), 28)
    bt = case.block_tables.clone()
    bt[2, 1] = case.num_blocks + 1
    for grid in (0, 3):
        out, _ = gpu_run(case, dev, tables=bt, grid=grid, min_units=1)
        assert torch.count_nonzero(out[0]) == 0
        assert torch.isnan(out[2].float()).all()
        idx, ref = oracle_rows(case, [(b, i) for b in (1, 3) for i in range(8)])
        compare(out[idx[:, 0], idx[:, 1]].double().numpy(), ref, torch.bfloat16)


@pytest.mark.parametrize("d,dtype", [(64, "e4m3"), (128, "e4m3"), (256, "e4m3"), (64, "bf16")], ids=lambda x: str(x))
def test_alternate_page_pairs(dev, d, dtype):
    """The arms whose warps form two pairs taking alternate ring stages: odd
    and even page counts (an odd segment is closed by a stage without tiles,
    which for a one-page segment is also the second pair's first), split
    items at many grids, windows, and a bad page id seen by either pair
    poisoning only its sequence.  Repeated calls give the same bits."""
    lens = [1, 32, 33, 64, 65, 95, 96, 97, 700, 1500, 0, 31]
    case = W.make_case(W.custom(f"pairs_{dtype}_d{d}", lens, 8, 2, d, dtype=dtype), 31)
    for window in (0, 40, 333):
        for grid in (0, 3, 13, 301):
            (_, _), plan = check_case(case, dev, window=window, grid=grid, min_units=1 if grid else 0)
            assert plan["group_tile"] == 8
    bt = case.block_tables.clone()
    bt[4, 1] = case.num_blocks + 2   # second page of a three-page context: the second pair's
    bt[5, 2] = -1                    # third page of another: the first pair's
    ok_rows = [(b, i) for b in (0, 1, 2, 3, 6, 7, 8, 9, 11) for i in range(8)]
    for grid in (0, 7):
        out, _ = gpu_run(case, dev, tables=bt, grid=grid, min_units=1)
        assert torch.isnan(out[4].float()).all() and torch.isnan(out[5].float()).all()
        assert torch.count_nonzero(out[10]) == 0
        idx, ref = oracle_rows(case, ok_rows)
        compare(out[idx[:, 0], idx[:, 1]].double().numpy(), ref, case.q.dtype, "pairs with bad pages")
    a, _ = gpu_run(case, dev, grid=13, min_units=1)
    b, _ = gpu_run(case, dev, grid=13, min_units=1)
    assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_head_dim_64_windows_and_boundaries(dev, dtype):
    """The head_dim 64 arm on the straddling contexts, with and without a
    window, split and unsplit."""
    case = W.make_case(W.custom("d64_edges", list(STRADDLE), 16, 8, 64, dtype=dtype), 22)
    for window in (0, 33, 300):
        check_case(case, dev, window=window)
        check_case(case, dev, window=window, grid=13, min_units=1)


def test_empty_contexts_give_zero_rows(dev):
    case = W.make_case(W.custom("empty", [0, 5, 0, 70, 0], 8, 2, 128), 10)
    out, _ = gpu_run(case, dev)
    for b in (0, 2, 4):
        assert torch.count_nonzero(out[b]) == 0
    idx, ref = oracle_rows(case, [(b, i) for b in (1, 3) for i in range(8)])
    compare(out[idx[:, 0], idx[:, 1]].double().numpy(), ref, torch.bfloat16)
    allempty = W.make_case(W.custom("allempty", [0, 0], 8, 2, 256), 10)
    out, _ = gpu_run(allempty, dev)
    assert torch.count_nonzero(out) == 0


def test_invalid_device_data_poisons_only_its_rows(dev):
    """A page id outside the pool or an impossible context length turns only the
    affected rows into NaN; nothing faults and other sequences are exact."""
    case = W.make_case(W.custom("bad", [40, 70, 33, 100], 8, 2, 128), 11)
    bt = case.block_tables.clone()
    lens = case.context_lens.clone()
    bt[1, 1] = case.num_blocks + 5        # sequence 1: page id past the pool
    bt[2, 0] = -3                         # sequence 2: negative page id
    lens[3] = case.workload.max_blocks_per_seq * 32 + 1  # sequence 3: longer than its table row
    for grid in (0, 3):
        out, _ = gpu_run(case, dev, tables=bt, lens=lens, grid=grid, min_units=1)
        assert torch.isnan(out[1].float()).all() and torch.isnan(out[2].float()).all()
        assert torch.isnan(out[3].float()).all()
        idx, ref = oracle_rows(case, [(0, i) for i in range(8)])
        compare(out[idx[:, 0], idx[:, 1]].double().numpy(), ref, torch.bfloat16)
    neg = case.context_lens.clone()
    neg[0] = -1
    out, _ = gpu_run(case, dev, lens=neg)
    assert torch.isnan(out[0].float()).all()


@pytest.mark.parametrize("w", [W.QWEN3_1P7B, W.D256_GQA4_F32, W.D64_GQA4_F32,
                               W.custom("f32_d128_g8", [1, 33, 700, 2000], 64, 8, 128, dtype="f32")],
                         ids=lambda w: w.name)
def test_deterministic_bits(dev, w):
    """Same inputs and plan, same bits: bf16 and fp32 storage (the fp32 row
    groups merge in a fixed order), several grids, repeated calls."""
    case = W.make_case(w, 12)
    for grid in (0, 40, 301):
        a, _ = gpu_run(case, dev, grid=grid, min_units=1 if grid else 0)
        for _ in range(3):
            b, _ = gpu_run(case, dev, grid=grid, min_units=1 if grid else 0)
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), grid


def test_default_plan(dev):
    case = W.make_case(W.QWEN3_1P7B, 0)
    _, plan = gpu_run(case, dev)
    props = torch.cuda.get_device_properties(0)
    assert plan["num_sms"] == props.multi_processor_count
    assert plan["grid_ctas"] == plan["num_sms"] * plan["ctas_per_sm"]
    assert plan["stages"] >= 2 and plan["group_tile"] == 8 and plan["subgroups"] == 1
    assert plan["tensor_cores"] == 1
    assert plan["workspace_bytes"] > 0


def test_default_segment_cost(dev):
    """The partition's default segment weight: 2 tiles for bf16 K/V, 6 for an
    FP8 cache or several new tokens per sequence; each result is the oracle's."""
    cases = ((W.make_case(W.QWEN3_1P7B, 0), 2), (W.make_case(W.QWEN3_1P7B_FP8, 0), 6),
             (W.make_case(W.custom("segdef_multi", [100, 40, 1200], 8, 2, 128, q_len=3), 0), 6))
    for case, cost in cases:
        _, plan = gpu_run(case, dev)
        assert plan["segment_cost"] == cost, case.workload.name
        if case.workload.q_len == 1:
            check_case(case, dev)
        else:
            check_multi(case, dev)


def test_side_stream_and_reuse(dev):
    """Calls on a non-default stream, back to back with different shapes, share
    the library workspace correctly."""
    s = torch.cuda.Stream()
    cases = [W.make_case(W.QWEN3_1P7B, 13), W.make_case(W.D256_GQA4, 13),
             W.make_case(W.custom("many", [3] * 300, 8, 8, 128), 13)]
    with torch.cuda.stream(s):
        for case in cases:
            out, _ = gpu_run(case, dev, stream=s, grid=97, min_units=1)
            idx, ref = oracle_rows(case)
            compare(out[idx[:, 0], idx[:, 1]].double().numpy(), ref, case.q.dtype, case.workload.name)


def test_scale_zero_gives_mean_of_values(dev):
    case = W.make_case(W.custom("scale0", [77], 4, 2, 128), 14)
    k, v = case.pool(dev)
    out = vt.decode(case.q.to(dev), k, v, case.block_tables.to(dev), case.context_lens.to(dev), scale=0.0)
    idx = torch.tensor([case.block_tables[0, t // 32] for t in range(77)])
    vv = v[idx.to(dev), torch.arange(77, device=dev) % 32].double()  # [77][Hkv][D]
    mean = vv.mean(0)
    for i in range(4):
        assert (out[0, i].double() - mean[i // 2]).abs().max() < 2e-2


@pytest.mark.parametrize("cost", [0, 1, 5, 33])
@pytest.mark.parametrize("w", [W.QWEN3_1P7B, W.D256_GQA4_W1024, W.D256_GQA4_F32], ids=lambda w: w.name)
def test_segment_cost(dev, w, cost):
    """Segment boundaries weigh `cost` tiles in the split: slices then start
    and end inside an item's weight as well as inside its pages, and CTAs
    whose slice is only weight get no tile.  Any weight gives the oracle's
    result, at several grids."""
    vt.vt_paged_attn_set_segment_cost(cost)
    case = W.make_case(w, 20)
    for grid in (0, 7, 64, 700):
        (_, _), plan = check_case(case, dev, grid=grid, min_units=1 if grid else 0)
        assert plan["segment_cost"] == cost


def test_segment_cost_ragged(dev):
    """Empty, one-page and long sequences, a window, and query subgroups,
    with a heavy segment weight and a grid that leaves CTAs without pages."""
    vt.vt_paged_attn_set_segment_cost(9)
    lens = [0, 1, 700, 31, 0, 33, 2000, 64, 5, 1000, 0, 257]
    case = W.make_case(W.custom("segcost_ragged", lens, 64, 4, 128), 21)
    for window in (0, 100):
        for grid in (0, 5, 300):
            out, _ = gpu_run(case, dev, grid=grid, min_units=1 if grid else 0, window=window)
            rows = [(b, i) for b in range(len(lens)) if lens[b] > 0 for i in range(64)]
            idx, ref = oracle_rows(case, rows, window=window)
            compare(out[idx[:, 0], idx[:, 1]].double().numpy(), ref, torch.bfloat16, f"w{window} g{grid}")
            for b in (0, 4, 10):
                assert torch.count_nonzero(out[b]) == 0


def _overlap_cases():
    return [W.make_case(W.QWEN3_1P7B, 18), W.make_case(W.custom("ovl_empty", [0, 70, 0, 1000, 33], 16, 4, 128), 18),
            W.make_case(W.D256_GQA4_W1024, 18), W.make_case(W.custom("ovl_f32", [5, 300, 2000], 8, 2, 128, dtype="f32"), 18),
            W.make_case(W.custom("ovl_fp8", [7, 500, 1200], 32, 8, 128, dtype="e4m3"), 18)]


def test_overlap_back_to_back(dev):
    """Programmatic dependent launches, decode after decode on one stream with
    no host synchronisation (each call starts while the previous one
    finishes), including empty sequences (rows written after the dependency
    wait) and a call that overwrites the previous call's output buffer."""
    vt.vt_paged_attn_set_overlap(True)
    cases = _overlap_cases()
    dev_in = []
    for case in cases:
        k, v = case.pool(dev)
        dev_in.append((case, case.q.to(dev), k, v, case.block_tables.to(dev), case.context_lens.to(dev)))
    outs = {(r, j): torch.full_like(x[1], float("nan")) for r in range(3) for j, x in enumerate(dev_in)}
    # a second batch of the first shape, for the write-after-write check
    other = W.make_case(W.QWEN3_1P7B, 19)
    ko, vo = other.pool(dev)
    o_in = (other.q.to(dev), ko, vo, other.block_tables.to(dev), other.context_lens.to(dev))
    shared = torch.full_like(dev_in[0][1], float("nan"))
    torch.cuda.synchronize()
    for r in range(3):
        for j, (case, q, k, v, bt, cl) in enumerate(dev_in):
            run_decode(case, q, k, v, bt, cl, out=outs[(r, j)])
            assert vt.vt_paged_attn_last_plan()["launch_overlap"] == 1
    case0, q0, k0, v0, bt0, cl0 = dev_in[0]
    vt.decode(q0, k0, v0, bt0, cl0, case0.workload.scale, out=shared)
    vt.decode(*o_in, other.workload.scale, out=shared)  # overwrites the rows just written
    torch.cuda.synchronize()
    assert vt.vt_paged_attn_device_status() == 0
    for j, (case, *_rest) in enumerate(dev_in):
        idx, ref = oracle_rows(case)
        for r in range(3):
            got = outs[(r, j)].cpu()
            compare(got[idx[:, 0], idx[:, 1]].double().numpy(), ref, case.q.dtype, f"{case.workload.name} rep {r}")
        assert torch.equal(outs[(0, j)].cpu().view(torch.uint8), outs[(2, j)].cpu().view(torch.uint8))
    idx, ref = oracle_rows(other)
    compare(shared.cpu()[idx[:, 0], idx[:, 1]].double().numpy(), ref, torch.bfloat16, "overwritten buffer")


def test_overlap_in_cuda_graph(dev):
    """The same launches captured in a CUDA graph (programmatic edges) and
    replayed: results equal the eager ones bit for bit."""
    vt.vt_paged_attn_set_overlap(True)
    cases = _overlap_cases()[:3]
    dev_in = []
    for case in cases:
        k, v = case.pool(dev)
        dev_in.append((case, case.q.to(dev), k, v, case.block_tables.to(dev), case.context_lens.to(dev),
                       torch.empty_like(case.q, device=dev)))

    def run_all():
        for case, q, k, v, bt, cl, out in dev_in:
            vt.decode(q, k, v, bt, cl, case.workload.scale, case.workload.window, out=out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run_all()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [x[-1].clone() for x in dev_in]
    for x in dev_in:
        x[-1].fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_all()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert vt.vt_paged_attn_device_status() == 0
    for e, x in zip(eager, dev_in):
        assert torch.equal(e.view(torch.uint8), x[-1].view(torch.uint8))


def test_device_status_clean(dev):
    assert vt.vt_paged_attn_device_status() == 0


def test_caller_workspace(dev):
    """vt_paged_attn_set_workspace: decodes on a caller-owned workspace give the
    oracle's results (split and unsplit, shapes growing and shrinking, so the
    counter region grows in place), report it in the plan, refuse a call the
    buffer cannot hold, and the library's own workspace takes over again
    after the buffer is withdrawn."""
    cases = [W.make_case(W.QWEN3_1P7B, 23), W.make_case(W.custom("ws_many", [3] * 700, 8, 8, 128), 23),
             W.make_case(W.D256_GQA4_F32_W1024, 23), W.make_case(W.QWEN3_1P7B, 24)]
    # the counter region only grows, so a buffer for calls of several shapes
    # holds the largest counter region plus the largest partials: the sum of
    # the calls' needs is more than enough
    need = sum(vt.vt_paged_attn_workspace_bytes(c.workload.num_seqs, c.workload.num_q_heads,
                                                 c.workload.num_kv_heads, c.workload.head_dim,
                                                 vt.VT_BF16 if c.q.dtype == torch.bfloat16 else vt.VT_F32)
               for c in cases)
    buf = torch.full((need,), 0x5A, dtype=torch.uint8, device=dev)  # dirty on purpose
    vt.vt_paged_attn_set_workspace(buf.data_ptr(), buf.numel())
    try:
        for case in cases:
            for grid in (0, 77):
                (_, _), plan = check_case(case, dev, grid=grid, min_units=1 if grid else 0)
                assert plan["scratch_source"] == 1 and plan["workspace_bytes"] <= buf.numel()
        small = torch.empty(vt.VT_MIN_WORKSPACE_BYTES, dtype=torch.uint8, device=dev)
        vt.vt_paged_attn_set_workspace(small.data_ptr(), small.numel())
        case = cases[0]
        k, v = case.pool(dev)
        with pytest.raises(vt.VtError) as err:
            vt.decode(case.q.to(dev), k, v, case.block_tables.to(dev), case.context_lens.to(dev))
        assert err.value.status == vt.VT_ERR_SCRATCH_LIMIT
        torch.cuda.synchronize()
    finally:
        vt.vt_paged_attn_set_workspace(0, 0)
    (_, _), plan = check_case(cases[0], dev)
    assert plan["scratch_source"] == 0


def _give_up(case, dev, entry):
    """One call whose CTA 0 withholds its second tile under a short wait limit
    (about 2 ms): returns the status word, the detail words and the output."""
    w = case.workload
    k, v = case.pool(dev)
    q, bt, cl = case.q.to(dev), case.block_tables.to(dev), case.context_lens.to(dev)
    out = torch.zeros_like(q)
    vt.vt_paged_attn_set_override(1, 1)  # one CTA holds every tile
    vt.vt_paged_attn_set_test_wait(1 << 22, 0, 1)
    try:
        B, Hq, D = q.shape
        st = entry(out.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), bt.data_ptr(), cl.data_ptr(), B, Hq,
                   w.num_kv_heads, D, 32, w.scale, w.window, torch.cuda.current_stream().cuda_stream,
                   bt.shape[1], case.num_blocks, vt.dtype_code(q))
        assert st == vt.VT_OK
    finally:
        vt.vt_paged_attn_set_test_wait(0, -1, -1)
        vt.vt_paged_attn_set_override(0, 0)
    torch.cuda.synchronize()
    detail = vt.vt_paged_attn_device_status_detail(n_words=5)
    status = vt.vt_paged_attn_device_status()
    return status, detail, out


@pytest.mark.parametrize("path", ["library", "caller_workspace", "noalloc"])
def test_bounded_wait_gives_up_and_reports(dev, path):
    """The failure path of a bounded wait, made to happen without any fault:
    a test hook shortens the wait limit and has CTA 0 withhold a tile.  The
    consumers' wait for it runs out, the kernel returns, the status reads
    back as a timeout of the page-tile wait (bit 0) with CTA 0 and a consumer
    thread recorded, on each scratch path; reading it clears it, and the next
    normal call is exact against the oracle."""
    case = W.make_case(W.custom("giveup", [100, 700], 16, 4, 128), 25)
    entry = vt.vt_paged_attn_decode_noalloc if path == "noalloc" else vt.vt_paged_attn_decode
    buf = None
    if path == "caller_workspace":
        buf = torch.empty(8 << 20, dtype=torch.uint8, device=dev)
        vt.vt_paged_attn_set_workspace(buf.data_ptr(), buf.numel())
    try:
        status, detail, _ = _give_up(case, dev, entry)
        assert status & 1, f"status {status:#x}"
        assert detail[0] & 1 and detail[1] == 1, detail   # CTA 0 gave up first
        assert detail[2] & 0xFF == 1 and (detail[2] >> 8) < 128, detail  # a consumer thread's tile wait
        assert vt.vt_paged_attn_device_status() == 0     # reading cleared it
        # the same path, normal operation again: exact against the oracle
        k, v = case.pool(dev)
        q, bt, cl = case.q.to(dev), case.block_tables.to(dev), case.context_lens.to(dev)
        out = torch.full_like(q, float("nan"))
        for grid in (0, 3):
            vt.vt_paged_attn_set_override(grid, 1 if grid else 0)
            st = entry(out.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), bt.data_ptr(), cl.data_ptr(), 2,
                       16, 4, 128, 32, case.workload.scale, 0, torch.cuda.current_stream().cuda_stream,
                       bt.shape[1], case.num_blocks, vt.VT_BF16)
            assert st == vt.VT_OK
            torch.cuda.synchronize()
            assert vt.vt_paged_attn_device_status() == 0
            idx, ref = oracle_rows(case)
            compare(out.cpu()[idx[:, 0], idx[:, 1]].double().numpy(), ref, torch.bfloat16, f"{path} grid {grid}")
    finally:
        vt.vt_paged_attn_set_override(0, 0)
        if buf is not None:
            vt.vt_paged_attn_set_workspace(0, 0)


@pytest.mark.parametrize("tile", [1, 2])
@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (128, "e4m3")], ids=lambda x: str(x))
def test_bounded_wait_gives_up_alternate_pairs(dev, d, dtype, tile):
    """The give-up path on the arms whose warp pairs take alternate stages:
    CTA 0 withholds a tile of the second pair (tile 1) or of the first
    (tile 2); the waits run out, the status reports a page-tile timeout by a
    consumer thread of CTA 0, and the next call is exact."""
    case = W.make_case(W.custom(f"giveup_pairs_{dtype}_d{d}", [100, 700], 16, 4, d, dtype=dtype), 29)
    w = case.workload
    k, v = case.pool(dev)
    q, bt, cl = case.q.to(dev), case.block_tables.to(dev), case.context_lens.to(dev)
    vt.vt_paged_attn_set_override(1, 1)
    vt.vt_paged_attn_set_test_wait(1 << 22, 0, tile)
    try:
        run_decode(case, q, k, v, bt, cl)
    finally:
        vt.vt_paged_attn_set_test_wait(0, -1, -1)
        vt.vt_paged_attn_set_override(0, 0)
    torch.cuda.synchronize()
    detail = vt.vt_paged_attn_device_status_detail(n_words=5)
    status = vt.vt_paged_attn_device_status()
    assert status & 1, f"status {status:#x}"
    assert detail[1] == 1 and detail[2] & 0xFF == 1 and (detail[2] >> 8) < 128, detail
    assert vt.vt_paged_attn_device_status() == 0
    for grid in (0, 3):
        check_case(case, dev, grid=grid, min_units=1 if grid else 0)


# ---------------------------------------------------------------------------
# Multi-token decode (q_len new tokens per sequence, causal within them)
# ---------------------------------------------------------------------------
def oracle_multi_rows(case, rows=None, window=None, lens=None):
    """The oracle's multi-token rows; an FP8 cache enters as its values in
    fp64 (codes decoded by torch's float8_e4m3fn, the decoder the oracle's own
    E4M3 decoding is pinned against, times the per-kv-head scales)."""
    import oracle
    o = oracle.default_oracle()
    w = case.workload
    k, v, bt = case.compact()
    q = case.q
    if case.fp8:
        ks, vs = case.scales()
        k = k.view(torch.float8_e4m3fn).to(torch.float64) * ks.double()[None, None, :, None]
        v = v.view(torch.float8_e4m3fn).to(torch.float64) * vs.double()[None, None, :, None]
        q = q.to(torch.float64)  # exact; the oracle takes one storage type for q and the caches
    cl = case.context_lens if lens is None else lens
    if rows is None:
        rows = [(b, j, i) for b in range(w.num_seqs) for j in range(w.q_len) for i in range(w.num_q_heads)]
    ref = o.decode_multi_rows(rows, W.to_oracle_array(q), W.to_oracle_array(k), W.to_oracle_array(v),
                              bt.numpy(), cl.numpy(), w.scale, w.window if window is None else window,
                              threads=THREADS)
    return np.asarray(rows), ref


def check_multi(case, dev, rows=None, **kw):
    out, plan = gpu_run(case, dev, **kw)
    w = case.workload
    assert plan["q_len"] == w.q_len and plan["head_dim"] == w.head_dim
    assert plan["group_tile"] * plan["subgroups"] >= w.q_len * (w.num_q_heads // w.num_kv_heads)
    idx, ref = oracle_multi_rows(case, rows, window=kw.get("window"))
    got = out[idx[:, 0], idx[:, 1], idx[:, 2]].to(torch.float64).numpy()
    return compare(got, ref, case.q.dtype, w.name), plan


@pytest.mark.parametrize("q_len", [2, 3, 4, 7])
@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8), (8, 8), (12, 4)])
def test_multi_token(dev, q_len, hq, hkv):
    """Every row of a multi-token decode (new tokens j attend causally to the
    first L - q_len + 1 + j tokens) against the oracle: contexts from exactly
    q_len up, straddling pages; windows; split and unsplit; query rows that
    span several tensor-core tiles (subgroups)."""
    lens = [q_len, q_len + 1, 31, 33, 100, 685]
    case = W.make_case(W.custom(f"multi_q{q_len}", lens, hq, hkv, 128, q_len=q_len), 30 + q_len)
    for window in (0, 5, 64):
        check_multi(case, dev, window=window)
        check_multi(case, dev, window=window, grid=9, min_units=1)


@pytest.mark.parametrize("d,dtype", [(128, "f32"), (256, "bf16"), (64, "bf16"), (512, "bf16"), (64, "f32")])
def test_multi_token_head_dims(dev, d, dtype):
    case = W.make_case(W.custom(f"multi_d{d}_{dtype}", [4, 40, 300, 97], 16, 4, d, dtype=dtype, q_len=4), 31)
    for window in (0, 50):
        check_multi(case, dev, window=window)
        check_multi(case, dev, window=window, grid=7, min_units=1)


def test_multi_token_q_len_one_is_decode(dev):
    """q_len = 1 through the multi-token entry point gives the single-token
    decode's bits."""
    case = W.make_case(W.QWEN3_1P7B, 32)
    single, _ = gpu_run(case, dev)
    k, v = case.pool(dev)
    q = case.q.to(dev)[:, None]
    out = vt.decode_multi(q, k, v, case.block_tables.to(dev), case.context_lens.to(dev), case.workload.scale)
    torch.cuda.synchronize()
    assert vt.vt_paged_attn_last_plan()["q_len"] == 1
    assert torch.equal(out[:, 0].cpu().view(torch.int16), single.view(torch.int16))


def test_multi_token_short_context_is_nan(dev):
    """A context shorter than its q_len new tokens turns only that sequence's
    rows into NaN; the other sequences are exact."""
    case = W.make_case(W.custom("multi_short", [10, 40, 70], 8, 2, 128, q_len=4), 33)
    lens = case.context_lens.clone()
    lens[1] = 3
    out, _ = gpu_run(case, dev, lens=lens)
    assert torch.isnan(out[1].float()).all()
    idx, ref = oracle_multi_rows(case, [(b, j, i) for b in (0, 2) for j in range(4) for i in range(8)], lens=lens)
    compare(out[idx[:, 0], idx[:, 1], idx[:, 2]].double().numpy(), ref, torch.bfloat16)


@pytest.mark.parametrize("q_len", [2, 3, 4, 7])
@pytest.mark.parametrize("hq,hkv,d", [(16, 8, 128), (32, 8, 128), (8, 8, 128), (12, 4, 128), (16, 4, 256),
                                      (16, 4, 64)])
def test_multi_token_fp8(dev, q_len, hq, hkv, d):
    """Several new tokens over an FP8 cache (vt_paged_attn_decode_multi_fp8):
    every row against the oracle on the dequantised cache, with windows, split
    and unsplit, query rows in one or several tensor-core tiles."""
    lens = [q_len, q_len + 1, 31, 33, 100, 685]
    case = W.make_case(W.custom(f"multi_fp8_q{q_len}_d{d}", lens, hq, hkv, d, dtype="e4m3", q_len=q_len),
                       40 + q_len)
    for window in (0, 5, 64):
        (_, _), plan = check_multi(case, dev, window=window)
        assert plan["dtype"] == vt.VT_E4M3
        check_multi(case, dev, window=window, grid=9, min_units=1)


def test_multi_token_fp8_q_len_one_is_decode(dev):
    """q_len = 1 through the FP8 multi-token entry gives the FP8 decode's bits."""
    case = W.make_case(W.QWEN3_1P7B_FP8, 34)
    single, _ = gpu_run(case, dev)
    k, v = case.pool(dev)
    ks, vs = case.scales(dev)
    q = case.q.to(dev)[:, None]
    out = vt.decode_fp8(q, k, v, ks, vs, case.block_tables.to(dev), case.context_lens.to(dev), case.workload.scale)
    torch.cuda.synchronize()
    assert vt.vt_paged_attn_last_plan()["q_len"] == 1
    assert torch.equal(out[:, 0].cpu().view(torch.int16), single.view(torch.int16))


@pytest.mark.parametrize("w", [W.MULTI_Q4, W.MULTI_Q4_FP8], ids=lambda w: w.name)
def test_multi_token_full_size_sampled(dev, w):
    """The multi-token benchmark batches in the benchmark's launch plan, all
    rows of sampled sequences."""
    case = W.make_case(w, 0)
    L = case.context_lens.numpy()
    pick = sorted({int(np.argmin(L)), int(np.argmax(L)), 7, 30, 55})
    rows = [(b, j, i) for b in pick for j in range(4) for i in range(32)]
    check_multi(case, dev, rows=rows)


# ---------------------------------------------------------------------------
# Seeded random configurations across the whole surface
# ---------------------------------------------------------------------------
_RANDOM_ARMS = [(64, "bf16"), (64, "e4m3"), (64, "f32"), (128, "bf16"), (128, "f32"), (128, "e4m3"),
                (128, "e4m3"), (128, "e4m3"), (256, "bf16"), (256, "f32"), (256, "e4m3"), (256, "e4m3"),
                (512, "bf16")]


@pytest.mark.parametrize("seed", range(48))
def test_random_configurations(dev, seed):
    """A seeded draw of head_dim and storage, group size, new tokens per
    sequence, window, context mix (empty, one-token, page-straddling and long
    contexts) and a forced or default grid; sampled rows of every sequence
    against the oracle."""
    rng = np.random.default_rng(1000 + seed)
    d, dtype = _RANDOM_ARMS[int(rng.integers(len(_RANDOM_ARMS)))]
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16]))
    q_len = int(rng.choice([1, 1, 1, 2, 4]))
    if q_len * g > 64:
        q_len = 1
    B = int(rng.integers(1, 9))
    pool = [0, 1, 2, 31, 32, 33, 63, 64, 65, 95, 97, 129, 300, 777, 1500]
    lens = [int(rng.choice(pool)) for _ in range(B)]
    lens = [max(L, q_len) if L > 0 else 0 for L in lens]
    if max(lens) == 0:
        lens[0] = 40
    window = int(rng.choice([0, 0, 1, 17, 64, 333]))
    grid = int(rng.choice([0, 0, 1, 3, 17, 200]))
    case = W.make_case(W.custom(f"rand{seed}", lens, hkv * g, hkv, d, dtype=dtype, q_len=q_len), 2000 + seed)
    out, plan = gpu_run(case, dev, window=window, grid=grid, min_units=1 if grid else 0)
    w = case.workload
    heads = sorted({0, w.num_q_heads - 1, int(rng.integers(w.num_q_heads))})
    live = [b for b in range(B) if lens[b] > 0]
    for b in range(B):
        if lens[b] == 0:  # decode: a zero row; several new tokens need L >= q_len: NaN rows
            if q_len == 1:
                assert torch.count_nonzero(out[b]) == 0
            else:
                assert torch.isnan(out[b].float()).all()
    if q_len == 1:
        idx, ref = oracle_rows(case, [(b, i) for b in live for i in heads], window=window)
        got = out[idx[:, 0], idx[:, 1]].to(torch.float64).numpy()
    else:
        rows = [(b, j, i) for b in live for j in range(q_len) for i in heads]
        idx, ref = oracle_multi_rows(case, rows, window=window)
        got = out[idx[:, 0], idx[:, 1], idx[:, 2]].to(torch.float64).numpy()
    compare(got, ref, case.q.dtype, f"seed {seed}: d{d} {dtype} g{g} q_len{q_len} W{window} grid{grid}")
