"""The allocation-free entry point against the regular one and the oracle (GPU).

vt_paged_attn_decode_noalloc serves callers that cannot let the library
allocate device memory (an engine that gave its whole budget to the KV-cache
pool, an external allocator that must own every byte, a decode loop that may
not enter the CUDA allocator).  It runs the same kernel with its scratch in a
fixed static device array.  This file checks, through the C-ABI, that two
calls in a row (the second reusing the array the first left behind) give the
regular entry point's results bit for bit under the same launch plan, that a
call on the default plan matches the oracle within the parity tolerances,
that the status words in the array read back clean, and that a call too
large for the array is refused before anything is launched.

It is named so that pytest collects it last, and it passes both alone in a
fresh process and after the other GPU tests.
"""
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


def _inputs(case, dev):
    k, v = case.pool(dev)
    return (case.q.to(dev), k, v, case.block_tables.to(dev), case.context_lens.to(dev))


def _call(entry, case, t, out):
    q, k, v, bt, cl = t
    w = case.workload
    B, Hq, D = q.shape
    nb, P, Hkv, _ = k.shape
    return entry(out.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), bt.data_ptr(), cl.data_ptr(), B, Hq,
                 Hkv, D, P, w.scale, w.window, torch.cuda.current_stream().cuda_stream, bt.shape[1], nb,
                 vt.dtype_code(q))


def _against_oracle(case, got):
    import oracle
    w = case.workload
    k, v, bt = case.compact()
    rows = [(b, i) for b in range(w.num_seqs) for i in range(w.num_q_heads)]
    ref = oracle.default_oracle().decode_rows(
        rows, W.to_oracle_array(case.q), W.to_oracle_array(k), W.to_oracle_array(v), bt.numpy(),
        case.context_lens.numpy(), w.scale, w.window, threads=THREADS)
    idx = np.asarray(rows)
    g = got.cpu()[idx[:, 0], idx[:, 1]].double().numpy()
    assert np.isfinite(g).all()
    err = g - ref
    maxabs = float(np.abs(err).max())
    if case.q.dtype == torch.float32:
        assert maxabs <= F32_MAXABS, maxabs
    else:
        nmse = float((err ** 2).sum() / (ref ** 2).sum())
        assert nmse <= BF16_NMSE and maxabs <= BF16_MAXABS, (nmse, maxabs)


def _noalloc_plan_ok():
    plan = vt.vt_paged_attn_last_plan()
    assert plan["scratch_source"] == 2
    assert plan["workspace_bytes"] <= vt.VT_NOALLOC_SCRATCH_BYTES
    return plan


def test_noalloc_matches_regular_entry_twice_in_a_row(dev):
    # Two different problems back to back: the second call finds the array
    # holding the first call's partials and counters.
    for w, seed in ((W.LARGE_GQA.with_(num_seqs=16), 3), (W.D256_GQA4_F32_W1024, 5)):
        case = W.make_case(w, seed)
        t = _inputs(case, dev)
        ref = torch.empty_like(t[0])
        got = torch.full_like(t[0], float("nan"))
        vt.vt_paged_attn_set_override(0, 1)  # many splits: exercise partials and the combine
        try:
            assert _call(vt.vt_paged_attn_decode, case, t, ref) == vt.VT_OK
            assert _call(vt.vt_paged_attn_decode_noalloc, case, t, got) == vt.VT_OK
            _noalloc_plan_ok()
        finally:
            vt.vt_paged_attn_set_override(0, 0)
        torch.cuda.synchronize()
        assert vt.vt_paged_attn_device_status() == 0
        # same kernel, same plan, same partial order: the same bits
        assert torch.equal(got.view(torch.uint8), ref.view(torch.uint8)), w.name
        _against_oracle(case, got)


def test_noalloc_default_plan_against_oracle(dev):
    """Two calls in a row on the default launch plan, each checked against
    the oracle."""
    for w, seed in ((W.QWEN3_1P7B, 6), (W.D256_GQA4, 6)):
        case = W.make_case(w, seed)
        t = _inputs(case, dev)
        got = torch.full_like(t[0], float("nan"))
        assert _call(vt.vt_paged_attn_decode_noalloc, case, t, got) == vt.VT_OK
        plan = _noalloc_plan_ok()
        assert plan["grid_ctas"] == plan["num_sms"] * plan["ctas_per_sm"]
        torch.cuda.synchronize()
        assert vt.vt_paged_attn_device_status() == 0
        _against_oracle(case, got)


def test_noalloc_refuses_a_call_larger_than_its_array(dev):
    # 300000 sequences x 8 kv heads need ~9.6 MB of arrival counters alone:
    # refused before launch, so these pointers are never dereferenced.
    case = W.make_case(W.TINY, 0)
    t = _inputs(case, dev)
    q, k, v, bt, cl = t
    st = vt.vt_paged_attn_decode_noalloc(q.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), bt.data_ptr(),
                                         cl.data_ptr(), 300000, 16, 8, 128, 32, 0.088, 0,
                                         torch.cuda.current_stream().cuda_stream, 4, 4, vt.VT_BF16)
    assert st == vt.VT_ERR_SCRATCH_LIMIT
    assert "scratch" in vt.vt_status_string(st)
