"""The C-ABI library on a machine without a GPU: it loads, exports every
entry point the header declares, and rejects bad arguments on the host before
touching CUDA."""
import ctypes
import re
from pathlib import Path

import pytest

import paged_attention_decode_kv_gb300 as vt

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "vt_paged_attn.h"


@pytest.fixture(scope="module")
def lib():
    from paged_attention_decode_kv_gb300 import build_lib
    build_lib.build()
    return vt.library()


def declared_functions():
    text = HEADER.read_text()
    return sorted(set(re.findall(r"VT_API\s+[\w\s\*]+?\b(vt_\w+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(vt.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_version_and_status_strings(lib):
    assert vt.vt_paged_attn_version() == 10100
    assert vt.vt_status_string(vt.VT_OK) == "ok"
    assert "unsupported" in vt.vt_status_string(vt.VT_ERR_UNSUPPORTED)
    assert vt.vt_status_string(99) == "unknown status"


def _call(**over):
    args = dict(out=0x1000, q=0x2000, k_cache=0x3000, v_cache=0x4000, block_tables=0x5000,
                context_lens=0x6000, num_seqs=2, num_q_heads=16, num_kv_heads=8, head_dim=128,
                block_size=32, scale=0.088, window=0, stream=None, max_blocks_per_seq=4, num_blocks=16,
                dtype=vt.VT_BF16)
    args.update(over)
    return vt.vt_paged_attn_decode(**args)


@pytest.mark.parametrize("over,status", [
    (dict(num_seqs=0, out=None, q=None), vt.VT_OK),           # empty batch: no-op, no launch
    (dict(num_seqs=-1), vt.VT_ERR_INVALID_ARG),
    (dict(out=None), vt.VT_ERR_INVALID_ARG),
    (dict(k_cache=None), vt.VT_ERR_INVALID_ARG),
    (dict(block_tables=None), vt.VT_ERR_INVALID_ARG),
    (dict(q=0x2008), vt.VT_ERR_INVALID_ARG),                  # 16-byte alignment
    (dict(context_lens=0x6002), vt.VT_ERR_INVALID_ARG),       # 4-byte alignment
    (dict(num_q_heads=12, num_kv_heads=8), vt.VT_ERR_INVALID_ARG),
    (dict(num_kv_heads=0), vt.VT_ERR_INVALID_ARG),
    (dict(head_dim=96), vt.VT_ERR_UNSUPPORTED),
    (dict(head_dim=512, dtype=vt.VT_F32), vt.VT_ERR_UNSUPPORTED),
    (dict(head_dim=1024), vt.VT_ERR_UNSUPPORTED),
    (dict(block_size=16), vt.VT_ERR_UNSUPPORTED),
    (dict(max_blocks_per_seq=0), vt.VT_ERR_INVALID_ARG),
    (dict(num_blocks=0), vt.VT_ERR_INVALID_ARG),
    (dict(num_blocks=1 << 27), vt.VT_ERR_UNSUPPORTED),        # token rows must fit int32
    (dict(scale=float("nan")), vt.VT_ERR_INVALID_ARG),
    (dict(scale=float("inf")), vt.VT_ERR_INVALID_ARG),
    (dict(dtype=7), vt.VT_ERR_INVALID_ARG),
])
def test_host_validation(lib, over, status):
    assert _call(**over) == status


def _fp8_call(multi, **over):
    args = dict(out=0x1000, q=0x2000, k_cache=0x3000, v_cache=0x4000, k_scale=0x7000, v_scale=0x7100,
                block_tables=0x5000, context_lens=0x6000, num_seqs=2, num_q_heads=16, num_kv_heads=8, head_dim=128,
                block_size=32, scale=0.088, window=0, stream=None, max_blocks_per_seq=4, num_blocks=16)
    if multi:
        args["q_len"] = 3
    args.update(over)
    return (vt.vt_paged_attn_decode_multi_fp8 if multi else vt.vt_paged_attn_decode_fp8)(**args)


@pytest.mark.parametrize("multi", [False, True])
@pytest.mark.parametrize("over,status", [
    (dict(num_seqs=0, out=None, q=None), vt.VT_OK),
    (dict(k_scale=None), vt.VT_ERR_INVALID_ARG),
    (dict(v_scale=None), vt.VT_ERR_INVALID_ARG),
    (dict(k_scale=0x7002), vt.VT_ERR_INVALID_ARG),             # 4-byte alignment
    (dict(head_dim=512), vt.VT_ERR_UNSUPPORTED),
    (dict(head_dim=96), vt.VT_ERR_UNSUPPORTED),
    (dict(q=0x2008), vt.VT_ERR_INVALID_ARG),
])
def test_fp8_host_validation(lib, multi, over, status):
    """The FP8 entry points, single- and multi-token, check their scales and
    shapes on the host."""
    assert _fp8_call(multi, **over) == status


def test_multi_token_host_validation(lib):
    base = dict(out=0x1000, q=0x2000, k_cache=0x3000, v_cache=0x4000, block_tables=0x5000, context_lens=0x6000,
                num_seqs=2, q_len=2, num_q_heads=16, num_kv_heads=8, head_dim=128, block_size=32, scale=0.088,
                window=0, stream=None, max_blocks_per_seq=4, num_blocks=16, dtype=vt.VT_BF16)
    assert vt.vt_paged_attn_decode_multi(**dict(base, q_len=0)) == vt.VT_ERR_INVALID_ARG
    assert vt.vt_paged_attn_decode_multi(**dict(base, dtype=vt.VT_E4M3)) == vt.VT_ERR_INVALID_ARG
    assert _fp8_call(True, q_len=0) == vt.VT_ERR_INVALID_ARG


def test_override_validation(lib):
    assert lib.vt_paged_attn_set_override(-1, 0) == vt.VT_ERR_INVALID_ARG
    assert lib.vt_paged_attn_set_override(0, -5) == vt.VT_ERR_INVALID_ARG
    assert lib.vt_paged_attn_set_override(0, 0) == vt.VT_OK


def test_overlap_and_segment_cost_validation(lib):
    assert lib.vt_paged_attn_set_overlap(2) == vt.VT_ERR_INVALID_ARG
    assert lib.vt_paged_attn_set_overlap(-1) == vt.VT_ERR_INVALID_ARG
    assert lib.vt_paged_attn_set_overlap(1) == vt.VT_OK
    assert lib.vt_paged_attn_set_overlap(0) == vt.VT_OK
    assert lib.vt_paged_attn_set_segment_cost(65) == vt.VT_ERR_INVALID_ARG
    for tiles in (-1, 0, 2, 64):
        assert lib.vt_paged_attn_set_segment_cost(tiles) == vt.VT_OK
    assert lib.vt_paged_attn_set_segment_cost(-1) == vt.VT_OK


def test_plan_struct_matches_header():
    """The ctypes mirror of vt_plan lists the header's fields in order."""
    text = (ROOT / "include" / "vt_paged_attn.h").read_text()
    body = text[text.index("typedef struct {", text.index("What the last successful")):text.index("} vt_plan;")]
    names = re.findall(r"^\s*(?:int|size_t)\s+(\w+);", body, re.M)
    assert names == [n for n, _ in vt.vt_plan._fields_]


def test_last_plan_before_any_launch(lib):
    p = vt.vt_plan()
    assert lib.vt_paged_attn_last_plan(None) == vt.VT_ERR_INVALID_ARG
    # this host thread has launched nothing
    assert lib.vt_paged_attn_last_plan(ctypes.byref(p)) == vt.VT_ERR_INVALID_ARG


def test_workspace_bytes_rejects_bad_shapes(lib):
    assert vt.vt_paged_attn_workspace_bytes(0, 16, 8, 128, vt.VT_BF16) == 0
    assert vt.vt_paged_attn_workspace_bytes(4, 12, 8, 128, vt.VT_BF16) == 0
    assert vt.vt_paged_attn_workspace_bytes(4, 16, 8, 96, vt.VT_BF16) == 0


def test_workspace_and_test_wait_validation(lib):
    """Arguments of the caller-owned workspace and of the wait test hook are
    checked on the host before CUDA is touched."""
    c_void = ctypes.c_void_p
    assert lib.vt_paged_attn_set_workspace(c_void(0x1000 + 16), 1 << 20, None) == vt.VT_ERR_INVALID_ARG
    assert lib.vt_paged_attn_set_workspace(c_void(0x1000), vt.VT_MIN_WORKSPACE_BYTES - 1, None) == \
        vt.VT_ERR_INVALID_ARG
    assert lib.vt_paged_attn_set_test_wait(1000, -1, 3) == vt.VT_ERR_INVALID_ARG
    assert lib.vt_paged_attn_set_test_wait(1000, 0, 3) == vt.VT_OK
    assert lib.vt_paged_attn_set_test_wait(0, -1, -1) == vt.VT_OK


def test_header_constants_match_binding():
    text = HEADER.read_text()
    assert re.search(r"#define VT_NOALLOC_SCRATCH_BYTES \(8u << 20\)", text)
    assert vt.VT_NOALLOC_SCRATCH_BYTES == 8 << 20
    assert re.search(r"#define VT_MIN_WORKSPACE_BYTES 4096u", text) and vt.VT_MIN_WORKSPACE_BYTES == 4096
