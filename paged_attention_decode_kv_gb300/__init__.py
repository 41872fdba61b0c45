"""GB300-native paged decode attention: Python binding of libvt_paged_attn.

The library (``_build/libvt_paged_attn.so``, built by ``build_lib.py``) does
every step of the decode on the GPU; this module only marshals arguments
through ctypes.  Functions named ``vt_*`` mirror the C entry points of
``include/vt_paged_attn.h`` one to one (pointers as Python ints); ``decode``
is a convenience wrapper that takes torch CUDA tensors.  There is no CPU
fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import threading
from pathlib import Path

LIBRARY_PATH = Path(__file__).resolve().parent / "_build" / "libvt_paged_attn.so"

(VT_OK, VT_ERR_INVALID_ARG, VT_ERR_UNSUPPORTED, VT_ERR_CUDA, VT_ERR_OOM, VT_ERR_DEVICE_TIMEOUT,
 VT_ERR_SCRATCH_LIMIT) = range(7)
VT_BF16, VT_F32, VT_E4M3 = 0, 1, 2
BLOCK_SIZE = 32

EXPORTED = ("vt_paged_attn_decode", "vt_paged_attn_decode_noalloc", "vt_paged_attn_decode_fp8",
            "vt_paged_attn_decode_multi", "vt_paged_attn_decode_multi_fp8",
            "vt_paged_attn_last_plan",
            "vt_paged_attn_set_override", "vt_paged_attn_set_overlap", "vt_paged_attn_set_segment_cost",
            "vt_paged_attn_set_workspace", "vt_paged_attn_set_test_wait",
            "vt_paged_attn_device_status", "vt_paged_attn_device_status_detail", "vt_paged_attn_workspace_bytes",
            "vt_paged_attn_release", "vt_status_string", "vt_last_cuda_error", "vt_paged_attn_version")
VT_NOALLOC_SCRATCH_BYTES = 8 << 20
VT_MIN_WORKSPACE_BYTES = 4096


class VtError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: status {status}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


class vt_plan(ctypes.Structure):
    _fields_ = [("grid_ctas", ctypes.c_int), ("ctas_per_sm", ctypes.c_int), ("num_sms", ctypes.c_int),
                ("consumer_warps", ctypes.c_int), ("tensor_cores", ctypes.c_int), ("stages", ctypes.c_int), ("group_tile", ctypes.c_int),
                ("subgroups", ctypes.c_int), ("min_units_per_cta", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("dtype", ctypes.c_int), ("smem_bytes", ctypes.c_size_t),
                ("workspace_bytes", ctypes.c_size_t), ("launch_overlap", ctypes.c_int),
                ("segment_cost", ctypes.c_int), ("scratch_source", ctypes.c_int), ("q_len", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


_lib = None
_lock = threading.Lock()


def library() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not LIBRARY_PATH.exists():
                raise RuntimeError(
                    f"{LIBRARY_PATH} is missing: build it with "
                    "`python -m paged_attention_decode_kv_gb300.build_lib` (needs nvcc)")
            lib = ctypes.CDLL(str(LIBRARY_PATH))
            c_int, c_void, c_float, c_size = ctypes.c_int, ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t
            lib.vt_paged_attn_decode.argtypes = [c_void] * 6 + [c_int] * 5 + [c_float, c_int, c_void, c_int,
                                                                               c_int, c_int]
            lib.vt_paged_attn_decode.restype = c_int
            lib.vt_paged_attn_decode_noalloc.argtypes = lib.vt_paged_attn_decode.argtypes
            lib.vt_paged_attn_decode_noalloc.restype = c_int
            lib.vt_paged_attn_decode_fp8.argtypes = [c_void] * 8 + [c_int] * 5 + [c_float, c_int, c_void, c_int,
                                                                                   c_int]
            lib.vt_paged_attn_decode_fp8.restype = c_int
            lib.vt_paged_attn_decode_multi.argtypes = [c_void] * 6 + [c_int] * 6 + [c_float, c_int, c_void, c_int,
                                                                                    c_int, c_int]
            lib.vt_paged_attn_decode_multi.restype = c_int
            lib.vt_paged_attn_decode_multi_fp8.argtypes = [c_void] * 8 + [c_int] * 6 + [c_float, c_int, c_void,
                                                                                         c_int, c_int]
            lib.vt_paged_attn_decode_multi_fp8.restype = c_int
            lib.vt_paged_attn_last_plan.argtypes = [ctypes.POINTER(vt_plan)]
            lib.vt_paged_attn_last_plan.restype = c_int
            lib.vt_paged_attn_set_override.argtypes = [c_int, c_int]
            lib.vt_paged_attn_set_override.restype = c_int
            lib.vt_paged_attn_set_overlap.argtypes = [c_int]
            lib.vt_paged_attn_set_overlap.restype = c_int
            lib.vt_paged_attn_set_segment_cost.argtypes = [c_int]
            lib.vt_paged_attn_set_segment_cost.restype = c_int
            lib.vt_paged_attn_set_workspace.argtypes = [c_void, c_size, c_void]
            lib.vt_paged_attn_set_workspace.restype = c_int
            lib.vt_paged_attn_set_test_wait.argtypes = [ctypes.c_longlong, c_int, c_int]
            lib.vt_paged_attn_set_test_wait.restype = c_int
            lib.vt_paged_attn_device_status.argtypes = [c_void, ctypes.POINTER(ctypes.c_uint)]
            lib.vt_paged_attn_device_status.restype = c_int
            lib.vt_paged_attn_device_status_detail.argtypes = [c_void, ctypes.POINTER(ctypes.c_uint), c_int]
            lib.vt_paged_attn_device_status_detail.restype = c_int
            lib.vt_paged_attn_workspace_bytes.argtypes = [c_int] * 5
            lib.vt_paged_attn_workspace_bytes.restype = c_size
            lib.vt_paged_attn_release.argtypes = []
            lib.vt_paged_attn_release.restype = None
            lib.vt_status_string.argtypes = [c_int]
            lib.vt_status_string.restype = ctypes.c_char_p
            lib.vt_last_cuda_error.argtypes = []
            lib.vt_last_cuda_error.restype = ctypes.c_char_p
            lib.vt_paged_attn_version.argtypes = []
            lib.vt_paged_attn_version.restype = c_int
            _lib = lib
    return _lib


def _check(status: int, where: str) -> None:
    if status != VT_OK:
        lib = library()
        detail = lib.vt_status_string(status).decode()
        cuda = lib.vt_last_cuda_error().decode()
        if cuda:
            detail += f"; {cuda}"
        raise VtError(status, where, detail)


# ---- C entry points, same names -------------------------------------------
def vt_paged_attn_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                         num_kv_heads, head_dim, block_size, scale, window, stream, max_blocks_per_seq,
                         num_blocks, dtype) -> int:
    """Raw call: pointers and the stream handle are ints; returns the status code."""
    return library().vt_paged_attn_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                          num_q_heads, num_kv_heads, head_dim, block_size, float(scale),
                                          int(window), stream, max_blocks_per_seq, num_blocks, dtype)


def vt_paged_attn_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_q_heads,
                                 num_kv_heads, head_dim, block_size, scale, window, stream, max_blocks_per_seq,
                                 num_blocks, dtype) -> int:
    """Raw call of the allocation-free entry point (scratch in a fixed static
    device array instead of a library allocation); returns the status code."""
    return library().vt_paged_attn_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens,
                                                  num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                                  float(scale), int(window), stream, max_blocks_per_seq,
                                                  num_blocks, dtype)


def vt_paged_attn_decode_multi(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, q_len, num_q_heads,
                               num_kv_heads, head_dim, block_size, scale, window, stream, max_blocks_per_seq,
                               num_blocks, dtype) -> int:
    """Raw call of the multi-token decode (q_len new tokens per sequence,
    causal within them); returns the status code."""
    return library().vt_paged_attn_decode_multi(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                                                q_len, num_q_heads, num_kv_heads, head_dim, block_size, float(scale),
                                                int(window), stream, max_blocks_per_seq, num_blocks, dtype)


def vt_paged_attn_decode_multi_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                                   num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, scale, window,
                                   stream, max_blocks_per_seq, num_blocks) -> int:
    """Raw call of the multi-token decode over an FP8 (E4M3) KV cache; returns
    the status code."""
    return library().vt_paged_attn_decode_multi_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                                    context_lens, num_seqs, q_len, num_q_heads, num_kv_heads,
                                                    head_dim, block_size, float(scale), int(window), stream,
                                                    max_blocks_per_seq, num_blocks)


def vt_paged_attn_decode_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, num_seqs,
                             num_q_heads, num_kv_heads, head_dim, block_size, scale, window, stream,
                             max_blocks_per_seq, num_blocks) -> int:
    """Raw call of the FP8 (E4M3) KV-cache decode; returns the status code."""
    return library().vt_paged_attn_decode_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                              context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                              block_size, float(scale), int(window), stream, max_blocks_per_seq,
                                              num_blocks)


def vt_paged_attn_last_plan() -> dict:
    p = vt_plan()
    _check(library().vt_paged_attn_last_plan(ctypes.byref(p)), "vt_paged_attn_last_plan")
    return p.as_dict()


def vt_paged_attn_set_override(grid_ctas: int = 0, min_units_per_cta: int = 0) -> None:
    """Force the CTA count and/or the minimum work per CTA (0: automatic)."""
    _check(library().vt_paged_attn_set_override(grid_ctas, min_units_per_cta), "vt_paged_attn_set_override")


def vt_paged_attn_set_overlap(enabled: bool) -> None:
    """Launch decodes as programmatic dependents of the previous kernel on the
    stream (that kernel must not write context_lens or block_tables)."""
    _check(library().vt_paged_attn_set_overlap(1 if enabled else 0), "vt_paged_attn_set_overlap")


def vt_paged_attn_set_segment_cost(tiles: int = -1) -> None:
    """Partition weight of a (sequence, kv head) boundary in tiles (-1: default, 2; 6 for FP8 or multi-token)."""
    _check(library().vt_paged_attn_set_segment_cost(tiles), "vt_paged_attn_set_segment_cost")


def vt_paged_attn_set_workspace(dev_ptr: int, nbytes: int, stream=None) -> None:
    """Use caller-owned device memory [dev_ptr, dev_ptr + nbytes) as the split
    workspace of the current device (dev_ptr 0: back to the library's own)."""
    _check(library().vt_paged_attn_set_workspace(dev_ptr or None, nbytes, _stream_handle(stream)),
           "vt_paged_attn_set_workspace")


def vt_paged_attn_set_test_wait(wait_limit_cycles: int = 0, withhold_cta: int = -1, withhold_tile: int = -1) -> None:
    """Test hook: shorten the kernel's bounded waits and make one CTA withhold
    a tile, so a wait gives up (0, -1, -1 restores normal operation)."""
    _check(library().vt_paged_attn_set_test_wait(wait_limit_cycles, withhold_cta, withhold_tile),
           "vt_paged_attn_set_test_wait")


def vt_paged_attn_device_status(stream=None) -> int:
    """Status word of bounded waits that gave up (0 = none); clears it."""
    word = ctypes.c_uint(0)
    library().vt_paged_attn_device_status(_stream_handle(stream), ctypes.byref(word))
    return int(word.value)


def vt_paged_attn_device_status_detail(stream=None, n_words: int = 5) -> list:
    """First n_words of the device status area (not cleared): status bits, then
    where the first bounded wait that gave up was (1 + CTA, bit | thread << 8,
    barrier address, parity)."""
    words = (ctypes.c_uint * n_words)()
    _check(library().vt_paged_attn_device_status_detail(_stream_handle(stream), words, n_words),
           "vt_paged_attn_device_status_detail")
    return [int(x) for x in words]


def vt_paged_attn_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, dtype) -> int:
    return int(library().vt_paged_attn_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, dtype))


def vt_paged_attn_release() -> None:
    library().vt_paged_attn_release()


def vt_status_string(status: int) -> str:
    return library().vt_status_string(status).decode()


def vt_paged_attn_version() -> int:
    return int(library().vt_paged_attn_version())


# ---- torch convenience -------------------------------------------------------
def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return VT_BF16
    if t.dtype == torch.float32:
        return VT_F32
    raise TypeError(f"storage dtype must be bfloat16 or float32, got {t.dtype}")


def decode(q, k_cache, v_cache, block_tables, context_lens, scale=None, window: int = 0, out=None,
           stream=None):
    """Decode attention for torch CUDA tensors.

    q [B][Hq][D]; k_cache, v_cache [num_blocks][32][Hkv][D]; block_tables
    [B][max_blocks] int32; context_lens [B] int32.  Returns out [B][Hq][D]
    (allocated unless given).  Asynchronous on ``stream`` (default: current).
    """
    import torch
    B, Hq, D = q.shape
    nb, P, Hkv, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache/v_cache must be [num_blocks][32][Hkv][head_dim] matching q")
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("block_tables", block_tables),
                    ("context_lens", context_lens)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise TypeError("q, k_cache and v_cache must share one dtype")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA tensor shaped and typed like q")
    if scale is None:
        scale = D ** -0.5
    st = vt_paged_attn_decode(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                              block_tables.data_ptr(), context_lens.data_ptr(), B, Hq, Hkv, D, P, scale,
                              window, _stream_handle(stream), block_tables.shape[1], nb, dtype_code(q))
    _check(st, "vt_paged_attn_decode")
    return out


def decode_fp8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens, scale=None, window: int = 0,
               out=None, stream=None):
    """Decode attention over an FP8 (E4M3) KV cache, for torch CUDA tensors.

    q [B][Hq][D] bf16, or [B][q_len][Hq][D] for several new tokens per
    sequence (vt_paged_attn_decode_multi_fp8); k_codes, v_codes
    [num_blocks][32][Hkv][D] uint8 E4M3 codes (or torch.float8_e4m3fn);
    k_scale, v_scale [Hkv] float32.  Returns out shaped like q, bf16
    (allocated unless given).  Asynchronous on ``stream``.
    """
    import torch
    if q.dim() == 4:
        B, q_len, Hq, D = q.shape
    else:
        B, Hq, D = q.shape
        q_len = 0
    if k_codes.dtype == torch.float8_e4m3fn:
        k_codes = k_codes.view(torch.uint8)
    if v_codes.dtype == torch.float8_e4m3fn:
        v_codes = v_codes.view(torch.uint8)
    nb, P, Hkv, D2 = k_codes.shape
    if D2 != D or v_codes.shape != k_codes.shape:
        raise ValueError("k_codes/v_codes must be [num_blocks][32][Hkv][head_dim] matching q")
    for name, t in (("q", q), ("k_codes", k_codes), ("v_codes", v_codes), ("k_scale", k_scale),
                    ("v_scale", v_scale), ("block_tables", block_tables), ("context_lens", context_lens)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dtype != torch.bfloat16 or k_codes.dtype != torch.uint8 or v_codes.dtype != torch.uint8:
        raise TypeError("q must be bfloat16 and the caches uint8 E4M3 codes")
    if k_scale.dtype != torch.float32 or v_scale.dtype != torch.float32 or k_scale.numel() != Hkv or \
            v_scale.numel() != Hkv:
        raise TypeError("k_scale and v_scale must be float32 [num_kv_heads]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA tensor shaped and typed like q")
    if scale is None:
        scale = D ** -0.5
    if q_len:
        st = vt_paged_attn_decode_multi_fp8(out.data_ptr(), q.data_ptr(), k_codes.data_ptr(), v_codes.data_ptr(),
                                            k_scale.data_ptr(), v_scale.data_ptr(), block_tables.data_ptr(),
                                            context_lens.data_ptr(), B, q_len, Hq, Hkv, D, P, scale, window,
                                            _stream_handle(stream), block_tables.shape[1], nb)
        _check(st, "vt_paged_attn_decode_multi_fp8")
    else:
        st = vt_paged_attn_decode_fp8(out.data_ptr(), q.data_ptr(), k_codes.data_ptr(), v_codes.data_ptr(),
                                      k_scale.data_ptr(), v_scale.data_ptr(), block_tables.data_ptr(),
                                      context_lens.data_ptr(), B, Hq, Hkv, D, P, scale, window,
                                      _stream_handle(stream), block_tables.shape[1], nb)
        _check(st, "vt_paged_attn_decode_fp8")
    return out


def decode_multi(q, k_cache, v_cache, block_tables, context_lens, scale=None, window: int = 0, out=None,
                 stream=None):
    """Multi-token decode for torch CUDA tensors: q [B][q_len][Hq][D]; the new
    tokens are the last q_len of each sequence's context_lens[b] cached tokens
    and attend causally.  Returns out [B][q_len][Hq][D]."""
    import torch
    B, q_len, Hq, D = q.shape
    nb, P, Hkv, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("k_cache/v_cache must be [num_blocks][32][Hkv][head_dim] matching q")
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("block_tables", block_tables),
                    ("context_lens", context_lens)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise TypeError("q, k_cache and v_cache must share one dtype")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA tensor shaped and typed like q")
    if scale is None:
        scale = D ** -0.5
    st = vt_paged_attn_decode_multi(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                    block_tables.data_ptr(), context_lens.data_ptr(), B, q_len, Hq, Hkv, D, P,
                                    scale, window, _stream_handle(stream), block_tables.shape[1], nb,
                                    dtype_code(q))
    _check(st, "vt_paged_attn_decode_multi")
    return out
