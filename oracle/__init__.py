"""CPU reference oracle for paged decode attention (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  It compiles ``paged_attn_oracle.c`` with the
host C compiler and calls it through ctypes; it never touches the CUDA
library and the CUDA library never touches it.

What the C code computes, and which page passages it follows, is stated at the
top of ``paged_attn_oracle.c``: plain two-pass softmax attention in float64 for
one query row per head, reading K/V through the block table of 32-token NHD
pages.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SOURCE = HERE / "paged_attn_oracle.c"
BUILD_DIR = HERE / "_build"
LIBRARY = BUILD_DIR / "libpaged_attn_oracle.so"

ELEM_BF16, ELEM_F32, ELEM_F64, ELEM_E4M3 = 0, 1, 2, 3
ERRORS = {0: "ok", -1: "bad argument", -2: "bad context length",
          -3: "page id out of range", -4: "out of memory"}

_build_lock = threading.Lock()


class OracleError(RuntimeError):
    pass


def build(source: Path = SOURCE, output: Path = LIBRARY, force: bool = False) -> Path:
    """Compile the oracle into a shared library with gcc (-O2, no fast-math)."""
    source, output = Path(source), Path(output)
    with _build_lock:
        if (not force and output.exists()
                and output.stat().st_mtime >= source.stat().st_mtime):
            return output
        output.parent.mkdir(parents=True, exist_ok=True)
        tmp = output.with_suffix(f".{os.getpid()}.tmp")
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", str(source), "-o", str(tmp), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, output)
    return output


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _elem_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return ELEM_BF16
    if a.dtype == np.float32:
        return ELEM_F32
    if a.dtype == np.float64:
        return ELEM_F64
    raise TypeError(f"oracle storage must be uint16 (bf16 bits), float32 or float64, got {a.dtype}")


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, library: Path | None = None):
        path = Path(library) if library is not None else build()
        self.path = path
        self._lib = ctypes.CDLL(str(path))
        c_int, c_void, c_double = ctypes.c_int, ctypes.c_void_p, ctypes.c_double
        common = [c_void, c_void, c_void, c_int, c_void, c_void, c_int, c_int,
                  c_int, c_int, c_int, c_int, c_int, c_double, c_int]
        self._lib.oracle_decode.argtypes = [c_void] + common
        self._lib.oracle_decode.restype = c_int
        self._lib.oracle_decode_rows.argtypes = [c_void, c_void, c_int] + common
        self._lib.oracle_decode_rows.restype = c_int
        self._lib.oracle_decode_rows_kv.argtypes = [c_void, c_void, c_int, c_void, c_int, c_void, c_void, c_int,
                                                    c_void, c_void] + common[4:]
        self._lib.oracle_decode_rows_kv.restype = c_int
        self._lib.oracle_decode_multi_rows.argtypes = [c_void, c_void, c_int, c_void, c_void, c_void, c_int, c_void,
                                                       c_void, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                                       c_int, c_double, c_int]
        self._lib.oracle_decode_multi_rows.restype = c_int

    @staticmethod
    def _prepare(q, k_cache, v_cache, block_tables, context_lens):
        q = np.ascontiguousarray(q)
        k_cache = np.ascontiguousarray(k_cache)
        v_cache = np.ascontiguousarray(v_cache)
        elem = _elem_code(q)
        if _elem_code(k_cache) != elem or _elem_code(v_cache) != elem:
            raise TypeError("q, k_cache and v_cache must share one storage type")
        if q.ndim != 3 or k_cache.ndim != 4 or k_cache.shape != v_cache.shape:
            raise ValueError("q is [B][Hq][D]; k_cache and v_cache are [blocks][P][Hkv][D]")
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        return q, k_cache, v_cache, bt, cl, elem

    def decode(self, q, k_cache, v_cache, block_tables, context_lens, scale, window=0):
        """All rows, float64 [B][Hq][D]."""
        q, k_cache, v_cache, bt, cl, elem = self._prepare(q, k_cache, v_cache, block_tables, context_lens)
        B, Hq, D = q.shape
        nb, P, Hkv, D2 = k_cache.shape
        assert D2 == D and bt.shape[0] == B and cl.shape == (B,)
        out = np.zeros((B, Hq, D), dtype=np.float64)
        rc = self._lib.oracle_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), elem,
                                     _ptr(bt), _ptr(cl), B, Hq, Hkv, D, P, bt.shape[1], nb,
                                     float(scale), int(window))
        if rc != 0:
            raise OracleError(ERRORS.get(rc, str(rc)))
        return out

    def decode_rows(self, rows, q, k_cache, v_cache, block_tables, context_lens, scale,
                    window=0, threads: int = 1):
        """Selected rows [(b, i), ...] -> float64 [len(rows)][D].

        ``threads`` > 1 splits the rows over host threads (ctypes releases the
        GIL during each call); the arithmetic of every row is unchanged.
        """
        q, k_cache, v_cache, bt, cl, elem = self._prepare(q, k_cache, v_cache, block_tables, context_lens)
        B, Hq, D = q.shape
        nb, P, Hkv, _ = k_cache.shape
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        out = np.zeros((rows.shape[0], D), dtype=np.float64)

        def run(lo, hi):
            if hi <= lo:
                return 0
            sub_rows = np.ascontiguousarray(rows[lo:hi])
            sub_out = out[lo:hi]
            return self._lib.oracle_decode_rows(
                _ptr(sub_out), _ptr(sub_rows), hi - lo, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                elem, _ptr(bt), _ptr(cl), B, Hq, Hkv, D, P, bt.shape[1], nb, float(scale),
                int(window))

        _over_threads(run, rows.shape[0], threads)
        return out

    def decode_rows_e4m3(self, rows, q, k_codes, v_codes, k_scale, v_scale, block_tables,
                         context_lens, scale, window=0, threads: int = 1):
        """Selected rows of a decode over an FP8 (E4M3) KV cache: k_codes and
        v_codes are uint8 code arrays [blocks][P][Hkv][D]; element (.., h, d)
        stands for its E4M3 value times k_scale[h] (v_scale[h]).  q is bf16 bits
        (uint16), float32 or float64.  Returns float64 [len(rows)][D].
        ``threads`` splits the rows over host threads as in decode_rows."""
        q = np.ascontiguousarray(q)
        q_elem = _elem_code(q)
        k_codes = np.ascontiguousarray(k_codes, dtype=np.uint8)
        v_codes = np.ascontiguousarray(v_codes, dtype=np.uint8)
        if q.ndim != 3 or k_codes.ndim != 4 or k_codes.shape != v_codes.shape:
            raise ValueError("q is [B][Hq][D]; k_codes and v_codes are [blocks][P][Hkv][D]")
        B, Hq, D = q.shape
        nb, P, Hkv, D2 = k_codes.shape
        ks = np.ascontiguousarray(k_scale, dtype=np.float64).reshape(Hkv)
        vs = np.ascontiguousarray(v_scale, dtype=np.float64).reshape(Hkv)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        assert D2 == D and bt.shape[0] == B and cl.shape == (B,)
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        out = np.zeros((rows.shape[0], D), dtype=np.float64)

        def run(lo, hi):
            if hi <= lo:
                return 0
            sub_rows = np.ascontiguousarray(rows[lo:hi])
            sub_out = out[lo:hi]
            return self._lib.oracle_decode_rows_kv(
                _ptr(sub_out), _ptr(sub_rows), hi - lo, _ptr(q), q_elem, _ptr(k_codes), _ptr(v_codes), ELEM_E4M3,
                _ptr(ks), _ptr(vs), _ptr(bt), _ptr(cl), B, Hq, Hkv, D, P, bt.shape[1], nb, float(scale),
                int(window))

        _over_threads(run, rows.shape[0], threads)
        return out

    def decode_multi_rows(self, rows, q, k_cache, v_cache, block_tables, context_lens, scale, window=0,
                          threads: int = 1):
        """Selected rows [(b, j, i), ...] of a multi-token decode -> float64
        [len(rows)][D].  q is [B][q_len][Hq][D] (bf16 bits, float32 or
        float64); the caches, block table and context lengths as for decode;
        new token j of sequence b attends to the first
        context_lens[b] - q_len + 1 + j tokens."""
        q = np.ascontiguousarray(q)
        if q.ndim != 4:
            raise ValueError("q is [B][q_len][Hq][D]")
        B, q_len, Hq, D = q.shape
        qq, k_cache, v_cache, bt, cl, elem = self._prepare(q.reshape(B * q_len, Hq, D), k_cache, v_cache,
                                                           block_tables, context_lens)
        nb, P, Hkv, D2 = k_cache.shape
        assert D2 == D and bt.shape[0] == B and cl.shape == (B,)
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
        out = np.zeros((rows.shape[0], D), dtype=np.float64)

        def run(lo, hi):
            if hi <= lo:
                return 0
            sub_rows = np.ascontiguousarray(rows[lo:hi])
            sub_out = out[lo:hi]
            return self._lib.oracle_decode_multi_rows(
                _ptr(sub_out), _ptr(sub_rows), hi - lo, _ptr(q), _ptr(k_cache), _ptr(v_cache), elem, _ptr(bt),
                _ptr(cl), B, q_len, Hq, Hkv, D, P, bt.shape[1], nb, float(scale), int(window))

        _over_threads(run, rows.shape[0], threads)
        return out


def _over_threads(run, n: int, threads: int) -> None:
    """run(lo, hi) over [0, n) in one piece, or split into `threads` contiguous
    pieces run on host threads; raises on the first nonzero return code."""
    if threads <= 1 or n < 2:
        rcs = [run(0, n)]
    else:
        bounds = np.linspace(0, n, threads + 1).astype(int)
        with ThreadPoolExecutor(max_workers=threads) as pool:
            rcs = list(pool.map(lambda j: run(bounds[j], bounds[j + 1]), range(threads)))
    for rc in rcs:
        if rc != 0:
            raise OracleError(ERRORS.get(rc, str(rc)))


_default: Oracle | None = None


def default_oracle() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
