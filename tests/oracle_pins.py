"""Pins for the CPU oracle: facts fixed by mathematics or by the pages, not by
the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with:
  * a library routine (torch's fp64 scaled_dot_product_attention on dense,
    contiguous K/V with its own GQA expansion),
  * a closed form (one token returns it; equal scores give the mean; window 1
    returns the last token; two tokens give a logistic blend; a hand-worked
    fixture under tests/golden/),
  * an invariance (physical page order, block size, splitting query heads),
  * the bfloat16 and FP8 E4M3 formats (codes whose values are fixed by the
    format; torch's float8_e4m3fn as an independent decoder).
``test_oracle.py`` runs them on the real oracle and ``test_oracle_mutants.py``
runs them on deliberately broken copies to show each plausible mistake is
caught by at least one of them.
"""
from __future__ import annotations

import json
import math
from pathlib import Path

import numpy as np
import torch
import torch.nn.functional as F

GOLDEN = Path(__file__).resolve().parent / "golden"
STRADDLE_CONTEXTS = (1, 31, 32, 33, 64, 100, 685, 1000)


# ----------------------------------------------------------------------------
# Layout helpers (no attention arithmetic): dense per-sequence K/V -> paged pool
# ----------------------------------------------------------------------------
def paginate(dense_k, dense_v, block_size, rng, num_blocks=None, pad_pages=3):
    """Scatter dense per-sequence K/V (lists of [L_b][Hkv][D] arrays) into a
    shuffled page pool.  Returns (k_cache, v_cache, block_tables, context_lens).
    Unused pool pages and in-page tails hold NaN."""
    lens = [k.shape[0] for k in dense_k]
    pages = [(L + block_size - 1) // block_size for L in lens]
    hkv, d = dense_k[0].shape[1], dense_k[0].shape[2]
    used = sum(pages)
    nb = num_blocks if num_blocks is not None else used + pad_pages
    perm = rng.permutation(nb)
    dtype = dense_k[0].dtype
    # NaN: bf16 bits, E4M3 code, float
    fill = 0x7FC0 if dtype == np.uint16 else (0x7F if dtype == np.uint8 else np.nan)
    k_cache = np.full((nb, block_size, hkv, d), fill, dtype=dtype)
    v_cache = np.full((nb, block_size, hkv, d), fill, dtype=dtype)
    maxb = max(max(pages), 1)
    bt = np.full((len(lens), maxb), perm[-1], dtype=np.int32)
    pos = 0
    for b, L in enumerate(lens):
        for t in range(L):
            page = perm[pos + t // block_size]
            k_cache[page, t % block_size] = dense_k[b][t]
            v_cache[page, t % block_size] = dense_v[b][t]
        bt[b, :pages[b]] = perm[pos:pos + pages[b]]
        pos += pages[b]
    return k_cache, v_cache, bt, np.asarray(lens, dtype=np.int32)


def sdpa_reference(q, dense_k, dense_v, scale, window=0):
    """torch fp64 scaled_dot_product_attention per sequence; q is [B][Hq][D]."""
    out = np.zeros(q.shape, dtype=np.float64)
    for b in range(q.shape[0]):
        L = dense_k[b].shape[0]
        if L == 0:
            continue
        qq = torch.from_numpy(np.asarray(q[b], dtype=np.float64))[None, :, None, :]
        kk = torch.from_numpy(np.asarray(dense_k[b], dtype=np.float64)).permute(1, 0, 2)[None]
        vv = torch.from_numpy(np.asarray(dense_v[b], dtype=np.float64)).permute(1, 0, 2)[None]
        mask = torch.ones((1, 1, 1, L), dtype=torch.bool)
        if window > 0 and L > window:
            mask[..., : L - window] = False
        o = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale,
                                           enable_gqa=True)
        out[b] = o[0, :, 0, :].numpy()
    return out


def _rand(rng, shape, kind):
    x = rng.standard_normal(shape)
    if kind == "f64":
        return x
    if kind == "f32":
        return x.astype(np.float32)
    # bf16: round float32 draws to bfloat16 with torch (RNE), keep the bits
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def widen(a):
    """Exact float64 value of oracle storage (uint16 = bf16 bits)."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    return a.astype(np.float64)


def _case(rng, lens, hq, hkv, d, kind):
    q = _rand(rng, (len(lens), hq, d), kind)
    dk = [_rand(rng, (L, hkv, d), kind) for L in lens]
    dv = [_rand(rng, (L, hkv, d), kind) for L in lens]
    return q, dk, dv


def _check_against_sdpa(oracle, rng, lens, hq, hkv, d, block_size, kind, window, tol):
    q, dk, dv = _case(rng, lens, hq, hkv, d, kind)
    kc, vc, bt, cl = paginate(dk, dv, block_size, rng)
    scale = 1.0 / math.sqrt(d)
    got = oracle.decode(q, kc, vc, bt, cl, scale, window)
    want = sdpa_reference(widen(q), [widen(k) for k in dk], [widen(v) for v in dv], scale, window)
    err = np.abs(got - want).max()
    assert err <= tol, f"oracle vs SDPA max |err| {err:.3e} (lens {lens}, g {hq // hkv}, W {window})"


# ----------------------------------------------------------------------------
# Pins
# ----------------------------------------------------------------------------
def pin_sdpa_small_shapes(oracle):
    """Brute force on dense K/V for tiny shapes, several GQA groups, block sizes
    and windows (fp64 storage)."""
    rng = np.random.default_rng(11)
    for hq, hkv in ((4, 4), (4, 2), (8, 2), (6, 3)):
        for block_size in (1, 4, 32):
            for window in (0, 1, 3, 7):
                _check_against_sdpa(oracle, rng, [1, 5, 9, 13], hq, hkv, 8, block_size,
                                    "f64", window, 1e-12)


def pin_sdpa_straddle_contexts(oracle):
    """Contexts straddling the 32-token page boundary (the list the head_dim-128
    decode PR's numerics table uses), head_dim 128, bf16 storage."""
    rng = np.random.default_rng(12)
    _check_against_sdpa(oracle, rng, list(STRADDLE_CONTEXTS), 4, 2, 128, 32, "bf16", 0, 1e-12)
    _check_against_sdpa(oracle, rng, list(STRADDLE_CONTEXTS), 4, 2, 128, 32, "bf16", 40, 1e-12)


def pin_sdpa_fp32_storage_d256(oracle):
    rng = np.random.default_rng(13)
    _check_against_sdpa(oracle, rng, [1, 33, 70], 8, 2, 256, 32, "f32", 0, 1e-12)
    _check_against_sdpa(oracle, rng, [1, 33, 70], 8, 2, 256, 32, "f32", 17, 1e-12)


def pin_sdpa_head_dim_64(oracle):
    """The head_dim 64 shape (the library's third arm): bf16 and fp32 storage,
    a window, GQA 4, against brute force."""
    rng = np.random.default_rng(23)
    _check_against_sdpa(oracle, rng, [1, 31, 33, 100], 8, 2, 64, 32, "bf16", 0, 1e-12)
    _check_against_sdpa(oracle, rng, [1, 31, 33, 100], 8, 2, 64, 32, "f32", 45, 1e-12)


def pin_sdpa_head_dim_512(oracle):
    """head_dim 512 (the widest arm the pages' kernels cover): bf16 storage,
    GQA 4, contexts across page boundaries, with and without a window,
    against brute force."""
    rng = np.random.default_rng(32)
    _check_against_sdpa(oracle, rng, [1, 31, 33, 70], 8, 2, 512, 32, "bf16", 0, 1e-12)
    _check_against_sdpa(oracle, rng, [1, 31, 33, 70], 8, 2, 512, 32, "bf16", 40, 1e-12)


def _e4m3_value(codes):
    """Values of E4M3 codes by torch's float8_e4m3fn (independent of the oracle)."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _e4m3_encode(x):
    """Nearest E4M3 codes of values within +-448 (torch's conversion)."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pin_e4m3_every_code(oracle):
    """A one-token context returns V exactly, so V holding all 256 E4M3 codes
    reads back each code's value: torch's decoder, and the format's closed
    forms (1, 2, 0.5, the largest 448, the smallest subnormal 2^-9, the
    smallest normal 2^-6, NaN for S.1111.111)."""
    D = 256
    q = np.zeros((1, 1, D))
    k = np.zeros((1, 32, 1, D), dtype=np.uint8)
    v = np.zeros((1, 32, 1, D), dtype=np.uint8)
    v[0, 0, 0] = np.arange(256, dtype=np.uint8)
    out = oracle.decode_rows_e4m3([(0, 0)], q, k, v, [1.0], [1.0], np.zeros((1, 1), np.int32),
                                  np.array([1], np.int32), 1.0)[0]
    want = _e4m3_value(np.arange(256))
    assert np.array_equal(np.isnan(out), np.isnan(want))
    assert np.array_equal(out[~np.isnan(out)], want[~np.isnan(want)])
    closed = {0x38: 1.0, 0x40: 2.0, 0x30: 0.5, 0x7E: 448.0, 0x01: 2.0 ** -9, 0x08: 2.0 ** -6,
              0x07: 7 * 2.0 ** -9, 0x78: 256.0, 0xB8: -1.0, 0xFE: -448.0, 0x00: 0.0}
    for c, val in closed.items():
        assert out[c] == val, (hex(c), out[c], val)
    assert np.isnan(out[0x7F]) and np.isnan(out[0xFF])


def _e4m3_case(rng, lens, hq, hkv, d):
    """bf16 queries; K/V drawn N(0,1), quantised per kv head so the largest
    magnitude maps to 448; returns codes, scales and the dequantised values."""
    q = _rand(rng, (len(lens), hq, d), "bf16")
    dk = [rng.standard_normal((L, hkv, d)) for L in lens]
    dv = [rng.standard_normal((L, hkv, d)) for L in lens]
    ks = np.array([max(np.abs(x[:, h]).max() for x in dk) / 448.0 for h in range(hkv)])
    vs = np.array([max(np.abs(x[:, h]).max() for x in dv) / 448.0 for h in range(hkv)])
    ck = [_e4m3_encode(x / ks[None, :, None]) for x in dk]
    cv = [_e4m3_encode(x / vs[None, :, None]) for x in dv]
    deq_k = [_e4m3_value(c) * ks[None, :, None] for c in ck]
    deq_v = [_e4m3_value(c) * vs[None, :, None] for c in cv]
    return q, ck, cv, ks, vs, deq_k, deq_v


def pin_e4m3_kv_against_sdpa(oracle):
    """FP8 (E4M3) KV cache with per-head scales: brute force on the
    dequantised K/V (code value times its head's scale), with and without a
    window, at GQA 4."""
    rng = np.random.default_rng(24)
    lens, hq, hkv, d = [1, 33, 70, 5], 8, 2, 64
    q, ck, cv, ks, vs, deq_k, deq_v = _e4m3_case(rng, lens, hq, hkv, d)
    kc, vc, bt, cl = paginate(ck, cv, 32, rng)
    rows = [(b, i) for b in range(len(lens)) for i in range(hq)]
    scale = 1.0 / math.sqrt(d)
    for window in (0, 20):
        got = oracle.decode_rows_e4m3(rows, q, kc, vc, ks, vs, bt, cl, scale, window)
        want = sdpa_reference(widen(q), deq_k, deq_v, scale, window).reshape(-1, d)
        err = np.abs(got - want).max()
        assert err <= 1e-12, f"E4M3 oracle vs SDPA max |err| {err:.3e} (W {window})"


def pin_e4m3_scales_act_per_head(oracle):
    """Doubling one kv head's value scale doubles exactly its query heads'
    rows and leaves the others; doubling a key scale equals doubling the
    softmax scale for that head's rows."""
    rng = np.random.default_rng(25)
    lens, hq, hkv, d = [9, 40], 4, 2, 32
    q, ck, cv, ks, vs, _, _ = _e4m3_case(rng, lens, hq, hkv, d)
    kc, vc, bt, cl = paginate(ck, cv, 32, rng)
    rows = [(b, i) for b in range(len(lens)) for i in range(hq)]
    base = oracle.decode_rows_e4m3(rows, q, kc, vc, ks, vs, bt, cl, 0.2)
    vs2 = vs.copy()
    vs2[1] *= 2
    doubled = oracle.decode_rows_e4m3(rows, q, kc, vc, ks, vs2, bt, cl, 0.2)
    for r, (b, i) in enumerate(rows):
        factor = 2.0 if i // (hq // hkv) == 1 else 1.0
        assert np.array_equal(doubled[r], base[r] * factor)
    ks2 = ks * 2
    got = oracle.decode_rows_e4m3(rows, q, kc, vc, ks2, vs, bt, cl, 0.2)
    want = oracle.decode_rows_e4m3(rows, q, kc, vc, ks, vs, bt, cl, 0.4)
    assert np.abs(got - want).max() <= 1e-15


def pin_context_one_returns_v(oracle):
    """softmax over one key is 1: the row is that token's value, bit for bit."""
    rng = np.random.default_rng(14)
    for kind in ("bf16", "f32", "f64"):
        q, dk, dv = _case(rng, [1, 1], 4, 2, 16, kind)
        kc, vc, bt, cl = paginate(dk, dv, 32, rng)
        got = oracle.decode(q, kc, vc, bt, cl, 0.25, 0)
        for b in range(2):
            for i in range(4):
                assert np.array_equal(got[b, i], widen(dv[b])[0, i // 2]), (kind, b, i)


def pin_equal_scores_give_mean(oracle):
    """q = 0 (or scale = 0) makes every score 0: the row is the mean of the
    window's values."""
    rng = np.random.default_rng(15)
    lens = [3, 32, 45]
    _, dk, dv = _case(rng, lens, 4, 2, 16, "f64")
    kc, vc, bt, cl = paginate(dk, dv, 32, rng)
    for window in (0, 10):
        for q, scale in ((np.zeros((3, 4, 16)), 0.5), (rng.standard_normal((3, 4, 16)), 0.0)):
            got = oracle.decode(q, kc, vc, bt, cl, scale, window)
            for b, L in enumerate(lens):
                t0 = max(0, L - window) if window > 0 else 0
                mean = dv[b][t0:L].mean(axis=0)
                for i in range(4):
                    np.testing.assert_allclose(got[b, i], mean[i // 2], rtol=0, atol=1e-14)


def pin_window_one_returns_last(oracle):
    rng = np.random.default_rng(16)
    lens = [1, 2, 32, 33, 77]
    q, dk, dv = _case(rng, lens, 4, 2, 16, "bf16")
    kc, vc, bt, cl = paginate(dk, dv, 32, rng)
    got = oracle.decode(q, kc, vc, bt, cl, 0.25, 1)
    for b, L in enumerate(lens):
        for i in range(4):
            assert np.array_equal(got[b, i], widen(dv[b])[L - 1, i // 2]), (b, i)


def pin_window_covering_context_is_no_window(oracle):
    rng = np.random.default_rng(17)
    lens = [5, 32, 64, 100]
    q, dk, dv = _case(rng, lens, 4, 2, 16, "bf16")
    kc, vc, bt, cl = paginate(dk, dv, 32, rng)
    full = oracle.decode(q, kc, vc, bt, cl, 0.25, 0)
    for window in (100, 101, 1 << 20):
        assert np.array_equal(oracle.decode(q, kc, vc, bt, cl, 0.25, window), full)


def pin_window_is_truncated_sequence(oracle):
    """Window W over a context of L equals the plain problem over the last W
    tokens laid out as a fresh sequence (in other pages)."""
    rng = np.random.default_rng(18)
    lens = [40, 70, 129]
    q, dk, dv = _case(rng, lens, 4, 2, 16, "bf16")
    kc, vc, bt, cl = paginate(dk, dv, 32, rng)
    for window in (1, 31, 32, 33, 64):
        got = oracle.decode(q, kc, vc, bt, cl, 0.25, window)
        tk = [k[-window:] for k in dk]
        tv = [v[-window:] for v in dv]
        kc2, vc2, bt2, cl2 = paginate(tk, tv, 32, rng)
        want = oracle.decode(q, kc2, vc2, bt2, cl2, 0.25, 0)
        assert np.array_equal(got, want), window


def pin_page_permutation_invariance(oracle):
    """Where the pages sit in the pool (and hence the table's ids) must not
    change a single bit of the output."""
    rng = np.random.default_rng(19)
    lens = list(STRADDLE_CONTEXTS[:6])
    q, dk, dv = _case(rng, lens, 4, 2, 32, "bf16")
    outs = []
    for seed in (1, 2, 3):
        kc, vc, bt, cl = paginate(dk, dv, 32, np.random.default_rng(seed), pad_pages=9)
        outs.append(oracle.decode(q, kc, vc, bt, cl, 0.2, 0))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def pin_block_size_invariance(oracle):
    """The same token sequence paged with 1-, 8- and 32-token pages gives the
    same bits."""
    rng = np.random.default_rng(20)
    lens = [1, 9, 40]
    q, dk, dv = _case(rng, lens, 4, 2, 16, "f32")
    outs = []
    for bs in (1, 8, 32):
        kc, vc, bt, cl = paginate(dk, dv, bs, rng)
        outs.append(oracle.decode(q, kc, vc, bt, cl, 0.3, 0))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def pin_gqa_value_head_mapping(oracle):
    """V of kv head h is the constant 2**h: every query head of group h must
    return exactly 2**h (weights sum to one; powers of two scale exactly)."""
    rng = np.random.default_rng(21)
    hq, hkv, d = 12, 3, 8
    lens = [7, 33]
    q, dk, _ = _case(rng, lens, hq, hkv, d, "f64")
    dv = [np.broadcast_to((2.0 ** np.arange(hkv))[None, :, None], (L, hkv, d)).copy()
          for L in lens]
    kc, vc, bt, cl = paginate(dk, dv, 32, rng)
    got = oracle.decode(q, kc, vc, bt, cl, 0.3, 0)
    for i in range(hq):
        assert np.array_equal(got[:, i], np.full((2, d), 2.0 ** (i // (hq // hkv)))), i


def pin_gqa_key_head_mapping(oracle):
    """Key head h has one dominant key, at token h; values encode the token
    index.  Query heads of group h must pick token h."""
    hq, hkv, d, L = 8, 4, 4, 6
    q = np.ones((1, hq, d))
    k = np.zeros((L, hkv, d))
    for h in range(hkv):
        k[h, h, :] = 20.0
    v = np.broadcast_to(np.arange(L, dtype=np.float64)[:, None, None], (L, hkv, d)).copy()
    kc, vc, bt, cl = paginate([k], [v], 4, np.random.default_rng(22))
    got = oracle.decode(q, kc, vc, bt, cl, 1.0, 0)
    for i in range(hq):
        np.testing.assert_allclose(got[0, i], i // (hq // hkv), rtol=0, atol=1e-9, err_msg=str(i))


def pin_two_token_logistic(oracle):
    """Two keys with scores a and b: row = v1 + (v0 - v1) / (1 + exp(b - a))."""
    a, b = 0.5, -1.25
    q = np.array([[[1.0, 0.0]]])
    k = np.array([[[a, 0.0]], [[b, 0.0]]])
    v = np.array([[[3.0, -1.0]], [[-2.0, 5.0]]])
    kc, vc, bt, cl = paginate([k], [v], 1, np.random.default_rng(23))
    got = oracle.decode(q, kc, vc, bt, cl, 1.0, 0)[0, 0]
    want = v[1, 0] + (v[0, 0] - v[1, 0]) / (1.0 + math.exp(b - a))
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)


def pin_large_scores_stay_finite(oracle):
    """Scores near 1600 overflow exp() unless the maximum is subtracted first;
    the row must equal the dominant token's value."""
    d, L = 16, 5
    q = np.full((1, 1, d), 10.0)
    k = np.zeros((L, 1, d))
    k[3, 0, :] = 10.0
    k[1, 0, :] = 9.0
    v = np.arange(L * d, dtype=np.float64).reshape(L, 1, d)
    kc, vc, bt, cl = paginate([k], [v], 2, np.random.default_rng(24))
    got = oracle.decode(q, kc, vc, bt, cl, 1.0, 0)[0, 0]
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, v[3, 0], rtol=0, atol=1e-12)


def pin_scores_scale_by_scale(oracle):
    """Doubling ``scale`` equals doubling every key."""
    rng = np.random.default_rng(25)
    q, dk, dv = _case(rng, [20], 2, 1, 8, "f64")
    kc, vc, bt, cl = paginate(dk, dv, 32, rng)
    a = oracle.decode(q, kc, vc, bt, cl, 0.5, 0)
    b = oracle.decode(q, kc * 2.0, vc, bt, cl, 0.25, 0)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)
    c = oracle.decode(q, kc, vc, bt, cl, 0.25, 0)
    assert np.abs(a - c).max() > 1e-3


def pin_decode_rows_matches_decode(oracle):
    """The row-sampling entry (what every large GPU parity check compares
    against) returns, for any list of (sequence, query head) pairs, exactly the
    rows of the whole-batch decode: pairs shuffled, repeated and out of order,
    a window, bf16 and fp32 storage, on one host thread and split over seven
    (a row count seven does not divide, so the split is uneven)."""
    rng = np.random.default_rng(30)
    hq, hkv, d = 6, 2, 16
    lens = [1, 33, 70, 5, 64]
    for kind in ("bf16", "f32"):
        q, dk, dv = _case(rng, lens, hq, hkv, d, kind)
        kc, vc, bt, cl = paginate(dk, dv, 32, rng)
        for window in (0, 20):
            full = oracle.decode(q, kc, vc, bt, cl, 0.3, window)
            pairs = [(b, i) for b in range(len(lens)) for i in range(hq)]
            order = rng.permutation(len(pairs))
            rows = [pairs[j] for j in order] + [(3, 5), (0, 0), (3, 5), (4, 1), (1, 4)]
            for threads in (1, 7):
                got = oracle.decode_rows(rows, q, kc, vc, bt, cl, 0.3, window, threads=threads)
                assert got.shape == (len(rows), d)
                for r, (b, i) in enumerate(rows):
                    assert np.array_equal(got[r], full[b, i]), (kind, window, threads, r, b, i)


def pin_e4m3_rows_over_threads(oracle):
    """The FP8 row-sampling entry gives each (sequence, query head) the same
    bits whether the rows run on one host thread, are split over seven, or
    are asked for one at a time (pairs shuffled and repeated)."""
    rng = np.random.default_rng(31)
    lens, hq, hkv, d = [1, 33, 70, 5, 40], 6, 2, 32
    q, ck, cv, ks, vs, _, _ = _e4m3_case(rng, lens, hq, hkv, d)
    kc, vc, bt, cl = paginate(ck, cv, 32, rng)
    pairs = [(b, i) for b in range(len(lens)) for i in range(hq)]
    rows = [pairs[j] for j in rng.permutation(len(pairs))] + [(2, 5), (0, 0), (2, 5)]
    one = oracle.decode_rows_e4m3(rows, q, kc, vc, ks, vs, bt, cl, 0.3, 20)
    seven = oracle.decode_rows_e4m3(rows, q, kc, vc, ks, vs, bt, cl, 0.3, 20, threads=7)
    assert np.array_equal(one, seven)
    for r, pair in enumerate(rows):
        single = oracle.decode_rows_e4m3([pair], q, kc, vc, ks, vs, bt, cl, 0.3, 20)[0]
        assert np.array_equal(one[r], single), (r, pair)


def pin_e4m3_multi_token_is_truncated_decode(oracle):
    """Several new tokens over an FP8 cache, computed as the multi-token rows
    on the cache's fp64 values (codes decoded by torch times the scales):
    new token j of a sequence with L cached tokens equals the FP8 decode of
    the same query over the first L - q_len + 1 + j tokens, with and without
    a window (the causal reading of a chunk, on the FP8 reading of a cache)."""
    rng = np.random.default_rng(41)
    lens, hq, hkv, d, q_len = [3, 33, 70, 40], 6, 2, 32, 3
    _, ck, cv, ks, vs, _, _ = _e4m3_case(rng, lens, hq, hkv, d)
    kc, vc, bt, cl = paginate(ck, cv, 32, rng)
    q = _rand(rng, (len(lens), q_len, hq, d), "bf16")
    k64 = _e4m3_value(kc) * ks[None, None, :, None]
    v64 = _e4m3_value(vc) * vs[None, None, :, None]
    rows = _all_multi_rows(len(lens), q_len, hq)
    for window in (0, 20):
        multi = oracle.decode_multi_rows(rows, widen(q), k64, v64, bt, cl, 0.25, window)
        for r, (b, j, i) in enumerate(rows):
            cl_j = cl.copy()
            cl_j[b] = cl[b] - q_len + 1 + j
            ref = oracle.decode_rows_e4m3([(b, i)], np.ascontiguousarray(q[:, j]), kc, vc, ks, vs, bt, cl_j, 0.25,
                                          window)[0]
            assert np.allclose(multi[r], ref, rtol=0, atol=1e-12), (window, b, j, i)


def _multi_case(rng, lens, q_len, hq, hkv, d, kind, block_size):
    q = _rand(rng, (len(lens), q_len, hq, d), kind)
    dk = [_rand(rng, (L, hkv, d), kind) for L in lens]
    dv = [_rand(rng, (L, hkv, d), kind) for L in lens]
    kc, vc, bt, cl = paginate(dk, dv, block_size, rng)
    return q, dk, dv, kc, vc, bt, cl


def _all_multi_rows(B, q_len, hq):
    return [(b, j, i) for b in range(B) for j in range(q_len) for i in range(hq)]


def pin_multi_token_against_sdpa(oracle):
    """Multi-token decode (q_len new tokens per sequence, the last q_len of its
    context) against brute force: torch fp64 SDPA on dense K/V with an
    explicit causal mask, new token j seeing keys t <= L - q_len + j (and,
    with a window W, t > L - q_len + j - W); several q_len, windows, GQA
    groups and page sizes."""
    rng = np.random.default_rng(33)
    for q_len, hq, hkv, d, bs, kind in ((3, 4, 2, 16, 32, "bf16"), (5, 6, 3, 8, 4, "f64"), (1, 4, 4, 8, 32, "f32"),
                                        (8, 8, 2, 128, 32, "bf16")):
        lens = [q_len, q_len + 1, 33, 70]
        q, dk, dv, kc, vc, bt, cl = _multi_case(rng, lens, q_len, hq, hkv, d, kind, bs)
        scale = 1.0 / math.sqrt(d)
        for window in (0, 2, 40):
            rows = _all_multi_rows(len(lens), q_len, hq)
            got = oracle.decode_multi_rows(rows, q, kc, vc, bt, cl, scale, window)
            want = np.zeros((len(lens), q_len, hq, d))
            for b, L in enumerate(lens):
                qq = torch.from_numpy(widen(q[b])).permute(1, 0, 2)[None]          # [1][Hq][q_len][D]
                kk = torch.from_numpy(widen(dk[b])).permute(1, 0, 2)[None]
                vv = torch.from_numpy(widen(dv[b])).permute(1, 0, 2)[None]
                pos = L - q_len + torch.arange(q_len)[:, None]                   # position of new token j
                t = torch.arange(L)[None, :]
                mask = t <= pos
                if window > 0:
                    mask &= t > pos - window
                o = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask[None, None], scale=scale,
                                                   enable_gqa=True)
                want[b] = o[0].permute(1, 0, 2).numpy()
            err = np.abs(got - want.reshape(-1, d)).max()
            assert err <= 1e-12, f"multi-token oracle vs SDPA max |err| {err:.3e} (q_len {q_len}, W {window})"


def pin_multi_token_reduces_to_decode(oracle):
    """q_len = 1 is the single-token decode, and the last new token of any
    q_len attends to the whole context exactly as the single-token decode of
    that token does (same bits)."""
    rng = np.random.default_rng(34)
    lens, hq, hkv, d = [4, 33, 70, 9], 4, 2, 16
    for q_len in (1, 4):
        q, dk, dv, kc, vc, bt, cl = _multi_case(rng, lens, q_len, hq, hkv, d, "bf16", 32)
        for window in (0, 5):
            rows = _all_multi_rows(len(lens), q_len, hq)
            got = oracle.decode_multi_rows(rows, q, kc, vc, bt, cl, 0.3, window).reshape(len(lens), q_len, hq, d)
            last = oracle.decode(np.ascontiguousarray(q[:, -1]), kc, vc, bt, cl, 0.3, window)
            assert np.array_equal(got[:, -1], last), (q_len, window)


def pin_multi_token_rejects_short_context(oracle):
    """A context shorter than the new tokens it must hold is refused."""
    from oracle import OracleError
    rng = np.random.default_rng(35)
    q, dk, dv, kc, vc, bt, cl = _multi_case(rng, [2, 5], 3, 2, 1, 8, "f64", 32)
    try:
        oracle.decode_multi_rows([(0, 0, 0)], q, kc, vc, bt, cl, 0.3, 0)
    except OracleError:
        pass
    else:
        raise AssertionError("oracle accepted a context shorter than q_len")
    oracle.decode_multi_rows([(1, 2, 1)], q, kc, vc, bt, cl, 0.3, 0)


def pin_query_heads_independent(oracle):
    """Each query head alone (Hq = Hkv = 1, its kv head's pages) gives the same
    bits as inside the full GQA problem."""
    rng = np.random.default_rng(26)
    hq, hkv, d = 6, 2, 16
    lens = [17, 40]
    q, dk, dv = _case(rng, lens, hq, hkv, d, "bf16")
    kc, vc, bt, cl = paginate(dk, dv, 32, rng)
    full = oracle.decode(q, kc, vc, bt, cl, 0.25, 0)
    for i in range(hq):
        h = i // (hq // hkv)
        one = oracle.decode(np.ascontiguousarray(q[:, i:i + 1]), np.ascontiguousarray(kc[:, :, h:h + 1]),
                            np.ascontiguousarray(vc[:, :, h:h + 1]), bt, cl, 0.25, 0)
        assert np.array_equal(one[:, 0], full[:, i]), i


def pin_hand_worked_fixture(oracle):
    fx = json.loads((GOLDEN / "hand_worked_decode.json").read_text())
    P, nb = fx["block_size"], fx["num_blocks"]
    hkv, d = fx["num_kv_heads"], fx["head_dim"]
    kc = np.full((nb, P, hkv, d), np.nan)
    vc = np.full((nb, P, hkv, d), np.nan)
    for t, (page, slot) in enumerate(fx["token_pages"]):
        kc[page, slot, 0] = fx["k_tokens"][t]
        vc[page, slot, 0] = fx["v_tokens"][t]
    q = np.asarray(fx["q"], dtype=np.float64)
    bt = np.asarray(fx["block_tables"], dtype=np.int32)
    cl = np.asarray(fx["context_lens"], dtype=np.int32)
    for window, key in ((0, "window_0"), (2, "window_2")):
        got = oracle.decode(q, kc, vc, bt, cl, fx["scale"], window)
        np.testing.assert_allclose(got, np.asarray(fx["expected"][key]), rtol=0,
                                   atol=fx["tolerance"], err_msg=key)


# bfloat16 bit patterns and the values the format assigns them.
BF16_VALUES = {0x3F80: 1.0, 0xC040: -3.0, 0x3F81: 1.0078125, 0x0001: 2.0 ** -133,
               0x7F7F: 3.3895313892515355e38, 0x8000: -0.0, 0x4049: 3.140625,
               0x3E80: 0.25, 0xBF00: -0.5}


def pin_bf16_widening(oracle):
    """One-token contexts return V exactly, so the row shows the oracle's
    reading of each stored bf16 bit pattern."""
    bits = list(BF16_VALUES)
    d = len(bits)
    v = np.asarray(bits, dtype=np.uint16).reshape(1, 1, d)
    k = np.zeros((1, 1, d), dtype=np.uint16)
    q = np.zeros((1, 1, d), dtype=np.uint16)
    kc, vc, bt, cl = paginate([k], [v], 32, np.random.default_rng(27))
    got = oracle.decode(q, kc, vc, bt, cl, 1.0, 0)[0, 0]
    for j, b in enumerate(bits):
        assert got[j] == BF16_VALUES[b], hex(b)


def pin_empty_context_is_zero_row(oracle):
    rng = np.random.default_rng(28)
    q, dk, dv = _case(rng, [5], 2, 1, 8, "f64")
    kc, vc, bt, cl = paginate(dk, dv, 32, rng)
    bt2 = np.concatenate([bt, bt])
    cl2 = np.asarray([0, 5], dtype=np.int32)
    q2 = np.concatenate([q, q])
    got = oracle.decode(q2, kc, vc, bt2, cl2, 0.3, 0)
    assert np.array_equal(got[0], np.zeros((2, 8)))
    assert np.array_equal(got[1], oracle.decode(q, kc, vc, bt, cl, 0.3, 0)[0])


def pin_rejects_bad_inputs(oracle):
    from oracle import OracleError
    rng = np.random.default_rng(29)
    q, dk, dv = _case(rng, [40], 2, 1, 8, "f64")
    kc, vc, bt, cl = paginate(dk, dv, 32, rng)
    for bad_bt, bad_cl in ((bt, np.asarray([-1], np.int32)),
                           (bt, np.asarray([bt.shape[1] * 32 + 1], np.int32)),
                           (np.where(bt >= 0, kc.shape[0], bt).astype(np.int32), cl),
                           (np.full_like(bt, -1), cl)):
        for call in (lambda: oracle.decode(q, kc, vc, bad_bt, bad_cl, 0.3, 0),
                     lambda: oracle.decode_rows([(0, 0), (0, 1)], q, kc, vc, bad_bt, bad_cl, 0.3, 0, threads=2)):
            try:
                call()
            except OracleError:
                continue
            raise AssertionError("oracle accepted an invalid input")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
