"""Plant plausible mistakes in copies of the oracle and show the pins catch each.

Every mutant is a one-line textual change to ``oracle/paged_attn_oracle.c``,
compiled with gcc into a temporary library and run through all pins in its own
process.  A mutant survives only if every pin passes; the test fails if any
survives, or if a mutant's anchor text no longer matches the source (so this
file stays in step with the oracle).  A few more mutants change the oracle's
Python front end (the split of sampled rows over host threads) and run the
pin that covers it.  The real oracle is never modified.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys
import textwrap
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
SOURCE = ROOT / "oracle" / "paged_attn_oracle.c"

# name -> (anchor text, replacement, which occurrence: int index or "all")
MUTANTS = {
    "gqa_modulo_head": ("const int h = i / group;", "const int h = i % num_kv_heads;", 0),
    "query_row_uses_kv_head": ("((size_t)b * num_q_heads + i) * head_dim;",
                               "((size_t)b * num_q_heads + h) * head_dim;", 0),
    "window_off_by_one": ("? L - window : 0", "? L - window + 1 : 0", 0),
    "window_ignored": ("(window > 0 && L - window > 0)", "(0 && L - window > 0)", 0),
    "page_index_halved": ("+ t / block_size]", "+ (t / block_size) / 2]", 0),
    "slot_shift_in_scores": ("const int slot = (t0 + j) % block_size;",
                             "const int slot = (t0 + j + 1) % block_size;", 0),
    "slot_shift_in_values": ("const int slot = (t0 + j) % block_size;",
                             "const int slot = (t0 + j + 1) % block_size;", 1),
    "hnd_instead_of_nhd": ("(((size_t)page * block_size + slot) * num_kv_heads + h) * head_dim + d",
                           "(((size_t)page * num_kv_heads + h) * block_size + slot) * head_dim + d", 0),
    "no_max_subtraction": ("exp(s[j] - M)", "exp(s[j])", 0),
    "min_instead_of_max": ("if (s[j] > M) M = s[j];", "if (s[j] < M) M = s[j];", 0),
    "exp2_instead_of_exp": ("exp(s[j] - M)", "exp2(s[j] - M)", 0),
    "scale_dropped": ("s[j] = scale * dot;", "s[j] = dot;", 0),
    "scale_squared": ("s[j] = scale * dot;", "s[j] = scale * scale * dot;", 0),
    "no_normalisation": ("out_row[d] /= Z;", "out_row[d] /= 1.0;", 0),
    "keys_as_values": ("out_row[d] += w * element(v_cache", "out_row[d] += w * element(k_cache", 0),
    "values_as_keys": ("const double kd = element(k_cache", "const double kd = element(v_cache", 0),
    "last_token_dropped": ("const int n = L - t0;", "const int n = L - t0 - (L > t0 + 1);", 0),
    "bf16_shift_15": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 15", 0),
    "bf16_low_half": ("((uint32_t)bits) << 16", "((uint32_t)bits)", 0),
    "e4m3_bias_8": ("ldexp(1.0 + (double)man / 8.0, ex - 7)", "ldexp(1.0 + (double)man / 8.0, ex - 8)", 0),
    "e4m3_no_subnormals": ("(ex == 0) ? ldexp", "(0) ? ldexp", 0),
    "e4m3_nan_is_a_value": ("if (ex == 0xF && man == 0x7) return NAN;", "if (0) return NAN;", 0),
    "e4m3_sign_dropped": ("return sign ? -mag : mag;", "return mag;", 0),
    "value_scale_on_keys": ("num_kv_heads, head_dim)) * ks;", "num_kv_heads, head_dim)) * vs;", 0),
    "key_scale_dropped": ("num_kv_heads, head_dim)) * ks;", "num_kv_heads, head_dim));", 0),
    "value_scale_dropped": ("num_kv_heads, head_dim)) * vs;", "num_kv_heads, head_dim));", 0),
    "rows_pair_swapped": ("window, rows[2 * r],\n        rows[2 * r + 1]);", "window, rows[2 * r + 1],\n        rows[2 * r]);", 0),
    "rows_kv_pair_swapped": ("rows[2 * r], rows[2 * r + 1]);", "rows[2 * r + 1], rows[2 * r]);", 0),
    "rows_output_not_advanced": ("out + (size_t)r * head_dim, q, k_cache", "out, q, k_cache", 0),
    "multi_causal_off_by_one": ("const int32_t Lj = L - q_len + 1 + j;", "const int32_t Lj = L - q_len + j;", 0),
    "multi_causal_ignored": ("const int32_t Lj = L - q_len + 1 + j;", "const int32_t Lj = L;", 0),
    "multi_token_offset_dropped": ("((size_t)b * q_len + j) * num_q_heads", "((size_t)b * q_len) * num_q_heads", 0),
    "multi_rows_j_i_swapped": ("rows[3 * r + 1], rows[3 * r + 2]);", "rows[3 * r + 2], rows[3 * r + 1]);", 0),
    "scale_of_kv_head_zero": ("const double ks = k_scale ? k_scale[h] : 1.0;", "const double ks = k_scale ? k_scale[0] : 1.0;", 0),
}


def _mutate(src: str, anchor: str, repl: str, which) -> str:
    count = src.count(anchor)
    assert count >= 1, f"anchor {anchor!r} not in oracle source"
    if which == "all":
        return src.replace(anchor, repl)
    assert which < count, f"anchor {anchor!r} occurs {count} times"
    parts = src.split(anchor)
    return anchor.join(parts[: which + 1]) + repl + anchor.join(parts[which + 1:])


RUNNER = textwrap.dedent("""
    import json, sys
    sys.path.insert(0, {tests!r}); sys.path.insert(0, {root!r})
    import oracle
    from oracle_pins import ALL_PINS
    o = oracle.Oracle({lib!r})
    failed = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except Exception as e:
            failed.append(pin.__name__)
    print(json.dumps(failed))
""")


def test_every_mutant_is_caught(tmp_path):
    import oracle
    src = SOURCE.read_text()
    procs = {}
    for name, (anchor, repl, which) in MUTANTS.items():
        c_file = tmp_path / f"{name}.c"
        c_file.write_text(_mutate(src, anchor, repl, which))
        lib = oracle.build(c_file, tmp_path / f"lib{name}.so", force=True)
        code = RUNNER.format(tests=str(ROOT / "tests"), root=str(ROOT), lib=str(lib))
        env = dict(os.environ, OMP_NUM_THREADS="1")
        procs[name] = subprocess.Popen([sys.executable, "-c", code], stdout=subprocess.PIPE,
                                       stderr=subprocess.PIPE, text=True, env=env)
    survivors, report = [], {}
    for name, p in procs.items():
        out, err = p.communicate(timeout=600)
        if p.returncode != 0:
            report[name] = f"crashed rc={p.returncode}"
            continue
        failed = json.loads(out.strip().splitlines()[-1])
        report[name] = failed
        if not failed:
            survivors.append(name)
    assert not survivors, f"mutants not caught by any pin: {survivors}\n{report}"


def test_unmutated_copy_passes_all_pins(tmp_path):
    """Control: the same harness on an unchanged copy reports no failing pin."""
    import oracle
    c_file = tmp_path / "same.c"
    c_file.write_text(SOURCE.read_text())
    lib = oracle.build(c_file, tmp_path / "libsame.so", force=True)
    code = RUNNER.format(tests=str(ROOT / "tests"), root=str(ROOT), lib=str(lib))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, check=True)
    assert json.loads(out.stdout.strip().splitlines()[-1]) == []


# Mistakes planted in a copy of the oracle's Python front end (the host-thread
# split of the row-sampling entries), run through every pin.
PY_MUTANTS = {
    "thread_split_results_dropped": ("sub_out = out[lo:hi]", "sub_out = out[lo:hi].copy()"),
    "thread_split_rows_shifted": ("sub_rows = np.ascontiguousarray(rows[lo:hi])",
                                  "sub_rows = np.ascontiguousarray(rows[max(lo - 1, 0):hi - (lo > 0)])"),
    "thread_split_last_part_dropped": ("range(threads)))", "range(threads - 1)))"),
    "thread_split_rc_ignored": ("    for rc in rcs:\n        if rc != 0:\n            raise OracleError(ERRORS.get(rc, str(rc)))",
                                "    for rc in rcs:\n        pass"),
}

PY_RUNNER = textwrap.dedent("""
    import importlib.util, json, sys
    sys.path.insert(0, {tests!r}); sys.path.insert(0, {root!r})
    spec = importlib.util.spec_from_file_location("oracle_mut", {init!r})
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    from oracle_pins import ALL_PINS
    o = mod.Oracle({lib!r})
    failed = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except Exception:
            failed.append(pin.__name__)
    print(json.dumps(failed))
""")


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_python_front_end_mutant_is_caught(tmp_path, name):
    import oracle
    anchor, repl = PY_MUTANTS[name]
    src = (ROOT / "oracle" / "__init__.py").read_text()
    init = tmp_path / "oracle_mut.py"
    init.write_text(_mutate(src, anchor, repl, 0))
    lib = oracle.build()
    code = PY_RUNNER.format(tests=str(ROOT / "tests"), root=str(ROOT), init=str(init), lib=str(lib))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, check=True)
    assert json.loads(out.stdout.strip().splitlines()[-1]) != [], f"mutant {name} survived"
