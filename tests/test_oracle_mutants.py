"""Plants plausible mistakes in a copy of the oracle (on the CPU) and checks
that at least one pin fails for every one of them, while the unmodified copy
passes them all.  Each variant runs in its own process, so a mistake that
reads out of bounds and crashes also counts as caught."""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))

# (name, text in the oracle source, replacement)
MUTANTS = [
    ("interleaved_head_map", "const int h = hq / G;", "const int h = hq % sh->num_kv_heads;"),
    ("dropped_scale", "s[t - lo] = scale * dot;", "s[t - lo] = dot;"),
    ("window_off_by_one", "*lo = (window > 0 && L > window) ? L - window : 0;",
     "*lo = (window > 0 && L > window) ? L - window + 1 : 0;"),
    ("wrong_slot", "int64_t slot = t % sh->page_size;",
     "int64_t slot = (t + 1) % sh->page_size;"),
    ("no_normalisation", "for (int d = 0; d < D; ++d) out[d] /= Z;", ""),
    ("scores_from_v", "const uint16_t* k = kv_row(sh, k_pages, page_table, b, t, h);\n    double dot = 0.0;\n    for (int d = 0; d < D; ++d) dot += H[qrow[d]] * H[k[d]];\n    s[t - lo]",
     "const uint16_t* k = kv_row(sh, v_pages, page_table, b, t, h);\n    double dot = 0.0;\n    for (int d = 0; d < D; ++d) dot += H[qrow[d]] * H[k[d]];\n    s[t - lo]"),
    ("max_not_subtracted", "double w = exp(s[t - lo] - m);", "double w = exp(s[t - lo]);"),
    ("head_stride_swapped", "int64_t off = (((int64_t)phys * sh->page_size + slot) * sh->num_kv_heads + h) * sh->head_dim;",
     "int64_t off = (((int64_t)phys * sh->num_kv_heads + h) * sh->page_size + slot) * sh->head_dim;"),
    ("subnormal_exponent", "mag = ldexp((double)f, -24);", "mag = ldexp((double)f, -25);"),
    ("merge_ignores_shift", "double c = exp(m[i] - M);", "double c = 1.0;"),
    ("partial_max_unscaled", "if (scale * dot > m) m = scale * dot;", "if (dot > m) m = dot;"),
    ("row_batch_index", "const int b = row / sh->num_q_heads;", "const int b = row % sh->batch;"),
    ("multi_causal_off_by_one", "int32_t len_t = (L < 0 || L > cap) ? -1 : (int32_t)(L - T + t + 1);",
     "int32_t len_t = (L < 0 || L > cap) ? -1 : (int32_t)(L - T + t);"),
    ("multi_query_row_stride", "int st = one_row(&one, q + ((int64_t)b * T + t) * sh->num_q_heads * D,",
     "int st = one_row(&one, q + ((int64_t)t * sh->batch + b) * sh->num_q_heads * D,"),
    ("bf16_exponent_bias", "mag = ldexp(128.0 + (double)f, e - 134);",
     "mag = ldexp(128.0 + (double)f, e - 135);"),
    ("append_wrong_slot", "(((int64_t)phys * sh->page_size + t % sh->page_size) * sh->num_kv_heads + h) *",
     "(((int64_t)phys * sh->page_size + (t + 1) % sh->page_size) * sh->num_kv_heads + h) *"),
    ("append_no_bound_check", "      if (t >= cap) {\n        err = 1;\n      } else {",
     "      if (0) {\n        err = 1;\n      } else {"),
]


def _run(src_text, tmp_path, name):
    d = tmp_path / name
    d.mkdir()
    (d / "variant.c").write_text(src_text)
    lib = d / "libvariant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-pthread", str(d / "variant.c"), "-o", str(lib), "-lm"], check=True)
    return subprocess.run([sys.executable, os.path.join(HERE, "oracle_pins.py"), str(lib)],
                          capture_output=True, text=True, timeout=300)


def test_unmodified_copy_passes(tmp_path):
    r = _run(oracle.source_text(), tmp_path, "control")
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    r = _run(src.replace(old, new), tmp_path, name)
    assert r.returncode != 0, f"no pin caught {name}: {r.stdout}"
