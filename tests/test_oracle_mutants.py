"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each one.

Every mutant is a one-line edit of ``oracle/pkd_oracle.c`` in a scratch copy (never the
oracle itself): a wrong GQA head map, an off-by-one window, a dropped max-subtraction, a
wrong lse, a soft cap without the division, swapped strides, a wrong kv-length rule, an
unweighted merge, a missing v_scale, wrong fp16 / e4m3 decoders, and for several query tokens
per request a causal limit one past the query, reversed token positions and token-major rows,
for the positional encodings a reversed RoPE rotation, a rope_scale that multiplies and an
ALiBi bias of the wrong sign and the wrong half of
the 2m-head slope set for head counts that are not a power of two, and an MLA logit without its rope (kpe) part.  The pin suite in
``test_oracle_pins.py`` runs against each mutant and must fail.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "gqa_head_map": ("const int h = g / group;", "const int h = g % p->num_kv_heads;"),
    "window_off_by_one": ("first = pos - p->window_left;", "first = pos + 1 - p->window_left;"),
    "causal_limit_past_query": ("if (t_end > pos + 1) t_end = pos + 1;",
                                "if (t_end > pos + 2) t_end = pos + 2;"),
    "query_tokens_reversed": ("const int64_t pos = n - p->q_len + j;",
                              "const int64_t pos = n - 1 - j;"),
    "rope_rotation_reversed": ("x[i] = x0 * c - x1 * s;", "x[i] = x0 * c + x1 * s;"),
    "rope_scale_multiplies": ("const double a = (pos / rope_scale)", "const double a = (pos * rope_scale)"),
    "alibi_distance_sign": ("slope * (double)(t - pos)", "slope * (double)(pos - t)"),
    "alibi_other_heads_take_even_entries": ("-4.0 * (2 * (g - m) + 1) / m",
                                            "-4.0 * (2 * (g - m) + 2) / m"),
    "mla_rope_part_dropped": ("dot += load_elem(q_pe, w * dp + d, q_dtype) * load_elem(kpe, row * dp + d, kv_dtype);",
                              "dot += 0.0;"),
    "query_rows_token_major": ("(((int64_t)i * p->q_len + j) * p->num_qo_heads + g) * D",
                               "(((int64_t)j * p->batch + i) * p->num_qo_heads + g) * D"),
    "lse_without_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "soft_cap_no_division": ("tanh(x / p->logits_soft_cap)", "tanh(x)"),
    "slot_head_strides_swapped": ("slot * p->slot_stride + (int64_t)h * p->head_stride",
                                  "slot * p->head_stride + (int64_t)h * p->slot_stride"),
    "kv_len_rule": ("(int64_t)page_size * (pages - 1) + last_page_len[i]",
                    "(int64_t)page_size * pages + last_page_len[i] - page_size - 1"),
    "merge_unweighted": ("const double w = exp(lse_parts[c] - M);", "const double w = 1.0;"),
    "v_scale_dropped": ("w * p->v_scale * load_elem", "w * load_elem"),
    "f16_exponent_bias": ("ldexp(1024.0 + (double)m, e - 25)",
                          "ldexp(1024.0 + (double)m, e - 24)"),
    "e4m3_subnormal": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "pkd_oracle.c")).read()
    assert src.count(before) == 1, f"mutation site for {name} not found"
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    (tmp_path / "oracle" / "pkd_oracle.c").write_text(src.replace(before, after))
    shutil.copytree(os.path.join(ROOT, "tests"), tmp_path / "tests",
                    ignore=shutil.ignore_patterns("__pycache__"))
    shutil.copy(os.path.join(ROOT, "workloads.py"), tmp_path / "workloads.py")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
