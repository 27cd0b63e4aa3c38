"""Planted mistakes in a COPY of the oracle must fail its pins (CPU only).

Each case edits one line of a temporary copy of oracle/oracle.c (or, where named,
of the oracle's Python wrapper: a padded-layout gather) (a sign, an
index, a dropped term, a transposed operand, an unreset position, an unstable
order), rebuilds that copy, and runs tests/test_oracle_pins.py against it in a
subprocess.  The committed oracle is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "rope_sign": ("out[ib] = b * c + a * s;", "out[ib] = b * c - a * s;"),
    "rope_frequency": ("return (double)p * pow(theta, -2.0 * (double)j / (double)d);",
                       "return (double)p * pow(theta, -1.0 * (double)j / (double)d);"),
    "position_not_reset": ("load_rotated(P, P->q, i, h, p + S->off, S->q + p * d);",
                           "load_rotated(P, P->q, i, h, i + S->off, S->q + p * d);"),
    "qkv_query_position_unshifted": ("load_rotated(P, P->q, i, h, p + S->off, S->q + p * d);",
                                     "load_rotated(P, P->q, i, h, p, S->q + p * d);"),
    "qkv_top_left_alignment": ("const int64_t last = p + S->off;", "const int64_t last = p;"),
    "mask_off_by_one": ("for (int64_t j = 0; j <= last; ++j) z += exp(s[j] - m);",
                        "for (int64_t j = 0; j < last; ++j) z += exp(s[j] - m); z += (last == 0);"),
    "bwd_dropped_D": ("double ds = pr[j] * (dp[j] - D);", "double ds = pr[j] * dp[j];"),
    "bwd_dk_wrong_operand": ("gk[j * d + c] += P->scale * ds * S.q[p * d + c];",
                             "gk[j * d + c] += P->scale * ds * S.k[p * d + c];"),
    "label_crosses_boundary": ("if (!ignored && i + 1 < cu[r + 1])",
                               "if (!ignored && i + 1 < total)"),
    "worklist_extra_tile": ("items[4 * n + 3] = (int32_t)ceil_div(last_row, BN);",
                            "items[4 * n + 3] = (int32_t)ceil_div(last_row, BN) + (t == 0);"),
    "worklist_unstable_ties": ("if (ny >= nx) break;", "if (ny > nx) break;"),
    "rope_interleaved_pairing": ("if (interleaved) { *ia = 2 * j; *ib = 2 * j + 1; }",
                                 "if (interleaved) { *ia = j; *ib = j + 1; }"),
    "padded_rows_from_cu": ("for p, n in zip(cp[:-1], L)", "for p, n in zip(cu[:-1], L)", "__init__.py"),
    "ffd_ascending": ("order = sorted(range(len(sizes)), key=lambda i: (-sizes[i], i))",
                      "order = sorted(range(len(sizes)), key=lambda i: (sizes[i], i))", "packing.py"),
    "ffd_room_off_by_one": ("if room[b] >= s:", "if room[b] > s:", "packing.py"),
    "lpt_fullest_rank": ("r = min(range(ranks), key=lambda k: (load[k], k))",
                         "r = max(range(ranks), key=lambda k: (load[k], k))", "packing.py"),
    "gqa_interleaved_heads": ("static int32_t kv_head(const orc_problem* P, int32_t h) { return h / (P->H / P->Hkv); }",
                              "static int32_t kv_head(const orc_problem* P, int32_t h) { return h % P->Hkv; }"),
    "ce_label_logit_sign": ("row[i] = (mx + log(s)) - zy;", "row[i] = (mx + log(s)) + zy;"),
    "ce_max_not_restored": ("row[i] = (mx + log(s)) - zy;", "row[i] = log(s) - zy;"),
    "ce_counts_ignored": ("if (ok[i]) { sr += row[i]; ++nr; }", "{ sr += row[i]; ++nr; }"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new, *where = MUTATIONS[name]
    fname = where[0] if where else "oracle.c"
    for sub in ("oracle", "tests", "variable_length_causal_gb300"):
        shutil.copytree(os.path.join(ROOT, sub), tmp_path / sub,
                        ignore=shutil.ignore_patterns("*.so", "__pycache__", "lib"))
    shutil.copy(os.path.join(ROOT, "pytest.ini"), tmp_path / "pytest.ini")
    src = (tmp_path / "oracle" / fname).read_text()
    assert src.count(old) == 1, name
    (tmp_path / "oracle" / fname).write_text(src.replace(old, new))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"mutation {name} survived the pins:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout
