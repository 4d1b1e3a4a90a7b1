"""Plant plausible mistakes in copies of the oracle's C source and check that the pins
catch every one of them (CPU only).  The real oracle source is never modified: each
mutant is a patched copy compiled into a temporary library and exercised in a
child process."""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, original text, replacement) -- each replacement is one plausible slip.
MUTANTS = [
    ("hash_sign_dropped", "cat[half + j] = -p;", "cat[half + j] = p;"),
    ("hash_R_transposed", "Rr[(size_t)k * half + j]", "Rr[(size_t)j * d + k]"),
    ("hash_last_index_ties", "if (cat[t] > cat[best]) best = t;", "if (cat[t] >= cat[best]) best = t;"),
    ("hash_margin_wrong", "cat[best] - second", "cat[best]"),
    ("sort_positions_descending", "return x->pos < y->pos ? -1 : 1;", "return x->pos < y->pos ? 1 : -1;"),
    ("sort_bstart_off_by_one", "bstart[bucket[i] + 1] += 1;", "bstart[bucket[i]] += 1;"),
    ("attend_self_not_masked", "if (t == s) continue;", ""),
    ("attend_bucket_not_masked", "if (bucket[j] != bucket[i]) continue;", ""),
    ("attend_causal_reversed", "if (causal && !(j < i)) continue;", "if (causal && !(j > i)) continue;"),
    ("attend_no_lookback", "int lo = (k - 1) * chunk;", "int lo = k * chunk;"),
    ("attend_next_chunk_instead",
     "int lo = (k - 1) * chunk;\n    if (lo < 0) lo = 0;\n    int hi = (k + 1) * chunk;",
     "int lo = k * chunk;\n    if (lo < 0) lo = 0;\n    int hi = (k + 2) * chunk;"),
    ("attend_keys_not_normalised", "score[a] = scale * dot * inv_norm[j];", "score[a] = scale * dot;"),
    ("attend_scale_dropped", "score[a] = scale * dot * inv_norm[j];", "score[a] = dot * inv_norm[j];"),
    ("attend_lse_unshifted", "lse_sorted[s] = mx + log(sum);", "lse_sorted[s] = log(sum);"),
    ("attend_self_logit_zero", "#define ORACLE_SELF_LOGIT (-1.0e5)", "#define ORACLE_SELF_LOGIT (0.0)"),
    ("combine_uniform_weights", "double w = exp(l[r] - LSE);", "double w = 1.0 / n_rounds;"),
    ("combine_lse_is_round_max", "double LSE = mx + log(sum);", "double LSE = mx;"),
    ("combine_rows_of_round0",
     "int s = inv[(size_t)r * L + i];\n            double w",
     "int s = inv[i];\n            double w"),
    ("combine_not_unsorted",
     "int s = inv[(size_t)r * L + i];\n            double w",
     "int s = i;\n            double w"),
    ("bwd_combine_no_mean_term", "dot += gi[c] * (src[c] - oi[c]);", "dot += gi[c] * src[c];"),
    ("bwd_combine_round_weight_dropped", "go[c] += w * gi[c];", "go[c] += gi[c];"),
    ("bwd_combine_lse_grad_dropped", "g_lse_r[(size_t)r * L + s] += w * (dot + g_lse[i]);",
     "g_lse_r[(size_t)r * L + s] += w * dot;"),
    ("bwd_attend_no_mean_term", "gv += gs[c] * (vj[c] - os[c]);", "gv += gs[c] * vj[c];"),
    ("bwd_attend_query_scale_dropped", "dq[(size_t)i * d + c] += ds * scale * kj[c] * inv_norm[j];",
     "dq[(size_t)i * d + c] += ds * kj[c] * inv_norm[j];"),
    ("bwd_attend_key_grad_transposed", "dkhat[(size_t)j * d + c] += ds * scale * qi[c];",
     "dkhat[(size_t)i * d + c] += ds * scale * kj[c];"),
    ("bwd_attend_dv_at_query", "dv[(size_t)j * d + c] += p * gs[c];", "dv[(size_t)i * d + c] += p * gs[c];"),
    ("bwd_attend_self_row_dropped", "for (int c = 0; c < d; ++c) dv[(size_t)i * d + c] += gs[c];", ""),
    ("inv_norm_unguarded", "inv_norm[j] = s > 0.0 ? 1.0 / sqrt(s) : 0.0;", "inv_norm[j] = 1.0 / sqrt(s);"),
    ("bwd_key_norm_jacobian_dropped", "inv_norm[j] * (g[c] - x[c] * inv_norm[j] * proj)",
     "inv_norm[j] * g[c]"),
    ("knn_duplicates_kept", "if (seen[j] != q) { seen[j] = q; all[n_all++] = j; }",
     "all[n_all++] = j;"),
    ("knn_causal_window", "L, chunk, 0,\n                                      s, cand);",
     "L, chunk, 1,\n                                      s, cand);"),
    ("knn_query_norm_dropped", "return dot * inv_norm[i] * inv_norm[j];", "return dot * inv_norm[j];"),
    ("knn_ties_to_larger_index", "(sim[t] == sim[b] && idx[t] < idx[b])", "(sim[t] == sim[b] && idx[t] > idx[b])"),
    ("knn_first_round_only", "for (int r = 0; r < n_rounds; ++r) {\n            int s = inv[(size_t)r * L + i];\n            int n = oracle_candidates(",
     "for (int r = 0; r < 1; ++r) {\n            int s = inv[(size_t)r * L + i];\n            int n = oracle_candidates("),
    ("exact_knn_keeps_self", "if (j == i) continue;\n            all[n] = j;", "all[n] = j;"),
]

RUNNER = r"""
import sys, traceback
sys.path.insert(0, {root!r})
import oracle
from tests import pins
orc = oracle.Oracle({lib!r})
for pin in pins.ALL_PINS:
    try:
        pin(orc)
    except Exception:
        print("CAUGHT_BY", pin.__name__)
        sys.exit(0)
print("SURVIVED")
"""


def test_mutant_table_applies():
    with open(oracle._SRC) as f:
        src = f.read()
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, name


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(mutant):
    name, old, new = mutant
    with open(oracle._SRC) as f:
        src = f.read()
    with tempfile.TemporaryDirectory() as tmp:
        c = os.path.join(tmp, "mutant.c")
        so = os.path.join(tmp, "libmutant.so")
        with open(c, "w") as f:
            f.write(src.replace(old, new))
        oracle.compile_source(c, so)
        res = subprocess.run([sys.executable, "-c", RUNNER.format(root=ROOT, lib=so)],
                             capture_output=True, text=True, timeout=300)
    # a crash of the child is also a detection; a clean run of every pin is not
    assert "SURVIVED" not in res.stdout, f"{name}: no pin failed"
    assert res.returncode != 0 or "CAUGHT_BY" in res.stdout, res.stderr[-2000:]
