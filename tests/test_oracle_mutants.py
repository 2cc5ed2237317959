"""The oracle's pins must be able to fail: each case plants one plausible mistake in a copy of
the oracle source (on the CPU), builds it, and checks that at least one pin rejects it."""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins
from tests import test_oracle_verify as vpins
from tests import test_oracle_sizing as spins

SRC = os.path.join(os.path.dirname(oracle.__file__), "dh_oracle.cpp")

# (name, text in the oracle, planted replacement, pins expected to catch it)
MUTANTS = [
    ("bf16_one_bit_too_many", "std::ldexp(x, 7 - e)", "std::ldexp(x, 8 - e)",
     ["test_round_bf16_matches_brute_force_on_doubles"]),
    ("bf16_ties_away", "std::nearbyint(q)", "std::round(q)",
     ["test_round_bf16_matches_torch_on_binary32_values"]),
    ("projection_drops_last_term", "for (int i = 0; i < d; ++i)\n      acc +=",
     "for (int i = 0; i < d - 1; ++i)\n      acc +=", ["test_project_rounds_to_activation_dtype"]),
    ("projection_transposed_U", "stored_value(U, dtype, (size_t)i * r + j)",
     "stored_value(U, dtype, (size_t)j * d + i)", ["test_project_rounds_to_activation_dtype"]),
    ("scores_skip_rounding", "t[j] = round_to_dtype(acc, dtype);", "t[j] = acc;",
     ["test_topk_matches_lexsort"]),
    ("topk_ascending", "order[v] = {-s[v], v};", "order[v] = {s[v], v};",
     ["test_topk_matches_lexsort"]),
    ("rescore_wrong_row", "stored_value(W, dtype, (size_t)v * d + c)",
     "stored_value(W, dtype, (size_t)c * vocab + v)", ["test_exact_logits_match_full_head"]),
    ("softmax_sign", "sum += std::exp(z[k] - m);", "sum += std::exp(m - z[k]);",
     ["test_K_equals_vocab_reduces_to_full_softmax", "test_softmax_invariants"]),
    ("tree_compares_own_argmax", "tok[n] == a[par[n]]", "tok[n] == a[n]",
     ["test_golden_trees", "test_random_trees_against_brute_force"]),
    ("argmax_last_tie", "if (arg < 0 || x > best) { best = x; arg = v; }",
     "if (arg < 0 || x >= best) { best = x; arg = v; }", ["test_golden_trees"]),
    ("argmax_takes_nan", "if (std::isnan(x)) continue;", "",
     ["test_tree_argmax_nan_ranks_below_numbers"]),
    ("deepest_tie_highest_index", "depth[n] > depth[best]", "depth[n] >= depth[best]",
     ["test_golden_trees"]),
    ("expand_ties_by_position", "return tk[x] < tk[y];", "return x < y;",
     ["test_golden_expansions", "test_expansion_matches_lexsort"]),
    ("expand_ascending", "return p[x] > p[y];", "return p[x] < p[y];",
     ["test_golden_expansions", "test_expansion_matches_lexsort"]),
    ("expand_drops_parent", "(float)(par * (double)p[k])", "(float)((double)p[k])",
     ["test_golden_expansions", "test_expansion_matches_lexsort"]),
    ("expand_keeps_at_threshold", "if (a > min_benefit) ++keep;", "if (a >= min_benefit) ++keep;",
     ["test_golden_expansions"]),
    ("verify_residual_keeps_draft_mass", "if (v >= 0 && v < vocab) w[v] -= cand_prob[((size_t)b * L + n) * K + k];",
     "if (v >= 0 && v < vocab) w[v] -= 0.0;",
     ["vpins.test_golden_verify", "vpins.test_emitted_tokens_follow_the_target_distribution"]),
    ("verify_accept_inverted", "if (!(u < ratio)) break;", "if (u < ratio) break;",
     ["vpins.test_golden_verify", "vpins.test_emitted_tokens_follow_the_target_distribution"]),
    ("verify_ignores_temperature", "p[v] = stored_value(logits, dtype, (row0 + i) * (size_t)vocab + v) / temperature;",
     "p[v] = stored_value(logits, dtype, (row0 + i) * (size_t)vocab + v);",
     ["vpins.test_golden_verify", "vpins.test_temperature_scales_the_target"]),
    ("verify_bonus_from_last_drafted_row", "probs_of_row(L, p);", "probs_of_row(L > 0 ? L - 1 : 0, p);",
     ["vpins.test_golden_verify", "vpins.test_emitted_tokens_follow_the_target_distribution"]),
    ("verify_draft_outside_list_rejected", "if (qx <= 0.0) continue;  // ratio +inf: accepted",
     "if (qx <= 0.0) break;", ["vpins.test_golden_verify"]),
    ("sizing_keeps_at_threshold", "if (!(kids[w].a > thr)) break;", "if (!(kids[w].a >= thr)) break;",
     ["spins.test_golden_sizing"]),
    ("sizing_total_not_marginal_cost", "const float dc = c[w + 1] - c[w];", "const float dc = c[w + 1];",
     ["spins.test_golden_sizing", "spins.test_random_frontiers_against_brute_force"]),
    ("sizing_ties_to_higher_parent", "if (x.f != y.f) return x.f < y.f;", "if (x.f != y.f) return x.f > y.f;",
     ["spins.test_golden_sizing", "spins.test_random_frontiers_against_brute_force"]),
    ("sizing_first_bin_always", "if (batch <= bin_batch[i]) { bin = i; break; }", "{ bin = 0; break; }",
     ["spins.test_golden_sizing", "spins.test_random_frontiers_against_brute_force"]),
]


def _run_pin(name):
    """Run every parametrisation of one pin; return True if any of them fails."""
    mod, _, attr = name.rpartition(".")
    fn = getattr({"vpins": vpins, "spins": spins}.get(mod, pins), attr)
    marks = getattr(fn, "pytestmark", [])
    params = [m for m in marks if m.name == "parametrize"]
    if not params:
        calls = [{}]
    else:
        argname, values = params[0].args[0], params[0].args[1]
        calls = [{argname: v} for v in values]
    for kw in calls:
        try:
            fn(**kw)
        except AssertionError:
            return True
    return False


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_planted_mistake(mutant, tmp_path, monkeypatch):
    name, old, new, catchers = mutant
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique in the oracle: {old!r}"
    mut = tmp_path / "mutant.cpp"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
                    str(mut), "-o", str(lib)], check=True)
    monkeypatch.setattr(oracle, "_lib", oracle.bind(str(lib)))
    assert any(_run_pin(c) for c in catchers), f"no pin caught mutant {name}"
