"""The pins catch plausible mistakes in the oracle (CPU only).

Each case plants one mistake in a copy of oracle.c (a wrong constant, a
dropped term, a flipped sign or comparison, a wrong index or draw), compiles
the copy with the oracle's own flags, runs the oracle's Python functions on
it, and requires that at least one pin of tests/test_oracle_*.py fails.
The unchanged source must pass every pin of the same battery.  Mistakes are
planted only in the CPU oracle, never in the CUDA library.
"""
import os

import pytest

import oracle
import test_oracle_fit as fit
import test_oracle_philox as px
import test_oracle_rowstats as rs
import test_oracle_verify as vf

# Pins, cheapest first: a mutant stops at the first one that fails.
BATTERY = [
    ("philox known answers", px.test_philox_known_answers),
    ("uniform counter mapping", px.test_uniform_mapping_matches_block_function),
    ("uniform range and grid", px.test_uniform_range_and_grid),
    ("row stats vs logsumexp", lambda: rs.test_row_stats_match_logsumexp(1000, 0.37, 4.0)),
    ("row stats ties", rs.test_row_stats_fp32_and_ties),
    ("row stats non-finite", rs.test_row_stats_nonfinite),
    ("feature is logit(q_max)", lambda: rs.test_feature_is_logit_of_qmax(100, 1)),
    ("feature clamp", rs.test_feature_clamp),
    ("confidence closed forms", rs.test_conf_closed_forms),
    ("kept length", rs.test_kept_len_survival),
    ("av_score row by row", rs.test_av_score_matches_row_by_row),
    ("greedy argmax matching", vf.test_greedy_is_argmax_matching),
    ("acceptance tie", vf.test_acceptance_tie_is_a_rejection),
    ("cdf tie", vf.test_cdf_tie_picks_the_next_token),
    ("q(d) = 0 accepts", vf.test_zero_draft_probability_accepts),
    ("output layout", vf.test_output_layout_and_margins_tiny),
    ("kept_len 0", vf.test_kept_len_zero_emits_plain_decode_token),
    ("error flags", vf.test_error_flags),
    ("temperature on both rows", vf.test_temperature_is_applied_to_both_rows),
    ("label eligibility", fit.test_label_eligibility_counts),
    ("gradient/Hessian finite differences", fit.test_gradient_and_hessian_by_finite_differences),
    ("Newton step = dense solve", fit.test_newton_delta_equals_dense_solve),
    ("unlabelled intercepts kept", fit.test_positions_without_labels_keep_their_intercept),
    ("no labels no update", fit.test_no_labels_no_update),
    ("round pooling", fit.test_round_accumulation_equals_pooled_data),
    ("damping", lambda: fit.test_damping_scales_the_step(10.0)),
    ("recovers known parameters", fit.test_recovers_known_parameters),
    ("footnote example", vf.test_footnote_two_token_example),
    ("draft == target", vf.test_draft_equal_target_always_accepts),
    ("exact enumeration V=8 K=2", lambda: vf.test_exact_enumeration_v8(2)),
    ("closed form tokens per verify", vf.test_tokens_per_verify_closed_form),
]

# (name, text in oracle.c, replacement): one plausible mistake each.
MUTANTS = [
    ("philox round multiplier", "prod_a = (uint64_t)0xD2511F53u", "prod_a = (uint64_t)0xD2511F35u"),
    ("philox key not bumped", "k1 = k1 + 0xBB67AE85u;", "k1 = k1 + 0u;"),
    ("philox words swapped", "y1 = (uint32_t)(prod_b & 0xffffffffu);", "y1 = (uint32_t)(prod_a & 0xffffffffu);"),
    ("uniform keeps 23 bits", "(out[draw % 4u] >> 8)", "(out[draw % 4u] >> 9)"),
    ("uniform counter words swapped", "ctr[0] = b; ctr[1] = pos;", "ctr[0] = pos; ctr[1] = b;"),
    ("argmax takes the last tie", "if (y > m) { m = y; arg = v; }", "if (y >= m) { m = y; arg = v; }"),
    ("E keeps the max", "if (v != arg) E += t;", "E += t;"),
    ("ln S from E", "st->lnS = log(S);", "st->lnS = log(E);"),
    ("feature sign", "x = -log(E);", "x = log(E);"),
    ("sigmoid sign", "exp(-(omega * x + beta))", "exp(omega * x + beta)"),
    ("survival threshold strict", "if (surv >= threshold) kept = i + 1;", "if (surv > threshold) kept = i + 1;"),
    ("draft rows at tau = 1", "orc_row_stats(drow0 + (size_t)i * rowb, dtype, V, tau, &dst[i]);",
     "orc_row_stats(drow0 + (size_t)i * rowb, dtype, V, 1.0, &dst[i]);"),
    ("acceptance u <= ratio", "accept = u < ratio;", "accept = u <= ratio;"),
    ("ratio inverted", "else ratio = exp(lp - lq);", "else ratio = exp(lq - lp);"),
    ("q(d) = 0 rejects", "if (lq == -INFINITY) ratio = INFINITY;", "if (lq == -INFINITY) ratio = 0.0;"),
    ("residual sign", "double x = p - q;", "double x = q - p;"),
    ("draw reuses the acceptance uniform", "orc_uniform(seed, sid, (uint32_t)a, 1u)",
     "orc_uniform(seed, sid, (uint32_t)a, 0u)"),
    ("cdf C(v) >= uR", "if (C > T) { tok = v; break; }", "if (C >= T) { tok = v; break; }"),
    ("greedy token from the previous row", "tok = tst[a].argmax;", "tok = tst[a > 0 ? a - 1 : 0].argmax;"),
    ("bonus row is the last draft row", "if (a == k || !(R > 0.0)) {\n                for (v = 0; v < V; v++) r[v] = exp(row_logprob(trow, dtype, tau, &tst[a], v));",
     "if (a == k || !(R > 0.0)) {\n                for (v = 0; v < V; v++) r[v] = exp(row_logprob(trow0 + (size_t)(a > 0 ? a - 1 : 0) * rowb, dtype, tau, &tst[a > 0 ? a - 1 : 0], v));"),
    ("gradient sign", "g[1 + i] += (s - y);", "g[1 + i] += (y - s);"),
    ("Hessian weight sigma", "double w = s * (1.0 - s);", "double w = s;"),
    ("labels past the first rejection", "last = a < k ? a : a - 1;", "last = k - 1;"),
    ("damping inverted", "theta[0] -= ntot / (ntot + damping_c) * delta[0];",
     "theta[0] -= damping_c / (ntot + damping_c) * delta[0];"),
    ("slope step drops the cross term", "H[0 * D + (1 + i)] += w * x;", "H[0 * D + (1 + i)] += w;"),
]

_SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def _first_failure():
    for name, pin in BATTERY:
        try:
            pin()
        except Exception as e:  # an assertion, or an error a wrong result leads to
            return name, e
    return None


def test_unchanged_oracle_passes_the_battery():
    assert _first_failure() is None


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(_SRC).read()
    assert src.count(old) == 1, "mutation site not unique: " + name
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mutant), str(tmp_path / "liboracle_mutant.so"))
    with oracle.using_library(lib):
        caught = _first_failure()
    assert caught is not None, "no pin fails with the mistake: " + name


# ---------------------------------------------------------------------------
# The steps around verification (oracle/budget.py, post_verify.py, tts.py,
# tree.py): the same check, with the mutated module loaded in place of the
# original and the package's entry point swapped for the mutant's.
# ---------------------------------------------------------------------------
import importlib.util  # noqa: E402

import test_oracle_next as nx  # noqa: E402

PY_BATTERY = {
    "budget": [
        ("budget brute force", lambda: nx.test_budget_brute_force_over_subsets(0)),
        ("budget brute force 2", lambda: nx.test_budget_brute_force_over_subsets(1)),
        ("budget constant cost", nx.test_budget_constant_cost_keeps_everything),
        ("budget linear cost", lambda: nx.test_budget_linear_cost_closed_form(0.6, 10.0, 1.0, False)),
        ("budget ragged rows", nx.test_budget_ragged_rows_and_survival_rounding),
        ("budget tie", nx.test_budget_tie_takes_the_smallest_budget),
    ],
    "post_verify": [
        ("post-verify hand-worked", nx.test_post_verify_hand_worked_cases),
        ("post-verify cache loop", lambda: nx.test_post_verify_kv_matches_the_cheatsheet_loop(0)),
        ("post-verify flags", nx.test_post_verify_flags),
    ],
    "tts": [
        ("tts KL vs library", nx.test_tts_kl_against_library_and_identity),
        ("tts gradient by finite differences", nx.test_tts_gradient_by_finite_differences),
    ],
    "tree": [
        ("tree chain = linear", nx.test_tree_chain_equals_linear_verification),
        ("tree greedy by hand", nx.test_tree_greedy_walk_by_hand),
        ("tree lossless", lambda: nx.test_tree_walk_is_lossless(2)),
    ],
}
PY_ENTRY = {"budget": ["av_budget", "survival"], "post_verify": ["post_verify"], "tts": ["tts_signal"],
            "tree": ["verify_tree", "tree_uniform"]}

PY_MUTANTS = [
    ("budget", "ranking ascending", "cand.sort(key=lambda t: (-t[0], t[1]))", "cand.sort(key=lambda t: (t[0], t[1]))"),
    ("budget", "estimate without the requests", "run = float(n_req)", "run = 0.0"),
    ("budget", "last maximum", "ratio[n] > best)", "ratio[n] >= best)"),
    ("budget", "survival not cumulative", "run = np.float32(run * c[b, i])", "run = np.float32(c[b, i])"),
    ("budget", "draft_len ignored", "for i in range(int(kl[b]))", "for i in range(K)"),
    ("post_verify", "unaccepted drafts not shifted", "nxt[b, j] = inp[b, j + 1]", "nxt[b, j] = inp[b, j]"),
    ("post_verify", "bonus gets a cache entry", "kv[b] += (a + 1) if a < k else k", "kv[b] += a + 1"),
    ("post_verify", "history misses the last token", "for j in range(a + 1):\n            pos", "for j in range(a):\n            pos"),
    ("tts", "KL direction", "terms = np.where(p > 0, p * (lp - lq), 0.0)", "terms = np.where(q > 0, q * (lq - lp), 0.0)"),
    ("tts", "gradient sign", "grad[b, k] = w[k] * (q - p) / tb", "grad[b, k] = w[k] * (p - q) / tb"),
    ("tts", "gradient without 1/tau", "grad[b, k] = w[k] * (q - p) / tb", "grad[b, k] = w[k] * (q - p)"),
    ("tts", "weights dropped", "kl[b, k] = w[k] * np.sum(terms)", "kl[b, k] = np.sum(terms)"),
    ("tree", "no residual after a rejected child", "p = r / np.sum(r)", "p = p"),
    ("tree", "final draw on word 0", "tree_uniform(seed, key, depth, 0, 1)", "tree_uniform(seed, key, depth, 0, 0)"),
    ("tree", "ratio inverted", "ratio = np.inf if q[x] == 0 else p[x] / q[x]", "ratio = np.inf if q[x] == 0 else q[x] / p[x]"),
]


def _load_mutant(mod, source, tmp_path):
    path = tmp_path / (mod + "_mutant.py")
    path.write_text(source)
    spec = importlib.util.spec_from_file_location("oracle._mutant_" + mod, str(path),
                                                  submodule_search_locations=None)
    m = importlib.util.module_from_spec(spec)
    m.__package__ = "oracle"
    spec.loader.exec_module(m)
    return m


def _py_first_failure(mod):
    for name, pin in PY_BATTERY[mod]:
        try:
            pin()
        except Exception as e:
            return name, e
    return None


def test_unchanged_python_oracles_pass_their_battery():
    for mod in PY_BATTERY:
        assert _py_first_failure(mod) is None, mod


@pytest.mark.parametrize("mod,name,old,new", PY_MUTANTS, ids=[m[0] + ": " + m[1] for m in PY_MUTANTS])
def test_planted_mistake_in_python_oracle_is_caught(tmp_path, monkeypatch, mod, name, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), mod + ".py")).read()
    assert src.count(old) == 1, "mutation site not unique: " + name
    m = _load_mutant(mod, src.replace(old, new), tmp_path)
    for fn in PY_ENTRY[mod]:
        monkeypatch.setattr(oracle, fn, getattr(m, fn))
    assert _py_first_failure(mod) is not None, "no pin fails with the mistake: " + name
