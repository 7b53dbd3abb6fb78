"""Mutation test of the pins of the oracle's post-verify step, emitted-token
law and draft cascade: plant one plausible mistake at a time in a copy of the oracle function
(on the CPU), and require that at least one pin rejects it."""
import inspect

import numpy as np
import pytest

import oracle
import test_oracle_cascade as tk
import test_oracle_commit as tc
import test_oracle_law as tl

COMMIT_PINS = [lambda: [tc.test_golden_cases(i) for i in range(len(tc._golden()[1]))],
               tc.test_list_formulation_random, tc.test_aimd_trajectory,
               tc.test_aimd_decrease_in_single_precision]
LAW_PINS = [lambda: tl.test_law_equals_target_law(1.0, 0, 1.0),
            lambda: tl.test_law_equals_target_law(0.9, 30, 0.9),
            tl.test_law_sums_to_one_and_beta_is_the_acceptance_rate, tl.test_special_cases]

CASCADE_PINS = [lambda: [tk.test_exact_law_by_enumeration(n) for n in sorted(tk.CASES)],
                tk.test_greedy_closed_form, tk.test_single_stage_is_the_verify_step,
                tk.test_identical_levels_accept_everything,
                tk.test_disjoint_smallest_level_rejects_at_slot_zero,
                tk.test_error_rows_and_ragged_gamma, tk.test_chi_square_per_slot]
PINS = {"commit": COMMIT_PINS, "law": LAW_PINS, "cascade": CASCADE_PINS}

MUTANTS = {
    "commit": {
        "one_draft_too_many": [("drafts[b, :a]]", "drafts[b, :a + 1]]")],
        "next_token_dropped": [("+ [t]", "+ []")],
        "kv_counts_the_new_token": [("kv[b] = min(L + a, L + len(kept))",
                                     "kv[b] = min(L + a + 1, L + len(kept))")],
        "aimd_branches_swapped": [("if valid and a == gc:", "if not (valid and a == gc):")],
        "aimd_decrease_rounds_up": [("int(np.floor(np.float32(gc) * np.float32(dec)))",
                                     "int(np.ceil(np.float32(gc) * np.float32(dec)))")],
        "error_rows_appended": [("0 <= a <= g and t >= 0 and L >= 0", "0 <= a <= g and L >= 0")],
        "capacity_ignored": [("kept = new_tokens[:room]", "kept = new_tokens")],
    },
    "law": {
        "beta_from_max": [("beta = float(np.minimum(p, q).sum())",
                           "beta = float(np.maximum(p, q).sum())")],
        "residual_sign": [("max(p[x] - q[x], 0.0)", "max(q[x] - p[x], 0.0)")],
        "rejection_weight_dropped": [("ps += (1.0 - beta) * max", "ps += 1.0 * max")],
        "accept_term_uses_p": [("ps = min(p[x], q[x])", "ps = p[x]")],
    },
    "cascade": {
        "resample_not_presented": [("tok[rows[rej], a[rej]] = t[rej]",
                                    "tok[rows[rej], a[rej]] = tok[rows[rej], a[rej]]")],
        "presented_count_not_cut": [("n[rej] = a[rej] + 1", "n[rej] = n[rej]")],
        "bonus_kept_at_every_stage": [("& (~resampled) & last", "& (~resampled)")],
        "bonus_kept_after_resample": [("& (~resampled) & last", "& last")],
        "smallest_law_at_every_stage": [("draft = levels[s][:, :gm]", "draft = levels[L][:, :gm]")],
        "every_stage_against_target": [("verify(levels[s - 1]", "verify(levels[0]")],
        "stages_top_down": [("        s = L - k\n", "        s = k + 1\n")],
        "uniforms_shared_by_stages": [("uniforms[k], temperature", "uniforms[0], temperature")],
    },
}


def _mutant(name, edits):
    src = inspect.getsource(getattr(oracle, name))
    for old, new in edits:
        assert src.count(old) == 1, f"mutation site not unique or missing: {old!r}"
        src = src.replace(old, new)
    ns = dict(vars(oracle))
    exec(compile(src, f"<mutant {name}>", "exec"), ns)
    return ns[name]


@pytest.mark.parametrize("fn,mut", [(f, m) for f in MUTANTS for m in MUTANTS[f]])
def test_mutant_is_caught(fn, mut, monkeypatch):
    monkeypatch.setattr(oracle, fn, _mutant(fn, MUTANTS[fn][mut]))
    caught = False
    for pin in PINS[fn]:
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            caught = True
            break
    assert caught, f"mutant {fn}/{mut} passed every pin"
