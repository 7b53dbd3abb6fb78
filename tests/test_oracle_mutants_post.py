"""Mutation test of the pins of the oracle's post-verify step and emitted-token
law: plant one plausible mistake at a time in a copy of the oracle function
(on the CPU), and require that at least one pin rejects it."""
import inspect

import numpy as np
import pytest

import oracle
import test_oracle_commit as tc
import test_oracle_law as tl

COMMIT_PINS = [lambda: [tc.test_golden_cases(i) for i in range(len(tc._golden()[1]))],
               tc.test_list_formulation_random, tc.test_aimd_trajectory,
               tc.test_aimd_decrease_in_single_precision]
LAW_PINS = [lambda: tl.test_law_equals_target_law(1.0, 0, 1.0),
            lambda: tl.test_law_equals_target_law(0.9, 30, 0.9),
            tl.test_law_sums_to_one_and_beta_is_the_acceptance_rate, tl.test_special_cases]

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
    for pin in (COMMIT_PINS if fn == "commit" else LAW_PINS):
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            caught = True
            break
    assert caught, f"mutant {fn}/{mut} passed every pin"
