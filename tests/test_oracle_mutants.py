"""Mutation test of the oracle's pins: plant one plausible mistake at a time
in a copy of the oracle's C source (on the CPU, in a temporary directory),
build it, and require that at least one pin rejects it.  A mutant that every
pin accepts would mean the pins cannot see that kind of error."""
import os
import shutil
import tempfile

import pytest

import oracle
from pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "spec_oracle.c")

MUTANTS = {
    "ratio_q_over_p": [("const double ratio = px / qx;", "const double ratio = qx / px;")],
    "accept_inverted": [("accept = u0 < ratio;", "accept = u0 > ratio;")],
    "acceptance_uses_draw_uniform": [("const double u0 = (double)u_i[0];",
                                      "const double u0 = (double)u_i[1];")],
    "residual_sign_q_minus_p": [("const double d = s->p[v] - s->q[v];",
                                 "const double d = s->q[v] - s->p[v];")],
    "residual_argmax_not_sampled": [
        ("int32_t tok = draw_icdf(s->w, V, (double)u_i[1], &dg->cdf_margin);",
         "int32_t tok = argmax_first(s->w, V); dg->cdf_margin = 1.0;")],
    "draw_uses_acceptance_uniform": [
        ("int32_t tok = draw_icdf(s->w, V, (double)u_i[1], &dg->cdf_margin);",
         "int32_t tok = draw_icdf(s->w, V, (double)u_i[0], &dg->cdf_margin);")],
    "topk_off_by_one": [("if (k_on) tau = srt[top_k - 1].z;", "if (k_on) tau = srt[top_k].z;")],
    "threshold_drops_ties": [("if (!(z[v] >= tau)) e[v] = 0.0;", "if (!(z[v] > tau)) e[v] = 0.0;")],
    "topp_not_renormalised": [("for (int32_t v = 0; v < V; ++v) prob[v] = e[v] / Z;",
                               "for (int32_t v = 0; v < V; ++v) prob[v] = e[v] / Zk;")],
    "topp_stops_one_group_late": [("      if (M / Zk >= top_p) {", "      if (M_prev / Zk >= top_p) {")],
    "temperature_multiplies": [("const double tmax = zmax / T;", "const double tmax = zmax * T;"),
                               ("exp(z[v] / T - tmax)", "exp(z[v] * T - tmax)")],
    "cdf_boundary_le": [("    if (target < C) {", "    if (target <= C) {")],
    "greedy_last_of_ties": [("if (z[v] > z[best]) best = v;", "if (z[v] >= z[best]) best = v;")],
    "q_zero_always_rejects": [("accept = px > 0.0;", "accept = 0;")],
    "accepted_len_off_by_one": [("    *acc_out = i;\n    *next_out = tok;",
                                 "    *acc_out = i + 1;\n    *next_out = tok;")],
    "bonus_uses_acceptance_uniform": [
        ("const int32_t tok = draw_icdf(s->p, V, (double)u_i[1], &dg->cdf_margin);",
         "const int32_t tok = draw_icdf(s->p, V, (double)u_i[0], &dg->cdf_margin);")],
}


@pytest.fixture(scope="module")
def tmpdir_mod():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", list(MUTANTS))
def test_mutant_is_caught(name, tmpdir_mod):
    src = open(SRC).read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation site not unique or missing: {old!r}"
        src = src.replace(old, new)
    path = os.path.join(tmpdir_mod, f"{name}.c")
    open(path, "w").write(src)
    lib = oracle.build(force=True, src=path, out=os.path.join(tmpdir_mod, f"lib{name}.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin_name, pin in PINS.items():
        try:
            pin(orc)
        except (AssertionError, IndexError, ValueError) as e:
            caught.append(pin_name)
            break
    assert caught, f"mutant {name} passed every pin"
