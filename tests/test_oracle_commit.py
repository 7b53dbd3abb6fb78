"""Pins of the oracle's post-verify step (token bookkeeping and the AIMD
draft-length controller) against hand-derived cases and against the plain
list formulation: the new sequence is the old one, then the accepted drafts,
then the next token, cut at the capacity."""
import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden():
    g = json.load(open(os.path.join(HERE, "golden", "commit.json")))
    return g, g["cases"]


@pytest.mark.parametrize("ci", range(len(_golden()[1])))
def test_golden_cases(ci):
    g, cases = _golden()
    c = cases[ci]
    gm = max(len(x["drafts"]) for x in cases)
    drafts = np.zeros((1, gm), np.int32)
    drafts[0, : len(c["drafts"])] = c["drafts"]
    r = oracle.commit([c["accepted_len"]], [c["next_token"]], drafts,
                      np.array([c["seq"]], np.int32), [c["seq_len"]], g["seq_capacity"],
                      gamma_per_row=[c["gamma"]], aimd=tuple(g["aimd"]))
    assert r["seq"][0].tolist() == c["want_seq"], c["why"]
    assert int(r["seq_len"][0]) == c["want_len"], c["why"]
    assert int(r["kv_len"][0]) == c["want_kv"], c["why"]
    assert int(r["gamma_next"][0]) == c["want_gamma"], c["why"]


def test_list_formulation_random():
    rng = np.random.default_rng(5)
    B, gm, cap = 300, 6, 20
    drafts = rng.integers(0, 1000, size=(B, gm)).astype(np.int32)
    gam = rng.integers(0, gm + 1, size=B)
    acc = np.array([rng.integers(0, g + 1) for g in gam])
    nxt = rng.integers(0, 1000, size=B)
    nxt[::7] = -1  # error rows
    L = rng.integers(0, cap + 1, size=B)
    seq = rng.integers(0, 1000, size=(B, cap)).astype(np.int32)
    r = oracle.commit(acc, nxt, drafts, seq, L, cap, gamma_per_row=gam)
    for b in range(B):
        before = seq[b].tolist()
        if nxt[b] < 0:
            assert r["seq"][b].tolist() == before and r["seq_len"][b] == L[b]
            assert r["kv_len"][b] == L[b]
            continue
        want = (before[: L[b]] + drafts[b, : acc[b]].tolist() + [int(nxt[b])])[:cap]
        n = len(want)
        assert r["seq_len"][b] == n
        assert r["seq"][b, :n].tolist() == want
        assert r["seq"][b, n:].tolist() == before[n:]  # untouched beyond the new length
        assert r["kv_len"][b] == min(L[b] + acc[b], n)
        assert r["kv_len"][b] <= r["seq_len"][b]


def test_aimd_trajectory():
    # additive increase by 2 on full acceptance, halving (floor) on a rejection
    aimd = (1, 10, 2, 0.5)
    g, got = 4, []
    for full in [True, True, False, False, True, False, False, False, True]:
        acc = g if full else max(0, g - 1)
        r = oracle.commit([acc], [5], np.zeros((1, 16), np.int32), np.zeros((1, 64), np.int32),
                          [0], 64, gamma_per_row=[g], aimd=aimd)
        g = int(r["gamma_next"][0])
        got.append(g)
    assert got == [6, 8, 4, 2, 4, 2, 1, 1, 3]


def test_aimd_decrease_in_single_precision():
    # floor(g * d) with the product rounded to float32: 7 * 0.7 = 4.9 -> 4;
    # a factor of 1 keeps gamma; a factor of 0 drops to gamma_min
    for g, d, want in [(7, 0.7, 4), (5, 1.0, 5), (5, 0.0, 0), (3, 0.34, 1)]:
        r = oracle.commit([0], [1], np.zeros((1, 8), np.int32), np.zeros((1, 8), np.int32),
                          [0], 8, gamma_per_row=[g], aimd=(0, 8, 1, d))
        assert int(r["gamma_next"][0]) == want, (g, d)
