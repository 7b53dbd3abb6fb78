"""Pins of the oracle's multi-stage draft cascade ("CS3602_FINAL_SpeDec",
更多实现: a chain of draft models, each drafting for the next larger one)
against what the mathematics fixes, never against the cascade itself:

* exact enumeration (V <= 4, rational laws): the first emitted token follows
  the target's law p exactly, a second token is emitted with probability
  sum_x q_L(x) prod_s min(1, q_{s-1}(x) / q_s(x)) (every stage accepts the
  original draft), and then it follows p at the next slot;
* greedy closed form: the output is the target's argmax chain, as long as
  every level's argmax agrees with the drafts, plus one token;
* a single stage is the verify step (already pinned on its own);
* identical levels accept everything; a draft level with disjoint support
  rejects at slot 0;
* 2 * 10^5 rows with three draft levels: the token at each slot follows p
  there (chi-square), and only the last token can differ from the drafts.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle


def _logits(probs):
    """float32 logits whose softmax is the given law (-inf for zero)."""
    p = np.asarray([float(x) for x in probs])
    with np.errstate(divide="ignore"):
        return np.log(p).astype(np.float32)


def _cdf_points(w):
    """Interior CDF boundaries of a law (list of Fractions), in [0, 1]."""
    tot = sum(w)
    if tot == 0:
        return []
    c, out = Fraction(0), []
    for x in w:
        c += x
        out.append(c / tot)
    return out


def _cells(points):
    """Midpoints (float32) and widths of the cells of [0, 1) cut at points."""
    cuts = sorted({Fraction(0), Fraction(1)} | {x for x in points if 0 < x < 1})
    mids = [np.float32(float((a + b) / 2)) for a, b in zip(cuts, cuts[1:])]
    widths = [float(b - a) for a, b in zip(cuts, cuts[1:])]
    return mids, widths


def _slot_cells(P, Q):
    """Cells of the acceptance and draw uniforms of one stage at one slot:
    every ratio p(t)/q(t), every CDF boundary of p (bonus) and of the
    normalised residual max(0, p - q); P, Q lists of Fractions (Q may be None
    at a bonus-only slot)."""
    acc, draw = [], list(_cdf_points(P))
    if Q is not None:
        acc = [p / q for p, q in zip(P, Q) if q > 0]
        draw += _cdf_points([max(Fraction(0), p - q) for p, q in zip(P, Q)])
    return _cells(acc), _cells(draw)


def enumerate_cascade(laws, G=1):
    """Exact law of the cascade output, by enumeration of the draft token and
    of every uniform over the cells between its possible decision points.

    laws[l][i] is level l's law at slot i (lists of Fractions): G + 1 slots
    for l < L, G for the smallest level L.  Returns {output tuple: prob}."""
    L = len(laws) - 1
    V = len(laws[0][0])
    slots = []  # (stage, slot, column, cells)
    for k in range(L):
        s = L - k
        for i in range(G + 1):
            Q = laws[s][i] if i < G else None
            (am, aw), (dm, dw) = _slot_cells(laws[s - 1][i], Q)
            if i < G:
                slots.append((k, i, 0, list(zip(am, aw))))
            slots.append((k, i, 1, list(zip(dm, dw))))
    combos = list(itertools.product(*[c for *_, c in slots]))
    drafts = list(itertools.product(range(V), repeat=G))
    n = len(combos) * len(drafts)
    u = np.full((L, n, G + 1, 2), 0.5, np.float32)
    wt = np.empty(n)
    tok = np.empty((n, G), np.int32)
    r = 0
    for dr in drafts:
        wd = math.prod(float(laws[L][i][dr[i]]) for i in range(G))
        for c in combos:
            w = wd
            for (k, i, col, _), (mid, width) in zip(slots, c):
                u[k, r, i, col] = mid
                w *= width
            wt[r] = w
            tok[r] = dr
            r += 1
    lv = [np.broadcast_to(np.stack([_logits(x) for x in laws[l]])[None],
                          (n, len(laws[l]), V)) for l in range(L + 1)]
    res = oracle.cascade(lv, tok, u, 1.0)
    assert (res["row_status"] & oracle.ERROR_MASK).max() == 0
    out = {}
    for j in range(n):
        if wt[j] == 0:
            continue
        m = int(res["out_len"][j])
        key = tuple(int(x) for x in res["out_tokens"][j, :m])
        # only the last output token can differ from the drafts
        assert key[:-1] == tuple(int(x) for x in tok[j, : m - 1]), (key, tok[j])
        out[key] = out.get(key, 0.0) + wt[j]
    return out


def _fr(*xs, den=8):
    return [Fraction(x, den) for x in xs]


CASES = {
    # three levels, V = 4, eighths: target, middle, smallest
    "three_levels": [[_fr(3, 1, 4, 0), _fr(1, 2, 2, 3)],
                     [_fr(1, 4, 1, 2), _fr(2, 2, 2, 2)],
                     [_fr(2, 1, 0, 5)]],
    # the middle level puts no mass where the target does
    "middle_disjoint": [[_fr(4, 4, 0, 0), _fr(0, 1, 3, 4)],
                        [_fr(0, 0, 5, 3), _fr(1, 1, 1, 5)],
                        [_fr(2, 2, 2, 2)]],
    # four levels, V = 3
    "four_levels": [[_fr(1, 2, 1, den=4), _fr(2, 1, 1, den=4)],
                    [_fr(3, 1, 0, den=4), _fr(1, 1, 2, den=4)],
                    [_fr(1, 1, 2, den=4), _fr(0, 2, 2, den=4)],
                    [_fr(0, 3, 1, den=4)]],
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_exact_law_by_enumeration(name):
    laws = CASES[name]
    L = len(laws) - 1
    V = len(laws[0][0])
    dist = enumerate_cascade(laws, G=1)
    assert abs(sum(dist.values()) - 1.0) < 1e-12
    p0, p1 = [float(x) for x in laws[0][0]], [float(x) for x in laws[0][1]]
    first = np.zeros(V)
    second = np.zeros((V, V))
    for key, w in dist.items():
        first[key[0]] += w
        if len(key) == 2:
            second[key[0], key[1]] += w
    np.testing.assert_allclose(first, p0, rtol=0, atol=1e-12)
    # a second token: the original draft x accepted at every stage
    want_two = np.zeros(V)
    for x in range(V):
        a = float(laws[L][0][x])
        for s in range(L, 0, -1):
            q, p = laws[s][0][x], laws[s - 1][0][x]
            a *= float(min(Fraction(1), p / q)) if q > 0 else 0.0
        want_two[x] = a
    np.testing.assert_allclose(second.sum(axis=1), want_two, rtol=0, atol=1e-12)
    # ... and it follows the target's law at slot 1
    for x in range(V):
        if want_two[x] > 0:
            np.testing.assert_allclose(second[x] / want_two[x], p1, rtol=0, atol=1e-12)


def _random_levels(rng, L, B, G, V, scale=1.5, shared=False):
    shape = (1,) if shared else (B,)
    lv = [(rng.normal(size=shape + (G + 1, V)) * scale).astype(np.float32) for _ in range(L)]
    lv.append((rng.normal(size=shape + (G, V)) * scale).astype(np.float32))
    if shared:
        lv = [np.broadcast_to(x, (B,) + x.shape[1:]) for x in lv]
    return lv


def test_greedy_closed_form():
    rng = np.random.default_rng(21)
    L, B, G, V = 3, 400, 4, 5
    lv = _random_levels(rng, L, B, G, V)
    am = [np.argmax(x, axis=2) for x in lv[:L]]  # [B, G+1] per level < L
    d = am[0][:, :G].copy()
    # mostly agreeing drafts, so that long prefixes occur
    flip = rng.random((B, G)) < 0.25
    d[flip] = rng.integers(0, V, flip.sum())
    u = rng.random((L, B, G + 1, 2), dtype=np.float32)
    r = oracle.cascade(lv, d.astype(np.int32), u, 0.0)
    for b in range(B):
        agree = 0
        while agree < G and all(am[l][b, agree] == d[b, agree] for l in range(L)):
            agree += 1
        want = list(d[b, :agree]) + [int(am[0][b, agree])]
        m = int(r["out_len"][b])
        assert r["out_tokens"][b, :m].tolist() == want, (b, d[b], [a[b] for a in am])
        assert (r["out_tokens"][b, m:] == -1).all()


def test_single_stage_is_the_verify_step():
    rng = np.random.default_rng(22)
    B, G, V = 300, 3, 9
    lv = _random_levels(rng, 1, B, G, V)
    d = rng.integers(0, V, (B, G)).astype(np.int32)
    u = rng.random((1, B, G + 1, 2), dtype=np.float32)
    gam = rng.integers(0, G + 1, B).astype(np.int32)
    for T, k, p in ((1.0, 0, 1.0), (0.8, 4, 0.9), (0.0, 0, 1.0)):
        c = oracle.cascade(lv, d, u, T, k, p, gamma_per_row=gam)
        v = oracle.verify(lv[0], lv[1], d, u[0], T, k, p, gamma_per_row=gam)
        assert np.array_equal(c["stage_accepted"][0], v["accepted_len"])
        assert np.array_equal(c["row_status"], v["row_status"])
        for b in range(B):
            a = int(v["accepted_len"][b])
            want = list(d[b, :a]) + [int(v["next_token"][b])]
            assert c["out_tokens"][b, : c["out_len"][b]].tolist() == want


def test_identical_levels_accept_everything():
    rng = np.random.default_rng(23)
    B, G, V = 64, 3, 11
    z = (rng.normal(size=(B, G + 1, V)) * 2).astype(np.float32)
    lv = [z, z, z, z[:, :G]]
    d = rng.integers(0, V, (B, G)).astype(np.int32)
    u = rng.random((3, B, G + 1, 2), dtype=np.float32)
    r = oracle.cascade(lv, d, u, 1.0)
    assert (r["out_len"] == G + 1).all()
    assert np.array_equal(r["out_tokens"][:, :G], d)
    assert (r["stage_accepted"] == G).all()
    # the bonus is level 0's draw at slot G with the last stage's uniform
    v = oracle.verify(z, z[:, :G], d, u[2], 1.0)
    assert np.array_equal(r["out_tokens"][:, G], v["next_token"])


def test_disjoint_smallest_level_rejects_at_slot_zero():
    rng = np.random.default_rng(24)
    B, G, V = 64, 3, 8
    lv = _random_levels(rng, 2, B, G, V)
    lv[0][:, :, V // 2:] = -np.inf   # target and middle level on tokens < V/2
    lv[1][:, :, V // 2:] = -np.inf
    lv[2][:, :, : V // 2] = -np.inf  # smallest level on tokens >= V/2
    d = rng.integers(V // 2, V, (B, G)).astype(np.int32)
    u = rng.random((2, B, G + 1, 2), dtype=np.float32)
    r = oracle.cascade(lv, d, u, 1.0)
    assert (r["stage_accepted"][0] == 0).all()
    assert (r["out_len"] == 1).all()
    assert (r["out_tokens"][:, 0] < V // 2).all()


def test_error_rows_and_ragged_gamma():
    rng = np.random.default_rng(25)
    B, G, V = 40, 3, 7
    lv = _random_levels(rng, 2, B, G, V)
    d = rng.integers(0, V, (B, G)).astype(np.int32)
    gam = rng.integers(0, G + 1, B).astype(np.int32)
    d[3, 0] = V          # bad token: stage 0 error
    lv[0][5, 0, 2] = np.nan  # bad target logit, read at stage 1
    gam[7] = G + 1       # bad gamma
    u = rng.random((2, B, G + 1, 2), dtype=np.float32)
    r = oracle.cascade(lv, d, u, 1.0, gamma_per_row=gam)
    for b in (3, 5, 7):
        assert r["out_len"][b] == 0 and (r["out_tokens"][b] == -1).all()
        assert r["row_status"][b] & oracle.ERROR_MASK
    assert r["stage_accepted"][1, 3] == -1  # no stage after the error
    ok = np.setdiff1d(np.arange(B), [3, 5, 7])
    assert (r["out_len"][ok] >= 1).all() and (r["out_len"][ok] <= gam[ok] + 1).all()
    # gamma_b = 0: the target's own draw at slot 0 (every stage passes it on)
    z = np.nonzero(gam[ok] == 0)[0]
    assert (r["out_len"][ok][z] == 1).all()


def test_chi_square_per_slot():
    rng = np.random.default_rng(26)
    L, N, G, V = 3, 200_000, 3, 10
    lv = _random_levels(rng, L, N, G, V, shared=True)
    laws = [[scipy.special.softmax(lv[l][0, i].astype(np.float64)) for i in range(lv[l].shape[1])]
            for l in range(L + 1)]
    d = np.stack([rng.choice(V, size=N, p=laws[L][i]) for i in range(G)], axis=1).astype(np.int32)
    u = rng.random((L, N, G + 1, 2), dtype=np.float32)
    r = oracle.cascade(lv, d, u, 1.0, threads=4)
    m = r["out_len"]
    assert (m >= 1).all()
    for b in range(0, N, 97):  # only the last token can differ from the drafts
        assert np.array_equal(r["out_tokens"][b, : m[b] - 1], d[b, : m[b] - 1])
    for i in range(G + 1):
        x = r["out_tokens"][m > i, i]
        obs = np.bincount(x, minlength=V)
        exp = laws[0][i] * len(x)
        keep = exp >= 5
        stat = ((obs[keep] - exp[keep]) ** 2 / exp[keep]).sum()
        pval = scipy.stats.chi2.sf(stat, keep.sum() - 1)
        assert pval > 1e-3, (i, len(x), pval)
    # P(len = G + 1): the original drafts accepted at every stage
    a = np.ones(N)
    for s in range(L, 0, -1):
        for i in range(G):
            q, p = laws[s][i][d[:, i]], laws[s - 1][i][d[:, i]]
            a *= np.minimum(1.0, p / q)
    want = a.mean()   # given the drafts, the acceptance coins are independent
    got = float(np.mean(m == G + 1))
    assert abs(got - want) < 5 * math.sqrt(want * (1 - want) / N), (got, want)
