"""Pins for the fp64 oracle: checks against what the pages and the mathematics
fix, never against the oracle itself.

Each pin takes an ``oracle.Oracle`` (the real build, or a mutant compiled by
the mutation test) and raises AssertionError on a mismatch.  The pins are:

* ``golden``        hand-derived cases in tests/golden (closed forms).
* ``greedy``        greedy mode == the first-argmax rule via ``np.argmax``.
* ``filters``       filtered law == brute force by full sort (``np.sort``,
                    ``np.unique``) and ``scipy.special.softmax``.
* ``law_exact``     exact enumeration at V <= 8: the output law equals p
                    ("CS3602_FINAL_SpeDec", "2. 困惑度测试(PPL)": P(x) = min(p,q)
                    + (p - min(p,q)) = p), unfiltered and filtered.
* ``identities``    residual mass = 1 - sum min(p, q); sum p = 1;
                    P(accepted_len >= i) = prod_j beta_j.
* ``special``       p == q accepts every draft; disjoint supports reject at 0
                    and resample from p; top-k 1 == greedy; u = 0; gamma_b = 0;
                    error statuses.
* ``chi_square``    10^6 draws: the first emitted token is distributed as p.
"""
from __future__ import annotations

import glob
import json
import math
import os

import numpy as np
import scipy.special
import scipy.stats

import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------- helpers
def brute_law(z, T, top_k=0, top_p=1.0):
    """Filtered tempered softmax by brute force (full sort, library softmax)."""
    z = np.asarray(z, np.float64)
    V = len(z)
    keep = np.ones(V, bool)
    if 0 < top_k < V:
        keep = z >= np.sort(z)[::-1][top_k - 1]
    w = scipy.special.softmax(np.where(keep, z / T, -np.inf))
    if top_p < 1.0:
        for v in np.unique(z[keep])[::-1]:
            if w[z >= v].sum() >= top_p:
                keep &= z >= v
                break
        w = np.where(keep, w, 0.0)
        w = w / w.sum()
    return w


def batch(target, draft, tokens, uniforms):
    return (np.ascontiguousarray(target, np.float32), np.ascontiguousarray(draft, np.float32),
            np.ascontiguousarray(tokens, np.int32), np.ascontiguousarray(uniforms, np.float32))


def midgrid(n):
    """Midpoints of n equal cells of [0, 1), as float32 (exact for n <= 2^23)."""
    return ((np.arange(n, dtype=np.float64) + 0.5) / n).astype(np.float32)


def enumerate_law(orc, zt, zd, T, top_k, top_p, G=1 << 16):
    """Output law of one verify step with gamma = 1, by enumeration.

    P(out = y) = sum_x q(x) [A(x) 1{y = x} + (1 - A(x)) R(y)]: A(x) is the
    fraction of a midpoint grid of u0 accepting x, R(y) the fraction of a
    midpoint grid of u1 drawing y at a rejection.  Only the first emitted
    token is counted (the accepted draft, or the resample)."""
    V = len(zt)
    q = brute_law(zd, T, top_k, top_p)
    g = midgrid(G)
    xs = np.repeat(np.arange(V, dtype=np.int32), G)
    u = np.zeros((V * G, 2, 2), np.float32)
    u[:, 0, 0] = np.tile(g, V)
    u[:, 0, 1] = 0.5
    u[:, 1, 1] = 0.5
    tgt = np.broadcast_to(np.stack([zt, zt]).astype(np.float32), (V * G, 2, V))
    drf = np.broadcast_to(np.asarray(zd, np.float32)[None, None], (V * G, 1, V))
    r = orc.verify(tgt, drf, xs[:, None], u, T, top_k, top_p)
    acc = (r["accepted_len"] == 1).reshape(V, G).mean(axis=1)
    # residual law: x* with the smallest ratio, u0 just below 1 forces a reject
    p = brute_law(zt, T, top_k, top_p)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(q > 0, p / np.where(q > 0, q, 1), np.inf)
    xstar = int(np.argmin(ratio))
    law = np.zeros(V)
    reject_mass = float(np.sum(q * (1 - acc)))
    if reject_mass > 0:
        assert ratio[xstar] < 1
        u2 = np.zeros((G, 2, 2), np.float32)
        u2[:, 0, 0] = np.float32(1 - 2 ** -24)
        u2[:, 0, 1] = g
        r2 = orc.verify(np.broadcast_to(tgt[:1], (G, 2, V)), np.broadcast_to(drf[:1], (G, 1, V)),
                        np.full((G, 1), xstar, np.int32), u2, T, top_k, top_p)
        assert np.all(r2["accepted_len"] == 0)
        R = np.bincount(r2["next_token"], minlength=V)[:V] / G
        law += reject_mass * R
    law += q * acc
    return law, p, q, acc


# -------------------------------------------------------------------- pins
_ENV = {"exp": math.exp, "log": math.log, "sqrt": math.sqrt, "inf": math.inf}


def _ev(x):
    """Fixture values are numbers or closed-form expressions (strings)."""
    if isinstance(x, list):
        return [_ev(e) for e in x]
    return float(eval(x, dict(_ENV))) if isinstance(x, str) else x


def pin_golden(orc):
    files = sorted(glob.glob(os.path.join(GOLDEN, "*.json")))
    assert files, "no golden fixtures"
    for f in files:
        fx = json.load(open(f))
        for c in fx.get("laws", []):
            prob, _, st = orc.distribution(np.asarray(_ev(c["logits"]), np.float32), c["T"],
                                           c.get("top_k", 0), c.get("top_p", 1.0))
            want = np.array(_ev(c["expect"]), np.float64)
            assert st == 0, (f, c)
            np.testing.assert_allclose(prob, want, rtol=0, atol=1e-7, err_msg=f"{f}: {c['name']}")
        for c in fx.get("steps", []):
            tgt = np.asarray(_ev(c["target"]), np.float32)[None]
            drf = np.asarray(_ev(c["draft"]), np.float32).reshape(1, tgt.shape[1] - 1, tgt.shape[2])
            r = orc.verify(tgt, drf, np.asarray(c["tokens"], np.int32)[None],
                           np.asarray(c["uniforms"], np.float32)[None], c["T"],
                           c.get("top_k", 0), c.get("top_p", 1.0))
            got = (int(r["accepted_len"][0]), int(r["next_token"][0]))
            want = (c["expect"]["accepted_len"], c["expect"]["next_token"])
            assert got == want, f"{f}: {c['name']}: got {got} want {want}"


def pin_greedy(orc):
    rng = np.random.default_rng(11)
    B, G, V = 200, 3, 37
    tgt = rng.integers(-4, 5, size=(B, G + 1, V)).astype(np.float32)  # many ties
    drf = rng.normal(size=(B, G, V)).astype(np.float32)
    am = np.argmax(tgt, axis=2)  # first occurrence on ties
    tok = np.where(rng.random((B, G)) < 0.7, am[:, :G], rng.integers(0, V, (B, G))).astype(np.int32)
    r = orc.verify(tgt, drf, tok, rng.random((B, G + 1, 2), dtype=np.float32), 0.0)
    for b in range(B):
        i = 0
        while i < G and am[b, i] == tok[b, i]:
            i += 1
        assert (r["accepted_len"][b], r["next_token"][b]) == (i, am[b, i]), b
    assert np.all(r["row_status"] == 0)


def pin_filters(orc):
    rng = np.random.default_rng(12)
    for trial in range(60):
        V = int(rng.integers(2, 40))
        z = (np.round(rng.normal(size=V) * 4) / 2).astype(np.float32)  # ties on a 0.5 grid
        if trial % 7 == 0:
            z[rng.integers(0, V)] = -np.inf
        T = float(rng.choice([0.3, 1.0, 2.5]))
        k = int(rng.choice([0, 1, 2, 5, V - 1, V]))
        p = float(rng.choice([1.0, 0.95, 0.5, 0.1]))
        got, _, st = orc.distribution(z, T, k, p)
        assert st == 0
        np.testing.assert_allclose(got, brute_law(z, T, k, p), rtol=0, atol=1e-12,
                                   err_msg=f"V={V} T={T} k={k} p={p}")
        assert abs(got.sum() - 1) < 1e-12


def pin_law_exact(orc):
    rng = np.random.default_rng(13)
    cases = [(8, 1.0, 0, 1.0), (5, 1.0, 0, 1.0), (8, 0.7, 0, 1.0), (8, 1.0, 3, 1.0),
             (8, 1.3, 0, 0.8), (7, 1.0, 4, 0.7)]
    for V, T, k, p in cases:
        zt = (rng.normal(size=V) * 1.5).astype(np.float32)
        zd = (rng.normal(size=V) * 1.5).astype(np.float32)
        G = 1 << 16
        law, pt, q, acc = enumerate_law(orc, zt, zd, T, k, p, G)
        # grid error: 1/G per acceptance fraction, V/G on the residual law
        np.testing.assert_allclose(law, pt, rtol=0, atol=(V + 2) / G,
                                   err_msg=f"law != p at V={V} T={T} k={k} p={p}")
        # acceptance probability of x is min(1, p/q) (to grid resolution)
        with np.errstate(divide="ignore", invalid="ignore"):
            want = np.where(q > 0, np.minimum(1, pt / np.where(q > 0, q, 1)), np.nan)
        m = q > 0
        np.testing.assert_allclose(acc[m], want[m], rtol=0, atol=1.0 / G)


def pin_identities(orc):
    rng = np.random.default_rng(14)
    # residual mass W = sum max(0, p - q) = 1 - beta, beta = sum min(p, q)
    for _ in range(20):
        V = int(rng.integers(3, 60))
        zt = rng.normal(size=V).astype(np.float32) * 2
        zd = rng.normal(size=V).astype(np.float32) * 2
        p, q = brute_law(zt, 1.0), brute_law(zd, 1.0)
        x = int(np.argmin(p / q))
        u = np.array([[[1 - 2 ** -24, 0.5], [0.5, 0.5]]], np.float32)
        r = orc.verify(np.stack([zt, zt])[None], zd[None, None], np.array([[x]]), u, 1.0)
        assert r["accepted_len"][0] == 0
        beta = np.minimum(p, q).sum()
        assert abs(r["diag"]["residual_mass"][0] - (1 - beta)) < 1e-12
        pd, qd = r["p_draft"][0, 0], r["q_draft"][0, 0]
        assert abs(pd - p[x]) < 1e-7 and abs(qd - q[x]) < 1e-7
    # P(accepted_len >= i) = prod_{j < i} beta_j with fixed logits per position
    G, V, N = 3, 12, 200_000
    zt = (rng.normal(size=(G + 1, V)) * 1.5).astype(np.float32)
    zd = (rng.normal(size=(G, V)) * 1.5).astype(np.float32)
    qs = [brute_law(zd[i], 1.0) for i in range(G)]
    ps = [brute_law(zt[i], 1.0) for i in range(G)]
    betas = np.array([np.minimum(ps[i], qs[i]).sum() for i in range(G)])
    tok = np.stack([rng.choice(V, size=N, p=qs[i]) for i in range(G)], axis=1).astype(np.int32)
    u = rng.random((N, G + 1, 2), dtype=np.float32)
    r = orc.verify(np.broadcast_to(zt, (N, G + 1, V)), np.broadcast_to(zd, (N, G, V)), tok, u, 1.0)
    acc = r["accepted_len"]
    for i in range(1, G + 1):
        want = float(np.prod(betas[:i]))
        got = float(np.mean(acc >= i))
        assert abs(got - want) < 5 * math.sqrt(want * (1 - want) / N) + 1e-9, (i, got, want)


def pin_special(orc):
    rng = np.random.default_rng(15)
    V, G, B = 20, 4, 64
    z = (rng.normal(size=(B, G + 1, V)) * 2).astype(np.float32)
    u = rng.random((B, G + 1, 2), dtype=np.float32)
    tok = rng.integers(0, V, (B, G)).astype(np.int32)
    # identical target and draft logits: p == q, every draft accepted
    r = orc.verify(z, z[:, :G], tok, u, 1.0)
    assert np.all(r["accepted_len"] == G) and np.all(r["row_status"] == 0)
    r = orc.verify(z, z[:, :G], tok, u, 0.7, 5, 0.9)
    ok = np.array([brute_law(z[b, i], 0.7, 5, 0.9)[tok[b, i]] > 0 for b in range(B) for i in range(G)])
    # tokens outside the kept set have p = q = 0 -> rejected (q(x) == 0, p(x) == 0)
    first_bad = [next((i for i in range(G) if not ok.reshape(B, G)[b, i]), G) for b in range(B)]
    assert list(r["accepted_len"]) == first_bad
    # disjoint supports: every draft rejected at 0, resample law == p (u1 grid)
    Gd = 4096
    zt = np.full(6, -np.inf, np.float32)
    zt[:3] = [0.3, -0.2, 1.0]
    zd = np.full(6, -np.inf, np.float32)
    zd[3:] = [0.1, 0.5, -1.0]
    uu = np.zeros((Gd, 2, 2), np.float32)
    uu[:, 0, 0] = midgrid(Gd)
    uu[:, 0, 1] = midgrid(Gd)[::-1]
    r = orc.verify(np.broadcast_to(np.stack([zt, zt]), (Gd, 2, 6)), np.broadcast_to(zd, (Gd, 1, 6)),
                   np.full((Gd, 1), 4, np.int32), uu, 1.0)
    assert np.all(r["accepted_len"] == 0)
    np.testing.assert_allclose(np.bincount(r["next_token"], minlength=6) / Gd, brute_law(zt, 1.0),
                               atol=2.0 / Gd)
    # top-k = 1 gives the greedy tokens when the maximum is unique
    zc = rng.normal(size=(B, G + 1, V)).astype(np.float32)
    am = np.argmax(zc, axis=2).astype(np.int32)
    tk = np.where(rng.random((B, G)) < 0.6, am[:, :G], tok).astype(np.int32)
    r1 = orc.verify(zc, zc[:, :G] + 1, tk, u, 1.0, 1)
    r0 = orc.verify(zc, zc[:, :G] + 1, tk, u, 0.0)
    assert np.array_equal(r1["accepted_len"], r0["accepted_len"])
    assert np.array_equal(r1["next_token"], r0["next_token"])
    # u = 0: accept iff p(x) > 0; the draw takes the first token of positive weight
    zt = np.array([-np.inf, 1.0, 0.0, 2.0], np.float32)
    zd = np.array([0.0, 3.0, 0.0, 0.0], np.float32)
    u0 = np.zeros((1, 2, 2), np.float32)
    r = orc.verify(np.stack([zt, zt])[None], zd[None, None], np.array([[0]]), u0, 1.0)
    assert (r["accepted_len"][0], r["next_token"][0]) == (0, 2)  # p(0) = 0; residual {2, 3}
    r = orc.verify(np.stack([zt, zt])[None], zd[None, None], np.array([[1]]), u0, 1.0)
    assert (r["accepted_len"][0], r["next_token"][0]) == (1, 1)  # accepted; bonus u=0 -> 1
    # gamma_b = 0: the bonus draw from target row 0
    gam = np.zeros(B, np.int32)
    r = orc.verify(z, z[:, :G], tok, u, 1.0, gamma_per_row=gam)
    want = orc.sample(np.ascontiguousarray(z[:, 0]), 1.0, 0, 1.0, u[:, 0, 1])
    assert np.all(r["accepted_len"] == 0) and np.array_equal(r["next_token"], want)
    # bonus row is target row gamma_b (not gamma_b - 1)
    z2 = z.copy()
    z2[:, G] = -np.inf
    z2[:, G, 7] = 0.0
    r = orc.verify(z2, z2[:, :G], tok, u, 1.0)
    assert np.all(r["next_token"] == 7)
    # error statuses
    bad = z.copy()
    bad[0, 0, 3] = np.nan
    bad[1, 0, :] = -np.inf
    bad[2, 0, 5] = np.inf
    tk = tok.copy()
    tk[3, 0] = V
    tk[4, 0] = -1
    uu = u.copy()
    uu[5, 0, 0] = 1.0
    gm = np.full(B, G, np.int32)
    gm[6] = G + 1
    gm[7] = -1
    r = orc.verify(bad, z[:, :G], tk, uu, 1.0, gamma_per_row=gm)
    want = {0: O.BAD_LOGIT, 1: O.NO_FINITE, 2: O.BAD_LOGIT, 3: O.BAD_TOKEN, 4: O.BAD_TOKEN,
            5: O.BAD_UNIFORM, 6: O.BAD_GAMMA, 7: O.BAD_GAMMA}
    for b, bit in want.items():
        assert r["row_status"][b] & bit, (b, r["row_status"][b])
        assert (r["accepted_len"][b], r["next_token"][b]) == (0, -1)


def pin_chi_square(orc):
    """10^6 draws: the first emitted token of a verify step is distributed as
    p (the target law), whatever q is."""
    rng = np.random.default_rng(16)
    V, G, N = 16, 2, 1_000_000
    zt = (rng.normal(size=(G + 1, V)) * 1.5).astype(np.float32)
    zd = (rng.normal(size=(G, V)) * 1.5).astype(np.float32)
    q0 = brute_law(zd[0], 1.0)
    tok = np.zeros((N, G), np.int32)
    tok[:, 0] = rng.choice(V, size=N, p=q0)
    tok[:, 1] = rng.choice(V, size=N, p=brute_law(zd[1], 1.0))
    u = rng.random((N, G + 1, 2), dtype=np.float32)
    r = orc.verify(np.broadcast_to(zt, (N, G + 1, V)), np.broadcast_to(zd, (N, G, V)), tok, u, 1.0)
    first = np.where(r["accepted_len"] >= 1, tok[:, 0], r["next_token"])
    obs = np.bincount(first, minlength=V)
    exp = brute_law(zt[0], 1.0) * N
    chi2 = float(((obs - exp) ** 2 / exp).sum())
    pval = float(scipy.stats.chi2.sf(chi2, V - 1))
    assert pval > 1e-3, (chi2, pval)


PINS = {
    "golden": pin_golden,
    "greedy": pin_greedy,
    "filters": pin_filters,
    "special": pin_special,
    "law_exact": pin_law_exact,
    "identities": pin_identities,
    "chi_square": pin_chi_square,
}
