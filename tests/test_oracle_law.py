"""Pins of the oracle's emitted-token law ("CS3602_FINAL_SpeDec", section 2
困惑度测试 (PPL)): the page's proof says it equals the target law p for every
token, whatever q, and its terms have closed forms: beta is the expected
acceptance probability sum_x q(x) min(1, p(x)/q(x)); p = q gives beta = 1;
disjoint supports give beta = 0."""
import numpy as np
import pytest

import oracle


def _rows(seed, n, V, spread=2.0):
    rng = np.random.default_rng(seed)
    z = (rng.normal(size=(n, V)) * spread).astype(np.float32)
    w = (0.5 * z + rng.normal(size=(n, V)) * spread).astype(np.float32)
    return z, w


@pytest.mark.parametrize("T,k,p", [(1.0, 0, 1.0), (0.7, 0, 1.0), (1.0, 20, 1.0), (1.3, 0, 0.8),
                                   (0.9, 30, 0.9)])
def test_law_equals_target_law(T, k, p):
    z, w = _rows(1, 6, 300)
    for x in (0, 7, 123, 299):
        r = oracle.law(z, w, np.full(6, x), T, k, p)
        for i in range(6):
            pt, _, _ = oracle.distribution(z[i], T, k, p)
            assert abs(r["p_spec"][i] - pt[x]) <= 1e-12
            assert r["p_x"][i] == pt[x]


def test_law_sums_to_one_and_beta_is_the_acceptance_rate():
    z, w = _rows(2, 1, 200)
    V = 200
    r = oracle.law(np.repeat(z, V, 0), np.repeat(w, V, 0), np.arange(V), 1.0)
    assert abs(r["p_spec"].sum() - 1.0) <= 1e-12
    pt, _, _ = oracle.distribution(z[0], 1.0, 0, 1.0)
    qt, _, _ = oracle.distribution(w[0], 1.0, 0, 1.0)
    accept = sum(qt[x] * min(1.0, pt[x] / qt[x]) for x in range(V) if qt[x] > 0)
    assert abs(r["beta"][0] - accept) <= 1e-12


def test_special_cases():
    z, _ = _rows(3, 2, 64)
    r = oracle.law(z, z.copy(), [5, 9], 1.0)            # p == q
    assert np.allclose(r["beta"], 1.0, atol=1e-12)
    w = np.full_like(z, -np.inf)                          # disjoint supports
    z2 = z.copy()
    z2[:, 32:] = -np.inf
    w[:, 32:] = 0.0
    r = oracle.law(z2, w, [5, 40], 1.0)
    assert np.allclose(r["beta"], 0.0, atol=1e-15)
    pt, _, _ = oracle.distribution(z2[0], 1.0, 0, 1.0)
    assert abs(r["p_spec"][0] - pt[5]) <= 1e-12 and r["p_spec"][1] == 0.0
    r = oracle.law(z, z, [-1, 64], 1.0)                  # tokens out of range
    assert np.isnan(r["p_spec"]).all()
