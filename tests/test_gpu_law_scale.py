"""The law of the GPU verify step at scale, on the Dirichlet workload (B=4096
rows, gamma=4, V=1024, fp32; p and q ~ Dirichlet(0.3) per row and position,
stored as log-probabilities): the same logits are verified 245 times with
fresh draft tokens (drawn from q) and uniforms, about 10^6 position-0
draws in all.

"CS3602_FINAL_SpeDec", section "2. 困惑度测试(PPL)": the token emitted at a
position follows the target law p there, whatever q is (P(x) = min(p, q) +
(p - min(p, q)) = p).  Checked per position i: every row that reached i
contributes one draw from its own p_i (the accepted draft token, or the
resampled or bonus token); the rows are pooled with a chi-square statistic
per row (bins merged, in decreasing p, until each expects at least 5) summed
over rows, tested at level 1e-3.  Tokens outside p's support must never
appear.  Also the accepted-length law P(len >= i) = prod_{j<i} beta_j with
beta_j = sum_v min(p_j, q_j) (the acceptance rate the same section derives),
and the residual mass identity sum_v max(0, p - q) = 1 - beta at every
rejected position (debug output against the oracle's laws)."""
import numpy as np
import pytest
import scipy.stats

import oracle
from gpu_util import to_dev
from speculative_decoding_verify_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CALLS = 245
LEVEL = 1e-3


@pytest.fixture(scope="module")
def sv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_03_gb300 as m
    m.build()
    oracle.build()
    return m


def _laws(z):
    """p (or q) of every (row, position) as float64 [B, P, V], from the oracle."""
    B, P, V = z.shape
    out = np.empty((B, P, V))
    for b in range(B):
        for i in range(P):
            out[b, i], _, st = oracle.distribution(np.ascontiguousarray(z[b, i]), 1.0)
            assert st == 0
    return out


def _pooled_chi2(counts, laws):
    """Sum over rows of the per-row chi-square statistic of counts[b] against
    n_b * laws[b] (bins: tokens in decreasing law, merged until each bin
    expects >= 5; the last partial bin joins the one before); returns (stat,
    degrees of freedom, rows used)."""
    stat, dof, used = 0.0, 0, 0
    for c, p in zip(counts, laws):
        n = c.sum()
        if n < 10:
            continue
        o = np.argsort(-p, kind="stable")
        e = n * p[o]
        cs = np.cumsum(e)
        bins = np.floor((cs - e) / 5.0).astype(np.int64)  # bin of each token
        last = bins.max()
        if last == 0:
            continue
        tail = e[bins == last].sum()
        if tail < 5.0:
            bins[bins == last] = last - 1
            last -= 1
        eb = np.bincount(bins, weights=e, minlength=last + 1)
        ob = np.bincount(bins, weights=c[o], minlength=last + 1)
        stat += float(((ob - eb) ** 2 / eb).sum())
        dof += last
        used += 1
    return stat, dof, used


def _pit(counts, laws, rng):
    """F = sum of p over the tokens before x + U p(x) for every draw x (counts
    [B, V] of draws from laws [B, V]), tokens ordered by decreasing p."""
    o = np.argsort(-laws, axis=1, kind="stable")
    srt = np.take_along_axis(laws, o, axis=1)
    before = np.cumsum(srt, axis=1) - srt
    cb = np.empty_like(laws)
    np.put_along_axis(cb, o, before, axis=1)
    b, v = np.nonzero(counts)
    c = counts[b, v]
    bb, vv = np.repeat(b, c), np.repeat(v, c)
    return cb[bb, vv] + rng.random(len(bb)) * laws[bb, vv]


def test_dirichlet_law_at_scale(sv):
    import torch
    w = W.WORKLOADS[3]
    B, G, V = w.B, w.gamma_max, w.V
    batch = W.make_batch(w, 3001)
    zt, zd = batch["target"][:, :, :V], batch["draft"][:, :, :V]
    p = _laws(zt)          # [B, G+1, V]
    q = _laws(zd)          # [B, G, V]
    beta = np.minimum(p[:, :G], q).sum(axis=2)   # [B, G]
    qcdf = np.cumsum(q, axis=2)
    qcdf[:, :, -1] = np.inf
    tgt, drf = to_dev(batch["target"])[:, :, :V], to_dev(batch["draft"])[:, :, :V]
    rng = np.random.Generator(np.random.Philox(77))
    counts = np.zeros((B, G + 1, V), np.int64)
    reach = np.zeros(G + 2, np.int64)   # rows with accepted_len >= i, over all calls
    bad_resid = 0
    for c in range(CALLS):
        # draft tokens from q by the inverse CDF (numpy), uniforms fresh
        uq = rng.random((B, G))
        tok = (qcdf < uq[:, :, None]).sum(axis=2).astype(np.int32)
        uni = rng.random((B, G + 1, 2), dtype=np.float32)
        acc, nxt, dbg = sv.spec_verify(tgt, drf, to_dev(tok), to_dev(uni), 1.0, 0, 1.0,
                                       debug=True)
        torch.cuda.synchronize()
        acc, nxt = acc.cpu().numpy(), nxt.cpu().numpy()
        assert (dbg["row_status"].cpu().numpy() & oracle.ERROR_MASK).max() == 0
        resid = dbg["residual_mass"].cpu().numpy()
        for i in range(G + 1):
            reach[i] += int((acc >= i).sum())
        # position i < acc: the accepted draft; position acc: next_token
        for i in range(G):
            r = np.nonzero(acc > i)[0]
            np.add.at(counts, (r, i, tok[r, i]), 1)
        r = np.arange(B)
        np.add.at(counts, (r, acc, nxt), 1)
        # residual mass at the rejected position = 1 - beta there
        rej = np.nonzero(acc < G)[0]
        want = 1.0 - beta[rej, acc[rej]]
        bad_resid += int((np.abs(resid[rej] - want) > 1e-5).sum())
    assert bad_resid == 0
    # support: tokens with p = 0 are never emitted
    assert counts[p[:, :, :] == 0.0].sum() == 0
    # the emitted token at each position follows p there (pooled over rows)
    prng = np.random.Generator(np.random.Philox(78))
    for i in range(G + 1):
        stat, dof, used = _pooled_chi2(counts[:, i], p[:, i])
        if dof > 0:
            pval = float(scipy.stats.chi2.sf(stat, dof))
            print(f"position {i}: rows {used}, draws {counts[:, i].sum()}, chi2 {stat:.0f} "
                  f"dof {dof} p {pval:.3g}")
            assert pval > LEVEL, (i, stat, dof, pval)
        # every draw of the position (rows with few draws included): the
        # randomised probability integral transform F = P(before x) + U p(x),
        # tokens ordered by decreasing p, is uniform on [0, 1) exactly when x
        # follows p; a chi-square test over 100 equal bins
        pit = _pit(counts[:, i], p[:, i], prng)
        obs = np.bincount(np.minimum((pit * 100).astype(np.int64), 99), minlength=100)
        pval = float(scipy.stats.chisquare(obs).pvalue)
        print(f"position {i}: {len(pit)} draws, PIT p {pval:.3g}")
        assert pval > LEVEL, (i, pval)
    assert counts[:, 0].sum() == B * CALLS
    # accepted-length law: E[#rows with len >= i] = CALLS * sum_b prod_{j<i} beta_j
    for i in range(1, G + 1):
        pi = np.prod(beta[:, :i], axis=1)
        mean = CALLS * pi.sum()
        sd = np.sqrt(CALLS * (pi * (1 - pi)).sum())
        z = (reach[i] - mean) / sd
        print(f"P(len >= {i}): observed {reach[i] / (CALLS * B):.5f} "
              f"expected {mean / (CALLS * B):.5f} (z {z:.2f})")
        assert abs(z) < scipy.stats.norm.isf(LEVEL / 2), (i, reach[i], mean, sd)
