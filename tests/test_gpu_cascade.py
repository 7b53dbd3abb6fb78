"""GPU parity of the multi-stage draft cascade ("CS3602_FINAL_SpeDec", 更多实现:
a chain of draft models, each drafting for the next larger one) with the
oracle's cascade, element by element on seeded inputs; and its output law
on the GPU at scale (the token at each slot follows the target's law there).

A row may differ from the oracle only where some stage's decision passes
within 1e-6 of a boundary (acceptance ratio, CDF, top-p mass) in the
oracle's fp64 run, and such rows stay below 1e-4 of the draws: the rule of
the single verify step, applied to every stage."""
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
from gpu_util import EPS_BOUNDARY, MAX_DISAGREE, draft_tokens_for, to_dev
from speculative_decoding_verify_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_03_gb300 as m
    m.build()
    oracle.build()
    return m


def _case(wid, seed, n_levels, rows=None, **over):
    w = W.WORKLOADS[wid]
    if over:
        import dataclasses
        w = dataclasses.replace(w, **over)
    b = W.make_batch(w, seed, rows=rows)
    c = W.cascade_levels(b, n_levels, seed + 1)
    return w, b, c


def _run_gpu(sv, w, c, tok, gam, T, k, p, **kw):
    import torch
    V = w.V
    lv = [to_dev(x)[:, :, :V] for x in c["levels"]]
    res = sv.spec_cascade_verify(lv, to_dev(np.ascontiguousarray(tok, np.int32)),
                                 to_dev(c["uniforms"]), T, k, p,
                                 gamma_per_row=to_dev(gam) if gam is not None else None, **kw)
    torch.cuda.synchronize()
    return [r.cpu().numpy() for r in res]


def _run_oracle(w, c, tok, gam, T, k, p):
    V = w.V
    return oracle.cascade([x[:, :, :V] for x in c["levels"]], tok, c["uniforms"], T, k, p,
                          gamma_per_row=gam, threads=16)


def compare_cascade(o, g):
    """The R2 rule over a cascade: returns the counts."""
    out_tok, out_len, stage_acc, status = g
    mism = (o["out_len"] != out_len) | (o["out_tokens"] != out_tok).any(axis=1) | \
           (o["stage_accepted"] != stage_acc).any(axis=0)
    near = o["margin"].min(axis=0) < EPS_BOUNDARY
    hard = mism & ~near
    info = {"rows": len(out_len), "draws": o["draws"], "near": int(near.sum()),
            "disagree": int(mism.sum()), "hard": int(hard.sum())}
    if hard.any():
        j = np.nonzero(hard)[0][:5]
        raise AssertionError(f"rows {j} differ away from any boundary: oracle "
                             f"{o['out_tokens'][j]} {o['stage_accepted'][:, j].T} gpu "
                             f"{out_tok[j]} {stage_acc[:, j].T} margins {o['margin'][:, j].T}")
    assert mism.sum() <= MAX_DISAGREE * max(o["draws"], 1), info
    agree = ~mism
    assert np.array_equal(o["row_status"][agree], status[agree])
    return info


CASES = [
    # (workload, seed, levels, rows, T, top_k, top_p)
    (3, 501, 3, 512, 1.0, 0, 1.0),       # Dirichlet V=1024: warp-per-row kernels
    (3, 502, 4, 256, 1.0, 0, 1.0),
    (1, 503, 3, 64, 1.0, 50, 0.9),       # strip kernel, top-k then top-p
    (4, 504, 3, 40, 0.7, 100, 0.9),      # ragged gamma, bf16, padded positions
    (2, 505, 3, 24, 0.8, 0, 0.95),       # top-p alone, bf16
    (1, 506, 4, 64, 0.0, 0, 1.0),        # greedy
]


@pytest.mark.parametrize("wid,seed,nl,nrows,T,k,p", CASES)
def test_cascade_parity(sv, wid, seed, nl, nrows, T, k, p):
    w, b, c = _case(wid, seed, nl, rows=np.arange(nrows))
    tok = draft_tokens_for(b, T, k, p)
    gam = b["gamma_per_row"]
    g = _run_gpu(sv, w, c, tok, gam, T, k, p)
    o = _run_oracle(w, c, tok, gam, T, k, p)
    info = compare_cascade(o, g)
    print(w.name, nl, info)
    # the first stage rejects somewhere, so corrections are passed up
    gm = np.full(nrows, w.gamma_max) if gam is None else gam
    assert (o["stage_accepted"][0] < gm).any()


def test_single_stage_equals_verify(sv):
    import torch
    w, b, c = _case(1, 511, 2, rows=np.arange(64))
    tok = draft_tokens_for(b, 1.0, 50, 0.9)
    g = _run_gpu(sv, w, c, tok, None, 1.0, 50, 0.9)
    V = w.V
    acc, nxt = sv.spec_verify(to_dev(b["target"])[:, :, :V], to_dev(b["draft"])[:, :, :V],
                              to_dev(tok), to_dev(b["uniforms"]), 1.0, 50, 0.9)
    torch.cuda.synchronize()
    acc, nxt = acc.cpu().numpy(), nxt.cpu().numpy()
    assert np.array_equal(g[2][0], acc)
    for r in range(64):
        want = list(tok[r, : acc[r]]) + [int(nxt[r])]
        assert g[0][r, : g[1][r]].tolist() == want


def test_cluster_kernel_gives_the_same(sv):
    w, b, c = _case(1, 512, 3, rows=np.arange(32))
    tok = draft_tokens_for(b, 1.0, 50, 0.9)
    a = _run_gpu(sv, w, c, tok, None, 1.0, 50, 0.9)
    z = _run_gpu(sv, w, c, tok, None, 1.0, 50, 0.9, kernel="cluster")
    for x, y in zip(a, z):
        assert np.array_equal(x, y)


def test_error_rows(sv):
    w, b, c = _case(3, 513, 3, rows=np.arange(64))
    tok = draft_tokens_for(b, 1.0, 0, 1.0)
    gam = np.full(64, w.gamma_max, np.int32)
    tok[3, 0] = w.V                       # bad draft token: stage 0
    c["levels"][0][5, 0, 7] = np.nan      # bad target logit: read at stage 1
    gam[7] = w.gamma_max + 1              # bad draft length
    gam[9] = 0                            # no drafts: the target's own draw
    g = _run_gpu(sv, w, c, tok, gam, 1.0, 0, 1.0)
    o = _run_oracle(w, c, tok, gam, 1.0, 0, 1.0)
    compare_cascade(o, g)
    for r in (3, 5, 7):
        assert g[1][r] == 0 and (g[0][r] == -1).all() and g[3][r] & oracle.ERROR_MASK
    assert g[2][1, 3] == -1
    assert g[1][9] == 1


def test_cascade_law_at_scale(sv):
    """Fixed logits broadcast over N rows (row stride 0), three draft levels,
    gamma 3, V 64: the token at each slot, over the rows that reach it,
    follows the target's law there (chi-square at level 1e-3), and the
    rows that keep every draft plus the bonus are as frequent as the
    acceptance rule makes them (sum over drafts of q_L(x) prod_s min(1,
    q_{s-1}(x) / q_s(x)) per slot)."""
    import torch
    N, G, V, L = 200_000, 3, 64, 3
    rng = np.random.default_rng(31)
    lv_np = [(rng.normal(size=(G + 1, V)) * 1.5).astype(np.float32) for _ in range(L)]
    lv_np.append((rng.normal(size=(G, V)) * 1.5).astype(np.float32))
    laws = [[scipy.special.softmax(x[i].astype(np.float64)) for i in range(x.shape[0])]
            for x in lv_np]
    d = np.stack([rng.choice(V, size=N, p=laws[L][i]) for i in range(G)], axis=1).astype(np.int32)
    u = rng.random((L, N, G + 1, 2), dtype=np.float32)
    lv = [torch.from_numpy(x).cuda().unsqueeze(0).expand(N, -1, -1) for x in lv_np]
    out_tok, out_len, _, st = sv.spec_cascade_verify(lv, to_dev(d), to_dev(u), 1.0)
    torch.cuda.synchronize()
    out_tok, m, st = out_tok.cpu().numpy(), out_len.cpu().numpy(), st.cpu().numpy()
    assert (st & oracle.ERROR_MASK).max() == 0
    assert (m >= 1).all() and (m <= G + 1).all()
    # only the last token of a row can differ from its drafts
    body = np.arange(G)[None, :] < (m - 1)[:, None]
    assert (out_tok[:, :G][body] == d[body]).all()
    for i in range(G + 1):
        x = out_tok[m > i, i]
        obs = np.bincount(x, minlength=V)
        exp = laws[0][i] * len(x)
        keep = exp >= 5
        stat = float(((obs[keep] - exp[keep]) ** 2 / exp[keep]).sum())
        pval = float(scipy.stats.chi2.sf(stat, keep.sum() - 1))
        print(f"slot {i}: {len(x)} draws, chi2 {stat:.1f}, p {pval:.3g}")
        assert pval > 1e-3, (i, pval)
    a = np.ones(N)
    for s in range(L, 0, -1):
        for i in range(G):
            q, p = laws[s][i][d[:, i]], laws[s - 1][i][d[:, i]]
            a *= np.minimum(1.0, p / q)
    want, got = a.mean(), float(np.mean(m == G + 1))
    assert abs(got - want) < 4 * math.sqrt(want * (1 - want) / N), (got, want)
