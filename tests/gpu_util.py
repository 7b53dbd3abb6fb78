"""Helpers shared by the GPU tests: run the CUDA path and the oracle on the
same seeded inputs and compare them."""
from __future__ import annotations

import os

import numpy as np

import oracle
from speculative_decoding_verify_03_gb300 import workloads as W

EPS_BOUNDARY = 1e-6    # a draw this close to a decision or CDF boundary is exempt
MAX_DISAGREE = 1e-4    # ... but such disagreements stay below this fraction of draws
PROB_TOL = 1e-5        # fp32 p(x), q(x), residual mass vs the fp64 oracle


def to_dev(a: np.ndarray):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def draft_tokens_for(batch, T, top_k, top_p):
    """Draft tokens drawn from the filtered draft law q by the oracle's sampler."""
    w = batch["workload"]
    d = batch["draft"][:, :, : w.V]
    n, G = d.shape[0], d.shape[1]
    if G == 0:
        return np.zeros((n, 0), np.int32)
    flat = np.ascontiguousarray(d).reshape(n * G, w.V)
    tok = oracle.sample(flat, T, top_k, top_p, batch["draft_uniforms"].reshape(-1))
    return tok.reshape(n, G)


def run_gpu(batch, tokens, T, top_k, top_p, debug=True, **kw):
    import speculative_decoding_verify_03_gb300 as sv
    w = batch["workload"]
    tgt = to_dev(batch["target"])[:, :, : w.V]
    drf = to_dev(batch["draft"])[:, :, : w.V]
    tok = to_dev(np.ascontiguousarray(tokens, np.int32))
    uni = to_dev(batch["uniforms"])
    gam = to_dev(batch["gamma_per_row"]) if batch["gamma_per_row"] is not None else None
    res = sv.spec_verify(tgt, drf, tok, uni, T, top_k, top_p, gamma_per_row=gam, debug=debug, **kw)
    import torch
    torch.cuda.synchronize()
    out = {"accepted_len": res[0].cpu().numpy(), "next_token": res[1].cpu().numpy()}
    if debug:
        out.update({k: v.cpu().numpy() for k, v in res[2].items()})
    return out


def run_oracle(batch, tokens, T, top_k, top_p, rows=None):
    w = batch["workload"]
    o = oracle.verify(batch["target"][:, :, : w.V], batch["draft"][:, :, : w.V], tokens,
                      batch["uniforms"], T, top_k, top_p,
                      gamma_per_row=batch["gamma_per_row"], rows=rows,
                      threads=min(16, os.cpu_count() or 1))
    n = len(o["accepted_len"])
    o["gamma"] = (batch["gamma_per_row"].astype(np.int64) if batch["gamma_per_row"] is not None
                  else np.full(n, w.gamma_max, np.int64))
    return o


def compare(o, g, rows=None, check_probs=True):
    """Parity of the CUDA outputs `g` with the oracle's `o` on `rows`.

    Token ids and accepted lengths must be identical, except on rows whose
    oracle decision path passes within EPS_BOUNDARY of a decision boundary
    (acceptance ratio, CDF boundary, top-p mass); those disagreements are
    counted and must stay below MAX_DISAGREE of all draws.  Statuses must be
    equal on agreeing rows; p(x), q(x) and the residual mass within PROB_TOL.
    Returns a summary dict."""
    if rows is None:
        rows = np.arange(len(o["accepted_len"]))
    d = o["diag"][rows]
    near = (d["accept_margin"] < EPS_BOUNDARY) | (d["cdf_margin"] < EPS_BOUNDARY) | \
           (d["topp_margin"] < EPS_BOUNDARY)
    oa, on = o["accepted_len"][rows], o["next_token"][rows]
    ga, gn = g["accepted_len"][rows], g["next_token"][rows]
    mism = (oa != ga) | (on != gn)
    hard = mism & ~near
    draws = int(d["n_tests"].sum() + d["n_draws"].sum())
    info = {"rows": len(rows), "draws": draws, "near": int(near.sum()),
            "disagree": int(mism.sum()), "hard": int(hard.sum())}
    if hard.any():
        j = np.nonzero(hard)[0][:5]
        raise AssertionError(f"disagreement away from any boundary at rows {rows[j]}: "
                             f"oracle {list(zip(oa[j], on[j]))} gpu {list(zip(ga[j], gn[j]))} "
                             f"margins {d[j]} status o={o['row_status'][rows][j]} "
                             f"g={g.get('row_status', np.zeros(len(rows)))[rows][j] if 'row_status' in g else None}")
    assert mism.sum() <= MAX_DISAGREE * max(draws, 1), info
    agree = ~mism
    # a row whose filtered law lies within EPS_BOUNDARY of a top-p boundary
    # is a filter-boundary event: its kept set may differ, so its p(x), q(x)
    # and residual mass are exempt like its tokens
    pagree = agree & (d["topp_margin"] >= EPS_BOUNDARY)
    if "row_status" in g:
        os_, gs = o["row_status"][rows][agree], g["row_status"][rows][agree]
        if not np.array_equal(os_, gs):
            j = np.nonzero(os_ != gs)[0][:5]
            raise AssertionError(f"status differs at rows {rows[agree][j]}: {os_[j]} vs {gs[j]}")
    if check_probs and "p_draft" in g:
        for key in ("p_draft", "q_draft"):
            a, b = o[key][rows][pagree], g[key][rows][pagree]
            both = ~np.isnan(a)
            assert np.array_equal(np.isnan(a), np.isnan(b)), f"{key}: evaluated positions differ"
            err = np.abs(a[both].astype(np.float64) - b[both])
            assert err.size == 0 or err.max() <= PROB_TOL, f"{key}: max err {err.max()}"
            info[f"{key}_maxerr"] = float(err.max()) if err.size else 0.0
        rej = pagree & (oa < o["gamma"][rows]) & ((o["row_status"][rows] & oracle.ERROR_MASK) == 0)
        a = o["diag"]["residual_mass"][rows][rej]
        b = g["residual_mass"][rows][rej]
        if a.size:
            err = np.abs(a - b)
            assert err.max() <= PROB_TOL, f"residual mass max err {err.max()}"
    return info


def compare_samples(want, got, cdf_margin, topp_margin):
    """Parity of GPU draws with the oracle's sampler (the same rule as
    compare): every differing draw must have its uniform within
    EPS_BOUNDARY of a CDF boundary or its law within EPS_BOUNDARY of a top-p
    boundary, and differing draws stay below MAX_DISAGREE of all draws."""
    near = (cdf_margin < EPS_BOUNDARY) | (topp_margin < EPS_BOUNDARY)
    mism = want != got
    hard = mism & ~near
    info = {"draws": int(len(want)), "near": int(near.sum()), "disagree": int(mism.sum()),
            "hard": int(hard.sum())}
    if hard.any():
        j = np.nonzero(hard)[0][:5]
        raise AssertionError(f"draws differ away from any boundary at {j}: oracle {want[j]} "
                             f"gpu {got[j]} margins {cdf_margin[j]} {topp_margin[j]}")
    assert mism.sum() <= MAX_DISAGREE * max(len(want), 1), info
    return info


def case(wid_or_w, seed, rows=None, **over):
    """Build a (possibly shrunk) workload batch."""
    w = W.WORKLOADS[wid_or_w] if isinstance(wid_or_w, int) else wid_or_w
    if over:
        from dataclasses import replace
        w = replace(w, **over)
    return W.make_batch(w, seed, rows=rows)
