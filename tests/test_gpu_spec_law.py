"""spec_law (the emitted-token law, for scoring) against the fp64 oracle:
probabilities within 1e-5 absolute, on fp32 and bf16 rows of several
vocabulary sizes and temperatures, unfiltered and filtered (top-k, top-p,
both; rows whose laws lie within 1e-6 of a top-p boundary are exempt, as in
the verify step's parity rule); NaN for out-of-range tokens and rows in
error."""
import numpy as np
import pytest

import oracle
from gpu_util import to_dev
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


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V,T", [(1024, 1.0), (5003, 0.7), (50304, 1.0), (152064, 0.8)])
def test_law_matches_oracle(sv, V, T, dtype):
    import torch
    rng = np.random.default_rng(V)
    n = 24
    z = (rng.normal(size=(n, V)) * 3).astype(np.float32)
    w = (0.8 * z + rng.normal(size=(n, V)) * 1.5).astype(np.float32)
    if dtype == "bf16":
        z, w = W.f32_to_bf16_bits(z), W.f32_to_bf16_bits(w)
    # tokens: the target argmax (large p), random ones (small p), one draft argmax
    zf = z if dtype == "f32" else (z.astype(np.uint32) << 16).view(np.float32)
    tok = rng.integers(0, V, size=n).astype(np.int32)
    tok[::3] = np.argmax(zf[::3], axis=1)
    want = oracle.law(z, w, tok, T)
    ps, beta, px, qx = sv.spec_law(to_dev(z), to_dev(w), to_dev(tok), T)
    torch.cuda.synchronize()
    for name, got in (("p_spec", ps), ("beta", beta), ("p_x", px), ("q_x", qx)):
        err = np.abs(got.cpu().numpy().astype(np.float64) - want[name])
        assert err.max() <= 1e-5, (name, err.max())


def test_law_errors(sv):
    import torch
    V, n = 777, 4
    rng = np.random.default_rng(1)
    z = rng.normal(size=(n, V)).astype(np.float32)
    w = rng.normal(size=(n, V)).astype(np.float32)
    z[2, 5] = np.nan
    w[3, :] = -np.inf
    tok = np.array([V, -1, 3, 3], np.int32)
    ps, beta, px, qx = sv.spec_law(to_dev(z), to_dev(w), to_dev(tok), 1.0)
    torch.cuda.synchronize()
    assert np.isnan(ps.cpu().numpy()).all()
    assert np.isfinite(beta.cpu().numpy()[:2]).all()


@pytest.mark.parametrize("wid,V,T,k,p", [
    (1, 50304, 1.0, 50, 0.9),      # the B=64 fp32 workload's filters
    (2, 128256, 0.8, 0, 0.95),     # top-p alone, bf16 Zipf logits
    (4, 152064, 0.7, 100, 0.9),    # top-k then top-p, bf16
    (1, 9001, 1.0, 7, 1.0),        # top-k alone
    (0, 20011, 1.0, 0, 0.9),       # top-p alone, flat N(0, 3^2) laws (large nuclei)
])
@pytest.mark.parametrize("path", ["strip", "row", "overflow"])
def test_filtered_law_matches_oracle(sv, wid, V, T, k, p, path):
    """path: "strip" (a workspace: the strip-parallel kernel), "row" (no
    workspace: one CTA per row), "overflow" (the strip kernel with a
    candidate capacity of 16, forcing its slice-wide fallback)."""
    import torch
    from dataclasses import replace
    w = replace(W.WORKLOADS[wid], B=6, V=V, pos_pad=0)
    b = W.make_batch(w, 900 + wid)
    G = w.gamma_max
    tg = np.ascontiguousarray(b["target"][:, :G, :V]).reshape(-1, V)
    dr = np.ascontiguousarray(b["draft"][:, :G, :V]).reshape(-1, V)
    n = tg.shape[0]
    rng = np.random.default_rng(V + k)
    tok = oracle.sample(dr, T, k, p, rng.random(n).astype(np.float32))
    tok[::4] = rng.integers(0, V, size=len(tok[::4]))  # some tokens outside the kept sets
    want = oracle.law(tg, dr, tok, T, k, p)
    kw = {"strip": {}, "row": {"workspace": None}, "overflow": {"list_capacity": 16}}[path]
    ps, beta, px, qx = sv.spec_law(to_dev(tg), to_dev(dr), to_dev(tok.astype(np.int32)), T, k, p,
                                   **kw)
    torch.cuda.synchronize()
    # rows near a top-p boundary (either law) are boundary events
    near = np.zeros(n, bool)
    for r in range(n):
        for z in (tg[r], dr[r]):
            _, mg, _ = oracle.distribution(np.ascontiguousarray(z), T, k, p)
            near[r] |= mg < 1e-6
    keep = ~near
    assert keep.sum() >= n - 2
    for name, got in (("p_spec", ps), ("beta", beta), ("p_x", px), ("q_x", qx)):
        err = np.abs(got.cpu().numpy().astype(np.float64) - want[name])[keep]
        assert err.max() <= 1e-5, (name, err.max())


@pytest.mark.parametrize("ws", ["auto", None])
def test_filtered_law_error_rows(sv, ws):
    """Filtered laws on either path: a token outside [0, V), a NaN logit, a
    row with no finite logit give NaN; the other rows are unaffected."""
    import torch
    rng = np.random.default_rng(41)
    n, V = 6, 30011
    z = (rng.normal(size=(n, V)) * 2).astype(np.float32)
    w = (rng.normal(size=(n, V)) * 2).astype(np.float32)
    z[2, 5] = np.nan
    w[3, :] = -np.inf
    tok = np.array([V, -1, 3, 3, 7, 11], np.int32)
    ps, beta, px, qx = sv.spec_law(to_dev(z), to_dev(w), to_dev(tok), 1.0, 20, 0.9, workspace=ws)
    torch.cuda.synchronize()
    ps = ps.cpu().numpy()
    assert np.isnan(ps[:4]).all()
    want = oracle.law(z[4:], w[4:], tok[4:], 1.0, 20, 0.9)
    assert np.abs(ps[4:] - want["p_spec"]).max() <= 1e-5
