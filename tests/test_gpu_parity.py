"""CUDA path vs the fp64 oracle, element by element, on seeded inputs.

Shrunk versions of every workload (several vocabulary tiles per CTA, ragged
tails, every cluster size), edge cases, determinism, and the full-size
workloads in the launch configuration the benchmark times (GPU on the whole
batch, oracle on sampled rows)."""
from dataclasses import replace

import numpy as np
import pytest

import oracle
from gpu_util import (case, compare, compare_samples, draft_tokens_for, run_gpu, run_oracle,
                      to_dev)
from speculative_decoding_verify_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_03_gb300 as sv
    sv.build()
    oracle.build()
    return sv


# Kernel selection: "cluster" forces the cluster-per-row kernel; "auto"
# (with a workspace) lets the strip-parallel kernel take greedy and top-k
# problems and the warp-per-row kernel small greedy or unfiltered ones (which
# hands its uncertain rows to the cluster kernel); "nows" (no workspace): the
# warp-per-row kernel redoes such rows itself, the rest run on the cluster
# kernel.
PATHS = {"cluster": dict(workspace=None, kernel="cluster"), "auto": dict(workspace="auto"),
         "nows": dict(workspace=None)}


def parity(batch, T, k, p, rows=None, **kw):
    tok = draft_tokens_for(batch, T, k, p)
    g = run_gpu(batch, tok, T, k, p, **kw)
    o = run_oracle(batch, tok, T, k, p, rows=rows)
    return compare(o, g, rows=rows), g, o


SMALL = [
    # (workload, overrides, T, top_k, top_p)
    (0, dict(B=8, V=5003), 0.0, 0, 1.0),
    (0, dict(B=8, V=5003), 1.0, 0, 1.0),
    (0, dict(B=6, V=20011, dtype="bf16"), 1.0, 0, 1.0),
    (1, dict(B=16, V=9001), 1.0, 50, 0.9),
    (1, dict(B=16, V=9001, dtype="bf16"), 0.6, 50, 0.9),
    (1, dict(B=12, V=9001), 1.0, 7, 1.0),
    (2, dict(B=12, V=30011, gamma_max=5), 0.8, 0, 0.95),
    (3, dict(B=64), 1.0, 0, 1.0),
    (4, dict(B=12, V=30011), 0.7, 100, 0.9),
]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("cluster", [1, 2, 4, 8])
@pytest.mark.parametrize("ci", range(len(SMALL)))
def test_parity_small(ci, cluster, path):
    wid, over, T, k, p = SMALL[ci]
    batch = case(wid, 100 + ci, **over)
    info, g, o = parity(batch, T, k, p, cluster_size=cluster, **PATHS[path])
    assert info["hard"] == 0


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("cap", [16, 64])
@pytest.mark.parametrize("ci", [3, 4, 5, 6, 8])
def test_parity_list_overflow_fallback(ci, cap, path):
    """A tiny candidate-list capacity forces the exact slice-wide selection
    for some or all rows; results must not change."""
    wid, over, T, k, p = SMALL[ci]
    batch = case(wid, 200 + ci, **over)
    info, g, o = parity(batch, T, k, p, list_capacity=cap, cluster_size=2,
                        **PATHS[path])
    assert info["hard"] == 0


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_greedy_ties_and_argmax(dtype, path):
    rng = np.random.default_rng(3)
    w = replace(W.WORKLOADS[0], B=32, V=4099, dtype=dtype)
    batch = W.make_batch(w, 7)
    # integer logits: many ties; greedy must pick the first maximum
    t = rng.integers(-3, 4, size=batch["target"].shape).astype(np.float32)
    batch["target"] = W.f32_to_bf16_bits(t) if dtype == "bf16" else t
    tok = np.argmax(t[:, :-1, : w.V], axis=2).astype(np.int32)
    tok[::3, 1] = (tok[::3, 1] + 1) % w.V
    g = run_gpu(batch, tok, 0.0, 0, 1.0, **PATHS[path])
    o = run_oracle(batch, tok, 0.0, 0, 1.0)
    compare(o, g)
    assert np.array_equal(g["accepted_len"], o["accepted_len"])
    assert np.array_equal(g["next_token"], o["next_token"])


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("V,k,p", [(3001, 20, 0.9), (1000, 0, 1.0), (1024, 0, 1.0)])
def test_error_rows_and_edge_cases(path, V, k, p):
    w = replace(W.WORKLOADS[1], B=16, V=V, dtype="f32")
    batch = W.make_batch(w, 9)
    T = 1.0
    tok = draft_tokens_for(batch, T, k, p)
    tg = batch["target"]
    tg[0, 0, 5] = np.nan
    tg[1, 0, :] = -np.inf
    tg[2, 0, 17] = np.inf
    tok[3, 0] = w.V
    tok[4, 0] = -5
    batch["uniforms"][5, 0, 0] = 1.0
    batch["uniforms"][6, 0, 0] = np.nan
    tg[7, 1, : w.V] = -np.inf  # error only if position 1 is reached
    tg[7, 1, 3] = 0.0
    batch["draft"][8] = tg[8, :-1]  # p == q: every draft accepted
    batch["gamma_per_row"] = np.full(w.B, w.gamma_max, np.int32)
    batch["gamma_per_row"][9] = 0
    batch["gamma_per_row"][10] = w.gamma_max + 1
    batch["gamma_per_row"][11] = -1
    tok8 = draft_tokens_for({"workload": w, "draft": batch["draft"][8:9],
                             "draft_uniforms": batch["draft_uniforms"][8:9]}, T, k, p)
    tok[8] = tok8[0]
    g = run_gpu(batch, tok, T, k, p, **PATHS[path])
    o = run_oracle(batch, tok, T, k, p)
    compare(o, g)
    assert g["row_status"][0] & oracle.BAD_LOGIT and g["accepted_len"][0] == 0
    assert g["row_status"][1] & oracle.NO_FINITE and g["next_token"][1] == -1
    assert g["row_status"][3] & oracle.BAD_TOKEN and g["row_status"][4] & oracle.BAD_TOKEN
    assert g["row_status"][5] & oracle.BAD_UNIFORM and g["row_status"][6] & oracle.BAD_UNIFORM
    assert g["accepted_len"][8] == w.gamma_max
    assert g["accepted_len"][9] == 0 and g["next_token"][9] >= 0
    assert g["row_status"][10] & oracle.BAD_GAMMA and g["row_status"][11] & oracle.BAD_GAMMA


@pytest.mark.parametrize("V", [1, 2, 7, 33, 257])
@pytest.mark.parametrize("T,k,p", [(0.0, 0, 1.0), (1.0, 0, 1.0), (0.9, 3, 1.0), (1.1, 0, 0.5),
                                   (1.0, 1, 1.0), (1.0, 0, 1e-6)])
@pytest.mark.parametrize("path", PATHS)
def test_tiny_vocabularies(V, T, k, p, path):
    w = replace(W.WORKLOADS[1], B=40, V=V, gamma_max=3)
    batch = W.make_batch(w, 11 + V)
    info, g, o = parity(batch, T, k, p, **PATHS[path])
    assert info["hard"] == 0


@pytest.mark.parametrize("wid,over,T,k,p", [
    (1, dict(B=24, V=9001), 1.0, 50, 0.9),
    (2, dict(B=8, V=30011), 0.8, 0, 0.95),
    (3, dict(B=128), 1.0, 0, 1.0),
    (4, dict(B=24, V=30011), 0.7, 100, 0.9),
])
@pytest.mark.parametrize("path", PATHS)
def test_bitwise_determinism(wid, over, T, k, p, path):
    batch = case(wid, 21, **over)
    tok = draft_tokens_for(batch, T, k, p)
    a = run_gpu(batch, tok, T, k, p, **PATHS[path])
    b = run_gpu(batch, tok, T, k, p, **PATHS[path])
    for key in a:
        assert np.array_equal(a[key].view(np.uint8), b[key].view(np.uint8)), key


@pytest.mark.parametrize("wid,over,T,k,p", [
    (1, dict(B=32, V=9001), 1.0, 50, 0.9),
    (2, dict(B=24, V=30011), 0.8, 0, 0.95),
    (3, dict(B=64), 1.0, 0, 1.0),
    (0, dict(B=16, V=5003), 0.0, 0, 1.0),
    (3, dict(B=2500, V=1000), 0.9, 0, 1.0),              # 10^4 draws, warp-per-row kernel
    (4, dict(B=160, V=20011, gamma_max=8), 0.7, 100, 0.9),  # 1280 draws, top-k then top-p
    (2, dict(B=160, V=12007, gamma_max=8), 0.8, 0, 0.95),   # 1280 draws, top-p alone
])
@pytest.mark.parametrize("ws", ["auto", None])
def test_sampler_parity(wid, over, T, k, p, ws):
    """The draft-token sampler against the oracle's, draw by draw, under the
    same rule as the verify step: a differing draw must lie within 1e-6 of a
    CDF or top-p boundary, and such draws stay below 1e-4 of all draws.  ws:
    "auto" (the strip-parallel and CTA-per-row kernels), None (the
    warp-per-row and cluster kernels)."""
    import speculative_decoding_verify_03_gb300 as sv
    batch = case(wid, 31, **over)
    w = batch["workload"]
    flat = np.ascontiguousarray(batch["draft"][:, :, : w.V]).reshape(-1, w.V)
    u = batch["draft_uniforms"].reshape(-1)
    want, cm, tm = oracle.sample(flat, T, k, p, u, margins=True)
    got = sv.spec_sample(to_dev(flat), to_dev(u), T, k, p, workspace=ws).cpu().numpy()
    info = compare_samples(want, got, cm, tm)
    assert info["hard"] == 0


def ramp_logits(rng, shape, V, per_bin, T):
    """Logits that fall linearly over a random permutation of the vocabulary,
    about per_bin[row] of them per 1/8 log2 unit of weight, plus a jitter of
    a quarter step: wide nuclei (thousands of tokens) whose top-p crossing
    lies where the pieces' candidates, the extension and the rescan's full
    region (at most 2048 entries) cannot reach it."""
    out = np.empty(shape + (V,), np.float32)
    for idx in np.ndindex(*shape):
        step = 0.125 * np.log(2.0) * T / per_bin[idx[0]]
        rank = rng.permutation(V)
        out[idx] = -step * rank + rng.random(V) * 0.25 * step
    return out


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mix", ["window", "mixed"])
def test_topp_rescan_window(dtype, mix):
    """Top-p alone on ramp laws whose nucleus holds about 10^4 tokens.  With
    about 400 logits per depth bin the rescan's region up to the crossing
    bin exceeds its 2048 entries but the window of bins around the crossing
    does not: the rescan then gives the threshold and the exact normaliser
    without a list, and the draws run over the strip; no position takes the
    slice-wide bisection (diagnostics word 0).  "mixed" rows span the list
    (60 per bin), the window (400) and the slice-wide path (3000).  The
    verify step, the sampler and the law evaluation match the oracle."""
    import speculative_decoding_verify_03_gb300 as sv
    import torch
    V, B, G, T, p = 20011, 6, 3, 1.0, 0.9
    rng = np.random.default_rng(77 if dtype == "f32" else 78)
    per_bin = np.full(B, 400) if mix == "window" else np.array([60, 400, 3000] * 2)
    batch = case(0, 79, B=B, V=V, gamma_max=G, dtype=dtype)
    tgt = ramp_logits(rng, (B, G + 1), V, per_bin, T)
    drf = ramp_logits(rng, (B, G), V, per_bin, T)
    if dtype == "bf16":
        tgt, drf = W.f32_to_bf16_bits(tgt), W.f32_to_bf16_bits(drf)
    batch["target"], batch["draft"] = tgt, drf
    tok = draft_tokens_for(batch, T, 0, p)
    P = sv.make_params(to_dev(tgt), to_dev(drf), T, 0, p)
    ws = torch.zeros(sv.workspace_bytes(P), dtype=torch.uint8, device="cuda")
    g = run_gpu(batch, tok, T, 0, p, workspace=ws)
    o = run_oracle(batch, tok, T, 0, p)
    info = compare(o, g)
    assert info["hard"] == 0
    diag = sv.read_diagnostics(ws)
    assert diag[3] > 0, diag
    if mix == "window":
        assert diag[0] == 0, diag
    # the sampler on the draft rows
    flat = np.ascontiguousarray(drf).reshape(-1, V)
    u = rng.random(len(flat)).astype(np.float32)
    want, cm, tm = oracle.sample(flat, T, 0, p, u, margins=True)
    got = sv.spec_sample(to_dev(flat), to_dev(u), T, 0, p, workspace="auto").cpu().numpy()
    assert compare_samples(want, got, cm, tm)["hard"] == 0
    # the law of the emitted token (strip law mode)
    tg = np.ascontiguousarray(tgt[:, :G]).reshape(-1, V)
    tokl = tok.reshape(-1).astype(np.int32)
    wl = oracle.law(tg, flat, tokl, T, 0, p)
    ps, beta, px, qx = sv.spec_law(to_dev(tg), to_dev(flat), to_dev(tokl), T, 0, p)
    torch.cuda.synchronize()
    near = np.zeros(len(tg), bool)
    for r in range(len(tg)):
        for z in (tg[r], flat[r]):
            _, mg, _ = oracle.distribution(np.ascontiguousarray(z), T, 0, p)
            near[r] |= mg < 1e-6
    for name, got_l in (("p_spec", ps), ("beta", beta), ("p_x", px), ("q_x", qx)):
        err = np.abs(got_l.cpu().numpy().astype(np.float64) - wl[name])[~near]
        assert err.max() <= 1e-5, (name, err.max())


# Full-size workloads: GPU on the whole batch in the benchmark's launch
# configuration, the oracle on a sample of rows.
FULL = [
    (1, 1.0, 50, 0.9, 64),
    (2, 0.8, 0, 0.95, 12),
    (3, 1.0, 0, 1.0, 512),
    (4, 0.7, 100, 0.9, 12),
    (0, 0.0, 0, 1.0, 1),
    (0, 1.0, 0, 1.0, 1),
]


# The two largest workloads, on 2 input sets x 128 oracle rows (>= 256 rows
# and several hundred draws each), in the benchmark's launch configuration.
@pytest.mark.parametrize("wid,T,k,p", [(2, 0.8, 0, 0.95), (4, 0.7, 100, 0.9)])
def test_parity_full_size_many_rows(wid, T, k, p):
    w = W.WORKLOADS[wid]
    tot = {"rows": 0, "draws": 0, "near": 0, "disagree": 0, "hard": 0}
    for s in range(2):
        batch = W.make_batch(w, 1000 * wid + 11 + s)
        rows = np.random.default_rng(wid + 10 * s).choice(w.B, size=128, replace=False)
        rows.sort()
        tok = draft_tokens_for(batch, T, k, p)
        g = run_gpu(batch, tok, T, k, p, workspace="auto")
        o = run_oracle(batch, tok, T, k, p, rows=rows)
        info = compare(o, g, rows=rows)
        for key in tot:
            tot[key] += info[key]
        del batch
    print(f"full-size parity, workload {wid}: {tot}")
    assert tot["rows"] >= 256 and tot["hard"] == 0
    assert tot["disagree"] <= 1e-4 * tot["draws"] or tot["disagree"] == 0


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("wid,T,k,p,nrows", FULL)
def test_parity_full_size(wid, T, k, p, nrows, path):
    w = W.WORKLOADS[wid]
    batch = W.make_batch(w, 1000 * wid + 1)
    rows = np.random.default_rng(wid).choice(w.B, size=min(nrows, w.B), replace=False)
    rows.sort()
    tok = draft_tokens_for(batch, T, k, p)
    g = run_gpu(batch, tok, T, k, p, **PATHS[path])
    o = run_oracle(batch, tok, T, k, p, rows=rows)
    info = compare(o, g, rows=rows)
    assert info["hard"] == 0


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V,T", [(1024, 1.0), (1024, 0.0), (777, 1.0), (777, 0.0), (64, 0.7)])
def test_small_vocab_dtypes(V, T, dtype, path):
    """The warp-per-row kernel's range: 16-byte loads when a lane's 32
    logits fit (V = 1024), element loads for a ragged last lane (V = 777),
    bf16 and fp32, greedy and sampling, ragged gamma per row."""
    batch = case(3, 41 + V, B=96, V=V, dtype=dtype)
    rng = np.random.default_rng(V)
    batch["gamma_per_row"] = rng.integers(0, batch["workload"].gamma_max + 1,
                                          size=96).astype(np.int32)
    info, g, o = parity(batch, T, 0, 1.0, **PATHS[path])
    assert info["hard"] == 0


@pytest.mark.parametrize("V", [20011, 60011])
@pytest.mark.parametrize("top_p", [0.8, 0.9, 0.95])
def test_topp_wide_nucleus_paths(V, top_p):
    """Top-p alone on flat laws (N(0, 3^2) logits): nuclei of several hundred
    to a few thousand tokens exceed what the pieces publish, so the decider
    extends its lists downwards from the strip, rescans the strip whole, or
    falls back to the slice-wide selection; results must not change.  The
    diagnostics count the extensions and rescans (word 3)."""
    import speculative_decoding_verify_03_gb300 as sv
    import torch
    batch = case(0, 300 + V % 97, B=8, V=V, gamma_max=3)
    T = 1.0
    tok = draft_tokens_for(batch, T, 0, top_p)
    w = batch["workload"]
    P = sv.make_params(to_dev(batch["target"])[:, :, : w.V], to_dev(batch["draft"])[:, :, : w.V],
                       T, 0, top_p)
    ws = torch.zeros(sv.workspace_bytes(P), dtype=torch.uint8, device="cuda")
    g = run_gpu(batch, tok, T, 0, top_p, workspace=ws)
    o = run_oracle(batch, tok, T, 0, top_p)
    info = compare(o, g)
    assert info["hard"] == 0
    diag = sv.read_diagnostics(ws)
    if top_p >= 0.9:
        assert diag[3] + diag[0] > 0, diag  # the lists had to grow
