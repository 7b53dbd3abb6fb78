"""The law of the GPU verify step at scale: over 10^6 rows that share one
set of target and draft logits (row stride 0) but draw their own draft
tokens and uniforms, the first emitted token (the draft token when it is
accepted, else the resampled one) must follow the filtered target law p,
whatever the draft law q is ("CS3602_FINAL_SpeDec", section "2.
困惑度测试(PPL)": the output law of speculative sampling is p).  A chi-square
test against p at level 1e-3 (fixed seeds), for every kernel selection;
tokens outside p's support must never appear."""
import numpy as np
import pytest
import scipy.stats

import oracle
from speculative_decoding_verify_03_gb300 import workloads as W

pytestmark = pytest.mark.gpu

N_ROWS = 1_000_000
CHUNK = 100_000

CASES = [
    # (V, dtype, temperature, top_k, top_p, spread of the logits)
    (1024, "f32", 1.0, 0, 1.0, 1.5),      # unfiltered
    (4096, "f32", 1.0, 50, 0.9, 3.0),     # top-k then top-p
    (3001, "bf16", 0.7, 100, 0.9, 2.0),   # bf16, ragged vocabulary
    (2048, "f32", 0.8, 0, 0.95, 2.0),     # top-p alone
]


@pytest.fixture(scope="module")
def sv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_03_gb300 as m
    m.build()
    oracle.build()
    return m


@pytest.mark.parametrize("path", ["cluster", "auto", "nows"])
@pytest.mark.parametrize("ci", range(len(CASES)))
def test_first_token_follows_p(sv, ci, path):
    import torch
    V, dtype, T, k, p, spread = CASES[ci]
    rng = np.random.default_rng(700 + ci)
    zt = (rng.normal(size=(2, V)) * spread).astype(np.float32)
    zd = (0.6 * zt[:1] + rng.normal(size=(1, V)) * spread * 0.8).astype(np.float32)
    if dtype == "bf16":
        zt_bits, zd_bits = W.f32_to_bf16_bits(zt), W.f32_to_bf16_bits(zd)
        zt = (zt_bits.astype(np.uint32) << 16).view(np.float32)
        zd = (zd_bits.astype(np.uint32) << 16).view(np.float32)
        dev_t = torch.from_numpy(zt_bits.view(np.int16)).view(torch.bfloat16).cuda()
        dev_d = torch.from_numpy(zd_bits.view(np.int16)).view(torch.bfloat16).cuda()
    else:
        dev_t = torch.from_numpy(zt).cuda()
        dev_d = torch.from_numpy(zd).cuda()
    p_law, _, st_p = oracle.distribution(zt[0], T, k, p)
    q_law, _, st_q = oracle.distribution(zd[0], T, k, p)
    assert st_p == 0 and st_q == 0
    counts = np.zeros(V, np.int64)
    kw = {"cluster": dict(workspace=None, kernel="cluster"), "auto": dict(workspace="auto"),
          "nows": dict(workspace=None)}[path]
    for c0 in range(0, N_ROWS, CHUNK):
        n = min(CHUNK, N_ROWS - c0)
        tok = rng.choice(V, size=(n, 1), p=q_law / q_law.sum()).astype(np.int32)
        uni = rng.random((n, 2, 2), dtype=np.float32)
        tgt = dev_t.unsqueeze(0).expand(n, 2, V)
        drf = dev_d.unsqueeze(0).expand(n, 1, V)
        acc, nxt = sv.spec_verify(tgt, drf, torch.from_numpy(tok).cuda(),
                                  torch.from_numpy(uni).cuda(), T, k, p, **kw)
        acc, nxt = acc.cpu().numpy(), nxt.cpu().numpy()
        first = np.where(acc >= 1, tok[:, 0], nxt)
        assert first.min() >= 0 and first.max() < V
        counts += np.bincount(first, minlength=V)
    support = p_law > 0
    assert counts[~support].sum() == 0, "tokens outside the support of p were emitted"
    exp = p_law[support] * N_ROWS
    obs = counts[support].astype(np.float64)
    # pool the bins with small expectations into one
    small = exp < 5.0
    if small.any():
        exp = np.append(exp[~small], exp[small].sum())
        obs = np.append(obs[~small], obs[small].sum())
    chi2 = float(((obs - exp) ** 2 / exp).sum())
    dof = max(1, len(exp) - 1)
    pval = float(scipy.stats.chi2.sf(chi2, dof))
    print(f"V {V} {dtype} T {T} k {k} p {p} {path}: chi2 {chi2:.1f} dof {dof} p-value {pval:.3g}")
    assert pval > 1e-3, (chi2, dof, pval)
