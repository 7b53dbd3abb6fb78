"""The post-verify step on the GPU against the oracle, bit-exact: random
rows (error rows, ragged gamma, rows at and past the sequence capacity),
and the verify step followed by the commit step on a workload batch."""
import numpy as np
import pytest

import oracle
from gpu_util import draft_tokens_for, run_gpu, to_dev
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


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("with_gamma", [False, True])
def test_commit_random(sv, seed, with_gamma):
    import torch
    rng = np.random.default_rng(seed)
    B, gm, cap = 1000, 8, 40
    drafts = rng.integers(0, 50000, size=(B, gm)).astype(np.int32)
    gam = rng.integers(0, gm + 1, size=B).astype(np.int32)
    gam[::97] = -1      # invalid draft lengths
    gam[5::101] = gm + 1
    acc = np.array([rng.integers(0, max(g, 0) + 1) for g in gam], np.int32)
    nxt = rng.integers(0, 50000, size=B).astype(np.int32)
    nxt[::13] = -1      # error rows of the verify step
    L = rng.integers(0, cap + 1, size=B).astype(np.int32)
    L[::17] = cap       # full rows
    seq = rng.integers(0, 50000, size=(B, cap)).astype(np.int32)
    aimd = (1, 12, 1, 0.5) if seed % 2 == 0 else (0, 6, 3, 0.7)
    g_arg = gam if with_gamma else None
    want = oracle.commit(acc, nxt, drafts, seq, L, cap, gamma_per_row=g_arg, aimd=aimd)
    dseq, dlen = to_dev(seq), to_dev(L)
    kv, gn = sv.spec_commit(to_dev(acc), to_dev(nxt), to_dev(drafts), dseq, dlen,
                            gamma_per_row=to_dev(gam) if with_gamma else None, aimd=aimd)
    torch.cuda.synchronize()
    assert np.array_equal(dseq.cpu().numpy(), want["seq"])
    assert np.array_equal(dlen.cpu().numpy(), want["seq_len"])
    assert np.array_equal(kv.cpu().numpy(), want["kv_len"])
    assert np.array_equal(gn.cpu().numpy(), want["gamma_next"])


def test_verify_then_commit(sv):
    import torch
    from dataclasses import replace
    w = replace(W.WORKLOADS[4], B=24, V=30011)
    batch = W.make_batch(w, 77)
    T, k, p = w.temperature, w.top_k, w.top_p
    tok = draft_tokens_for(batch, T, k, p)
    g = run_gpu(batch, tok, T, k, p, debug=False)  # its parity is pinned elsewhere
    cap = 64
    seq = np.zeros((w.B, cap), np.int32)
    L = np.full(w.B, 10, np.int32)
    gam = batch["gamma_per_row"]
    aimd = (1, w.gamma_max, 1, 0.5)
    want = oracle.commit(g["accepted_len"], g["next_token"], tok, seq, L, cap,
                         gamma_per_row=gam, aimd=aimd)
    dseq, dlen = to_dev(seq), to_dev(L)
    kv, gn = sv.spec_commit(to_dev(g["accepted_len"]), to_dev(g["next_token"]), to_dev(tok),
                            dseq, dlen, gamma_per_row=to_dev(gam), aimd=aimd)
    torch.cuda.synchronize()
    assert np.array_equal(dseq.cpu().numpy(), want["seq"])
    assert np.array_equal(dlen.cpu().numpy(), want["seq_len"])
    assert np.array_equal(kv.cpu().numpy(), want["kv_len"])
    assert np.array_equal(gn.cpu().numpy(), want["gamma_next"])
