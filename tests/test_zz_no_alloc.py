"""spec_verify_noalloc (the library's fixed device block as the workspace:
no caller workspace, no allocation) against spec_verify on the same inputs,
on two consecutive calls; and the rejection of a problem whose workspace
exceeds the block."""
import numpy as np
import pytest

from gpu_util import case, draft_tokens_for, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_03_gb300 as m
    m.build()
    return m


def _inputs(batch, tokens):
    w = batch["workload"]
    gam = to_dev(batch["gamma_per_row"]) if batch["gamma_per_row"] is not None else None
    return (to_dev(batch["target"])[:, :, : w.V], to_dev(batch["draft"])[:, :, : w.V],
            to_dev(np.ascontiguousarray(tokens, np.int32)), to_dev(batch["uniforms"]), gam)


@pytest.mark.parametrize("wid,over,T,k,p", [
    (1, dict(B=16, V=9001), 1.0, 50, 0.9),           # strip kernel (top-k)
    (4, dict(B=12, V=30011), 0.7, 100, 0.9),         # strip kernel, ragged, bf16
    (0, dict(B=8, V=5003), 0.0, 0, 1.0),             # strip kernel (greedy)
    (2, dict(B=8, V=30011, gamma_max=5), 0.8, 0, 0.95),  # strip kernel (top-p only)
])
def test_matches_spec_verify_on_consecutive_calls(sv, wid, over, T, k, p):
    import torch
    batch = case(wid, 500 + wid, **over)
    tok = draft_tokens_for(batch, T, k, p)
    tgt, drf, tk, uni, gam = _inputs(batch, tok)
    want = sv.spec_verify(tgt, drf, tk, uni, T, k, p, gamma_per_row=gam, debug=True)
    torch.cuda.synchronize()
    want = [x.cpu().numpy() for x in want[:2]] + [want[2][n].cpu().numpy() for n in sorted(want[2])]
    for _ in range(2):
        got = sv.spec_verify_noalloc(tgt, drf, tk, uni, T, k, p, gamma_per_row=gam, debug=True)
        torch.cuda.synchronize()
        got = [x.cpu().numpy() for x in got[:2]] + [got[2][n].cpu().numpy() for n in sorted(got[2])]
        for a, b in zip(want, got):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_rejects_a_problem_larger_than_the_block(sv):
    import torch
    B, G, V = 512, 8, 152064  # bf16, top-k 100: a strip workspace of ~114 MB
    tgt = torch.empty((B, G + 1, V), dtype=torch.bfloat16, device="cuda")
    drf = torch.empty((B, G, V), dtype=torch.bfloat16, device="cuda")
    tok = torch.zeros((B, G), dtype=torch.int32, device="cuda")
    uni = torch.zeros((B, G + 1, 2), dtype=torch.float32, device="cuda")
    P = sv.make_params(tgt, drf, 0.7, 100, 0.9)
    assert sv.workspace_bytes(P) > 64 << 20
    with pytest.raises(sv.SpecError, match="WORKSPACE"):
        sv.spec_verify_noalloc(tgt, drf, tok, uni, 0.7, 100, 0.9)
