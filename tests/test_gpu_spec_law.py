"""spec_law (the emitted-token law, for scoring) against the fp64 oracle:
probabilities within 1e-5 absolute, on fp32 and bf16 rows of several
vocabulary sizes and temperatures; NaN for out-of-range tokens and rows in
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
