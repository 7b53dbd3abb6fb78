"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function declared in include/*.h, and rejects invalid arguments
before touching the device."""
import ctypes
import glob
import os
import re

import pytest

import speculative_decoding_verify_03_gb300 as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    sv.build()
    return sv.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(spec_\w+)\s*\(", src, re.M):
            names.add(m.group(1))
    return names


def test_exports_every_declared_function(L):
    names = declared_functions()
    assert {"spec_verify", "spec_sample", "spec_verify_workspace_size", "spec_status_string",
            "spec_read_diagnostics"} <= names
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in range(5):
        assert L.spec_status_string(code)
    assert b"unknown" in L.spec_status_string(99)


def _params(**kw):
    base = dict(B=2, gamma_max=2, V=100, dtype=0, temperature=1.0, top_p=1.0, top_k=0, flags=0,
                target_pos_stride=100, target_row_stride=300, draft_pos_stride=100,
                draft_row_stride=200, gamma_per_row=None, cluster_size=0, list_capacity=0)
    base.update(kw)
    return sv.SpecParams(**base)


P = ctypes.c_void_p


def _call(L, params, target=1 << 20, draft=1 << 21, tokens=1 << 22, uni=1 << 23, acc=1 << 24,
          nxt=1 << 25, ws=None, ws_bytes=0):
    # fake (never dereferenced) device addresses: validation fails first
    return L.spec_verify(P(target), P(draft), P(tokens), P(uni),
                         ctypes.byref(params) if params is not None else None,
                         P(acc), P(nxt), None, P(ws) if ws else None, ws_bytes, None)


@pytest.mark.parametrize("bad", [
    dict(V=0), dict(V=-3), dict(V=(1 << 24) + 1), dict(B=-1), dict(gamma_max=-1),
    dict(dtype=2), dict(temperature=-1.0), dict(temperature=float("nan")),
    dict(temperature=float("inf")), dict(temperature=1e-38), dict(top_p=0.0),
    dict(top_p=-0.5), dict(top_p=float("nan")), dict(flags=2), dict(cluster_size=3),
    dict(cluster_size=16), dict(list_capacity=-1), dict(target_pos_stride=-1),
])
def test_invalid_params_rejected(L, bad):
    assert _call(L, _params(**bad)) == 1  # SPEC_ERR_INVALID_ARG


def test_invalid_pointers_rejected(L):
    assert _call(L, None) == 1
    assert _call(L, _params(), target=0) == 1
    assert _call(L, _params(), draft=0) == 1
    assert _call(L, _params(), tokens=0) == 1
    assert _call(L, _params(), uni=0) == 1
    assert _call(L, _params(), acc=0) == 1
    assert _call(L, _params(), nxt=0) == 1
    # greedy reads neither draft logits nor uniforms
    p = _params(temperature=0.0, B=0)
    assert _call(L, p, draft=0, uni=0) == 0


def test_workspace_checks(L):
    assert L.spec_verify_workspace_size(None) >= 16
    assert _call(L, _params(), ws=(1 << 26) + 8, ws_bytes=64) == 3  # misaligned
    assert _call(L, _params(), ws=1 << 26, ws_bytes=4) == 3         # too small


def test_empty_batch_is_noop(L):
    assert _call(L, _params(B=0), target=0, nxt=0, acc=0) in (0, 1)
    assert _call(L, _params(B=0)) == 0


def test_workspace_size_follows_kernel_selection(L):
    """Vocabularies up to 1024, greedy or unfiltered: the row kernels (the
    diagnostics words, plus, when sampling, the list of rows handed to the
    second kernel: 16 bytes a row after a 32-byte head); greedy, top-k or
    top-p beyond that: the strip kernel's exchange area;
    SPEC_FLAG_CLUSTER_KERNEL, and unfiltered sampling beyond 1024: the
    cluster kernel (diagnostics only)."""
    diag = L.spec_verify_workspace_size(None)
    size = lambda **kw: L.spec_verify_workspace_size(ctypes.byref(_params(**kw)))
    assert size(V=1024) == 32 + 2 * 16                   # unfiltered (B=2), row kernels
    assert size(V=1024, B=4096) == 32 + 4096 * 16
    assert size(V=1024, temperature=0.0, top_k=50) == diag  # greedy ignores filters
    assert size(V=1024, temperature=0.0) == diag         # greedy: nothing deferred
    assert size(V=1024, top_k=1024) == 32 + 2 * 16       # top-k >= V is off
    assert size(V=1025, temperature=0.0) > diag          # greedy, strip kernel
    assert size(V=1024, top_k=50) > diag                 # top-k, strip kernel
    assert size(V=5000, top_k=50, flags=sv.SPEC_FLAG_CLUSTER_KERNEL) == diag
    assert size(V=5000, top_p=0.9) > diag                # top-p alone: strip kernel
    assert size(V=1024, top_p=0.9) > diag
    assert size(V=5000) == diag                          # unfiltered: cluster kernel
    assert size(V=5000, top_p=0.9, flags=sv.SPEC_FLAG_CLUSTER_KERNEL) == diag


def _commit(L, B=4, gm=3, acc=1 << 20, nxt=1 << 21, tok=1 << 22, gam=None, seq=1 << 23,
            stride=16, cap=16, slen=1 << 24, kv=None, gn=None, aimd=None):
    # fake (never dereferenced) device addresses: validation fails first
    return L.spec_commit(B, gm, P(acc), P(nxt), P(tok) if tok else None, P(gam) if gam else None,
                         P(seq), stride, cap, P(slen), P(kv) if kv else None,
                         P(gn) if gn else None, ctypes.byref(aimd) if aimd else None, None)


def test_commit_argument_checks(L):
    ok = sv.SpecAimd(1, 8, 1, 0.5)
    assert _commit(L, B=-1) == 1
    assert _commit(L, gm=-1) == 1
    assert _commit(L, cap=-1) == 1
    assert _commit(L, stride=8, cap=16) == 1  # rows would overlap
    assert _commit(L, acc=0) == 1
    assert _commit(L, nxt=0) == 1
    assert _commit(L, seq=0) == 1
    assert _commit(L, slen=0) == 1
    assert _commit(L, tok=0) == 1              # drafts needed when gamma_max > 0
    assert _commit(L, gn=1 << 25) == 1         # gamma_next without a controller
    for bad in (sv.SpecAimd(-1, 8, 1, 0.5), sv.SpecAimd(4, 2, 1, 0.5), sv.SpecAimd(1, 8, -1, 0.5),
                sv.SpecAimd(1, 8, 1, 1.5), sv.SpecAimd(1, 8, 1, float("nan"))):
        assert _commit(L, gn=1 << 25, aimd=bad) == 1
    assert _commit(L, B=0, acc=0, nxt=0, seq=0, slen=0, gn=1 << 25, aimd=ok) == 0  # no-op


def test_law_argument_checks(L):
    def law(**kw):
        return L.spec_law(P(1 << 20), P(1 << 21), P(1 << 22), ctypes.byref(_params(**kw)),
                          P(1 << 23), None, None, None, None)
    # filtered laws are accepted (checked with B=0: nothing is launched on
    # these fake addresses)
    assert law(top_k=5, B=0) == 0
    assert law(top_p=0.5, B=0) == 0
    assert law(temperature=0.0) == 2  # a point mass
    assert law(V=0) == 1
    assert law(target_row_stride=10) == 1
    assert law(B=0) == 0


def _cascade(L, params, n_levels=3, levels=(1 << 20, 1 << 21, 1 << 22), tok=1 << 23,
             uni=1 << 24, out=1 << 25, olen=1 << 26, ws=1 << 27, ws_bytes=1 << 20):
    # fake (never dereferenced) device addresses: validation fails first
    arr = (ctypes.c_void_p * max(len(levels), 1))(*levels) if levels is not None else None
    return L.spec_cascade_verify(arr, n_levels, P(tok) if tok else None,
                                 P(uni) if uni else None,
                                 ctypes.byref(params) if params is not None else None,
                                 P(out) if out else None, P(olen) if olen else None, None, None,
                                 P(ws) if ws else None, ws_bytes, None)


def test_cascade_argument_checks(L):
    """Every stage's arguments are checked before the first launch; the
    workspace holds the cascade's own state (the presented tokens and five
    per-row words, each array on a 256-byte boundary) before the verify
    step's part."""
    p = _params()
    state = 256 * 6  # B=2, gamma_max=2: every array fits one 256-byte block
    for n in (2, 3, 5):
        assert L.spec_cascade_workspace_size(ctypes.byref(p), n) == \
            state + L.spec_verify_workspace_size(ctypes.byref(p))
    assert L.spec_cascade_workspace_size(ctypes.byref(p), 1) == 0
    assert L.spec_cascade_workspace_size(None, 3) == 0
    big = _params(B=1000, gamma_max=8)
    assert L.spec_cascade_workspace_size(ctypes.byref(big), 3) == \
        32000 + 5 * 4096 + L.spec_verify_workspace_size(ctypes.byref(big))
    assert _cascade(L, None) == 1
    assert _cascade(L, p, n_levels=1, levels=(1 << 20,)) == 1
    assert _cascade(L, p, levels=None) == 1
    assert _cascade(L, p, levels=(1 << 20, 0, 1 << 22)) == 1   # a middle level missing
    assert _cascade(L, p, tok=0) == 1
    assert _cascade(L, p, uni=0) == 1                          # sampling needs uniforms
    assert _cascade(L, p, out=0) == 1
    assert _cascade(L, p, olen=0) == 1
    assert _cascade(L, _params(top_p=0.0)) == 1                # the verify step's checks
    assert _cascade(L, _params(dtype=3)) == 1
    assert _cascade(L, p, ws=0) == 3
    assert _cascade(L, p, ws=(1 << 27) + 16) == 3              # not 256-byte aligned
    assert _cascade(L, p, ws_bytes=state - 4) == 3
    assert _cascade(L, p, levels=(1 << 20, 1 << 21, 0)) == 1   # sampling reads the smallest
    assert _cascade(L, _params(B=0)) == 0


def test_law_ws_argument_checks(L):
    """The workspace form of spec_law: its size is the strip kernel's for
    filtered laws and 0 otherwise; its argument checks are spec_law's."""
    size = lambda **kw: L.spec_law_workspace_size(ctypes.byref(_params(**kw)))
    assert size(V=50304, top_k=50, top_p=0.9) > 0
    assert size(V=50304, top_p=0.9) > 0
    assert size(V=50304) == 0                  # unfiltered: the row kernel
    assert size(V=50304, top_k=50, temperature=0.0) == 0
    assert L.spec_law_workspace_size(None) == 0

    def law(ws=None, **kw):
        return L.spec_law_ws(P(1 << 20), P(1 << 21), P(1 << 22), ctypes.byref(_params(**kw)),
                             P(1 << 23), None, None, None, P(ws) if ws else None, 1 << 20, None)
    assert law(top_k=5, B=0) == 0
    assert law(temperature=0.0, top_k=5) == 2  # a point mass
    assert law(V=0) == 1
    assert law(target_row_stride=10) == 1
    assert law(list_capacity=-1, top_k=5) == 1


def test_sample_ws_argument_checks(L):
    """The workspace form of spec_sample: the size is the verify step's for
    the same shape; its checks are spec_sample's (gamma_max 0)."""
    p = _params(gamma_max=0, top_k=50)
    assert L.spec_sample_workspace_size(ctypes.byref(p)) == L.spec_verify_workspace_size(ctypes.byref(p))

    def smp(ws=None, ws_bytes=0, **kw):
        return L.spec_sample_ws(P(1 << 20), P(1 << 21), ctypes.byref(_params(**kw)), P(1 << 22),
                                None, P(ws) if ws else None, ws_bytes, None)
    assert smp(gamma_max=1) == 1                       # a sampler has no drafts
    assert smp(gamma_max=0, V=0) == 1
    assert smp(gamma_max=0, ws=(1 << 26) + 8, ws_bytes=4096) == 3  # misaligned
    assert smp(gamma_max=0, B=0) == 0
