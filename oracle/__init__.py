"""fp64 CPU oracle for speculative-sampling verification (ctypes binding).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke``
and by the CPU-baseline leg of ``bench.py``; the product path never touches
it.  The C source (``spec_oracle.c``) shares no code with the CUDA library.

Arrays: logits are numpy ``float32`` or ``uint16`` (raw bfloat16 bit
patterns) with a contiguous last (vocabulary) axis; tokens ``int32``;
uniforms ``float32`` of shape ``[B, gamma_max + 1, 2]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_HDR = os.path.join(_HERE, "spec_oracle.h")
_LIB = os.path.join(_HERE, "libspecoracle.so")

F32, BF16 = 0, 1
BAD_TOKEN, BAD_LOGIT, NO_FINITE, Q_ZERO, BAD_GAMMA, BAD_UNIFORM = (1, 2, 4, 8, 16, 32)
ERROR_MASK = BAD_TOKEN | BAD_LOGIT | NO_FINITE | BAD_GAMMA | BAD_UNIFORM


class Params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("gamma_max", ctypes.c_int32), ("V", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("temperature", ctypes.c_double),
        ("top_k", ctypes.c_int32), ("top_p", ctypes.c_double),
        ("t_pos_stride", ctypes.c_int64), ("t_row_stride", ctypes.c_int64),
        ("d_pos_stride", ctypes.c_int64), ("d_row_stride", ctypes.c_int64),
    ]


class RowDiag(ctypes.Structure):
    _fields_ = [
        ("accept_margin", ctypes.c_double), ("cdf_margin", ctypes.c_double),
        ("topp_margin", ctypes.c_double), ("residual_mass", ctypes.c_double),
        ("n_tests", ctypes.c_int32), ("n_draws", ctypes.c_int32),
        ("fallback_p", ctypes.c_int32), ("pad", ctypes.c_int32),
    ]


DIAG_DTYPE = np.dtype([
    ("accept_margin", "f8"), ("cdf_margin", "f8"), ("topp_margin", "f8"),
    ("residual_mass", "f8"), ("n_tests", "i4"), ("n_draws", "i4"),
    ("fallback_p", "i4"), ("pad", "i4"),
])
assert DIAG_DTYPE.itemsize == ctypes.sizeof(RowDiag)

_lock = threading.Lock()


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with the system C compiler (plain -O2, IEEE math)."""
    stale = (not os.path.exists(out)) or any(
        os.path.getmtime(p) > os.path.getmtime(out) for p in (src, _HDR))
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall",
                        "-Wextra", "-fno-fast-math", "-I", _HERE, src, "-o", tmp, "-lm"],
                       check=True)
        os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_distribution.argtypes = [vp, i32, i32, dbl, i32, dbl, vp, vp]
    lib.oracle_distribution.restype = i32
    lib.oracle_verify_rows.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(Params),
                                       i32, i32, vp, vp, vp, vp, vp, vp]
    lib.oracle_verify_rows.restype = None
    lib.oracle_sample_rows.argtypes = [vp, i32, i64, i32, i32, dbl, i32, dbl, vp, vp, vp, vp]
    lib.oracle_sample_rows.restype = None
    return lib


_default = None


def _load():
    global _default
    with _lock:
        if _default is None:
            _default = _bind(build())
    return _default


def _ptr(a):
    return None if a is None else a.ctypes.data


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {a.dtype}")


def _check_last_contiguous(a: np.ndarray):
    if a.ndim and a.shape[-1] > 1 and a.strides[-1] != a.itemsize:
        raise ValueError("the vocabulary axis must be contiguous")


def distribution(z: np.ndarray, temperature: float, top_k: int = 0, top_p: float = 1.0,
                 lib=None):
    """Filtered tempered softmax of one row.  Returns (prob[V], topp_margin, status)."""
    z = np.ascontiguousarray(z)
    V = z.shape[-1]
    prob = np.zeros(V, np.float64)
    margin = np.zeros(1, np.float64)
    st = (lib or _load()).oracle_distribution(_ptr(z), _dtype_code(z), V, float(temperature),
                                     int(top_k), float(top_p), _ptr(prob), _ptr(margin))
    return prob, float(margin[0]), int(st)


def sample(logits: np.ndarray, temperature: float, top_k: int, top_p: float,
           u: np.ndarray, lib=None, threads: int | None = None, margins: bool = False):
    """One draw per row of ``logits[n, V]`` from its filtered law (argmax if T == 0).
    Rows are split over ``threads`` host threads (default: all cores).

    With ``margins=True`` returns ``(tokens, cdf_margin, topp_margin)``: per
    row, the distance of u from the ends of the chosen CDF interval (in units
    of the total weight) and the top-p margin of the row's law (+inf where
    there is none)."""
    _check_last_contiguous(logits)
    n, V = logits.shape
    u = np.ascontiguousarray(u, dtype=np.float32).reshape(n)
    out = np.empty(n, np.int32)
    cm = np.empty(n, np.float64)
    tm = np.empty(n, np.float64)
    L = lib or _load()
    rs = logits.strides[0] // logits.itemsize
    code = _dtype_code(logits)
    nt = max(1, min(threads or (os.cpu_count() or 1), n))
    step = (n + nt - 1) // nt

    def run(s):
        m = min(n, s + step) - s
        if m > 0:
            L.oracle_sample_rows(logits.ctypes.data + s * logits.strides[0], code, rs, m, V,
                                 float(temperature), int(top_k), float(top_p),
                                 u.ctypes.data + 4 * s, out.ctypes.data + 4 * s,
                                 cm.ctypes.data + 8 * s, tm.ctypes.data + 8 * s)

    if nt > 1:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(run, range(0, n, step)))
    else:
        run(0)
    if margins:
        return out, cm, tm
    return out


def verify(target: np.ndarray, draft: np.ndarray, draft_tokens: np.ndarray,
           uniforms: np.ndarray, temperature: float, top_k: int = 0,
           top_p: float = 1.0, gamma_per_row: np.ndarray | None = None,
           rows=None, threads: int = 1, lib=None) -> dict:
    """Verify rows of a batch.  ``target[B, gamma_max+1, V]``, ``draft[B, gamma_max, V]``
    (any row / position strides, contiguous vocabulary axis).

    Returns a dict of numpy arrays over all B rows (rows outside ``rows`` are
    left at -2): accepted_len, next_token, row_status, p_draft, q_draft, diag.
    """
    for a in (target, draft):
        _check_last_contiguous(a)
    B, G1, V = target.shape
    gm = G1 - 1
    if draft.shape[0] != B or draft.shape[1] != gm or draft.shape[2] != V:
        raise ValueError("draft must be [B, gamma_max, V]")
    if target.dtype != draft.dtype:
        raise TypeError("target and draft must share a dtype")
    draft_tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, gm)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, gm + 1, 2)
    if gamma_per_row is not None:
        gamma_per_row = np.ascontiguousarray(gamma_per_row, dtype=np.int32).reshape(B)
    isz = target.itemsize
    P = Params(B=B, gamma_max=gm, V=V, dtype=_dtype_code(target),
               temperature=float(temperature), top_k=int(top_k), top_p=float(top_p),
               t_pos_stride=target.strides[1] // isz, t_row_stride=target.strides[0] // isz,
               d_pos_stride=(draft.strides[1] // isz) if gm else V,
               d_row_stride=draft.strides[0] // isz)
    acc = np.full(B, -2, np.int32)
    nxt = np.full(B, -2, np.int32)
    st = np.full(B, -2, np.int32)
    pd = np.full((B, gm), np.nan, np.float32)
    qd = np.full((B, gm), np.nan, np.float32)
    diag = np.zeros(B, DIAG_DTYPE)
    lib = lib or _load()
    if rows is None:
        spans = [(0, B)]
    else:
        rows = np.asarray(rows, dtype=np.int64)
        spans = [(int(r), int(r) + 1) for r in rows]
    if threads > 1 and rows is None and B > 1:
        step = (B + threads * 4 - 1) // (threads * 4)
        spans = [(s, min(B, s + step)) for s in range(0, B, step)]

    def run(span):
        lib.oracle_verify_rows(_ptr(target), _ptr(draft), _ptr(draft_tokens), _ptr(uniforms),
                               _ptr(gamma_per_row), ctypes.byref(P), span[0], span[1],
                               _ptr(acc), _ptr(nxt), _ptr(st), _ptr(pd), _ptr(qd), _ptr(diag))

    if threads > 1 and len(spans) > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(run, spans))
    else:
        for s in spans:
            run(s)
    return {"accepted_len": acc, "next_token": nxt, "row_status": st,
            "p_draft": pd, "q_draft": qd, "diag": diag}


class Oracle:
    """The oracle API bound to one compiled library (the default build, or a
    variant compiled from another source file, e.g. by the mutation tests)."""

    def __init__(self, path: str | None = None):
        self.lib = _load() if path is None else _bind(path)

    def distribution(self, *a, **k):
        return distribution(*a, lib=self.lib, **k)

    def sample(self, *a, **k):
        return sample(*a, lib=self.lib, **k)

    def verify(self, *a, **k):
        return verify(*a, lib=self.lib, **k)


def commit(accepted_len, next_token, draft_tokens, seq, seq_len, seq_capacity,
           gamma_per_row=None, aimd=None) -> dict:
    """The step after the verify, row by row in plain Python: append the
    accepted draft tokens and the next token to each sequence ("Prepare
    speculative sampling", steps 3-4: the tokens are concatenated to the
    sequence), the key/value length both models keep (the context plus the
    accepted drafts), and the next draft length of an additive-increase /
    multiplicative-decrease controller ("CS3602_FINAL_SpeDec", 更多实现, the
    dynamic gamma; its constants are parameters: aimd = (gamma_min,
    gamma_max, increase, decrease), the decrease product in float32).

    Returns new arrays: seq, seq_len, kv_len, gamma_next (None without aimd).
    Inputs are not modified.
    """
    acc = np.asarray(accepted_len, np.int64)
    nxt = np.asarray(next_token, np.int64)
    B = acc.shape[0]
    drafts = np.asarray(draft_tokens, np.int32).reshape(B, -1)
    gm = drafts.shape[1]
    seq = np.array(seq, np.int32, copy=True)
    L0 = np.asarray(seq_len, np.int64)
    gam = (np.full(B, gm, np.int64) if gamma_per_row is None
           else np.asarray(gamma_per_row, np.int64))
    new_len = np.zeros(B, np.int32)
    kv = np.zeros(B, np.int32)
    gnext = None if aimd is None else np.zeros(B, np.int32)
    for b in range(B):
        g = int(gam[b])
        L, a, t = int(L0[b]), int(acc[b]), int(nxt[b])
        valid = 0 <= g <= gm and 0 <= a <= g and t >= 0 and L >= 0
        if valid:
            new_tokens = [int(x) for x in drafts[b, :a]] + [t]
            room = max(0, seq_capacity - L)
            kept = new_tokens[:room]
            for j, x in enumerate(kept):
                seq[b, L + j] = x
            new_len[b] = L + len(kept)
            kv[b] = min(L + a, L + len(kept))
        else:
            new_len[b] = L
            kv[b] = L
        if aimd is not None:
            gmin, gmax, inc, dec = aimd
            gc = min(max(g, 0), gm)
            if valid and a == gc:
                want = gc + inc
            else:
                want = int(np.floor(np.float32(gc) * np.float32(dec)))
            gnext[b] = min(max(want, gmin), gmax)
    return {"seq": seq, "seq_len": new_len, "kv_len": kv, "gamma_next": gnext}


def law(target: np.ndarray, draft: np.ndarray, tokens, temperature: float, top_k: int = 0,
        top_p: float = 1.0) -> dict:
    """The emitted-token law of the speculative sampler, row by row in fp64
    ("CS3602_FINAL_SpeDec", section 2 困惑度测试 (PPL)): with the filtered
    tempered laws p (target row) and q (draft row), the acceptance rate
    beta = sum min(p, q) and R = sum max(0, p - q), the token x is emitted
    with probability min(p(x), q(x)) + (1 - beta) max(0, p(x) - q(x)) / R
    (min(p(x), q(x)) when R = 0).  target, draft: [n, V] (float32 or raw
    bfloat16 uint16); tokens: [n].  Returns p_spec, beta, p_x, q_x (float64;
    NaN for a token outside [0, V) or a row in error)."""
    n, V = target.shape
    out = {k: np.full(n, np.nan) for k in ("p_spec", "beta", "p_x", "q_x")}
    for r in range(n):
        p, _, st_p = distribution(np.ascontiguousarray(target[r]), temperature, top_k, top_p)
        q, _, st_q = distribution(np.ascontiguousarray(draft[r]), temperature, top_k, top_p)
        if st_p or st_q:
            continue
        beta = float(np.minimum(p, q).sum())
        R = float(np.maximum(p - q, 0.0).sum())
        out["beta"][r] = beta
        x = int(tokens[r])
        if not 0 <= x < V:
            continue
        ps = min(p[x], q[x])
        if R > 0.0:
            ps += (1.0 - beta) * max(p[x] - q[x], 0.0) / R
        out["p_spec"][r], out["p_x"][r], out["q_x"][r] = ps, p[x], q[x]
    return out


def cascade(levels, draft_tokens, uniforms, temperature: float, top_k: int = 0,
            top_p: float = 1.0, gamma_per_row=None, threads: int = 1) -> dict:
    """Verification of a multi-stage draft cascade ("CS3602_FINAL_SpeDec",
    更多实现: several draft models in a chain, each one drafting for the next
    larger one, as the levels of a cache hierarchy serve each other).

    ``levels[0]`` is the target and ``levels[L]`` the smallest draft model,
    L = len(levels) - 1 >= 1.  The smallest model drew ``draft_tokens[B,
    gamma_max]`` from its laws ``levels[L][B, gamma_max, V]``; every other
    level l ran one forward pass over the same drafts, ``levels[l][B,
    gamma_max + 1, V]`` (position i scores the token after drafts 0..i-1).

    The pages give no algorithm; this is the plainest reading.  Stage k = 0 ..
    L-1 is one verify step of the tokens presented to it, with draft laws
    from level s = L - k and target laws from level s - 1 and its own
    uniforms ``uniforms[k]`` ([B, gamma_max + 1, 2]).  Per row, n tokens are
    presented (gamma_b at stage 0):
      - a rejection at slot a < n puts the resampled token at slot a, and the
        next stage sees the n = a + 1 tokens 0..a (a resample differs from
        the rejected token, so every later position's laws, computed after
        the original drafts, are then out of context and never read);
      - when all n are accepted, the bonus draw at slot n is kept only at
        the last stage and only if no stage resampled (the presented tokens
        are then the original drafts, the context of level 0's slot-n law);
        otherwise it is discarded and the next stage sees the same n.
    Every stage's output follows its target level's law at every slot it
    reaches (the verify step's guarantee, whatever the presented tokens'
    law, as long as each one follows the draft level's law given the ones
    before it, which the stage below ensures), so the cascade's output
    follows the target's law.

    Returns out_tokens [B, gamma_max + 1] (-1 beyond out_len), out_len [B]
    (0 for a row in error), stage_accepted [L, B] (-1 for stages after the
    row's error), row_status [B] (the stages' bits, or-ed), margin [L, B]
    (the smallest of the stage's acceptance, CDF and top-p margins; +inf
    after an error) and draws (acceptance tests plus draws, all stages)."""
    L = len(levels) - 1
    if L < 1:
        raise ValueError("a cascade needs the target and at least one draft level")
    d = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    B, gm = d.shape
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(L, B, gm + 1, 2)
    n = (np.full(B, gm, np.int64) if gamma_per_row is None
         else np.asarray(gamma_per_row, np.int64).copy())
    tok = np.full((B, gm + 1), -1, np.int32)
    tok[:, :gm] = d
    resampled = np.zeros(B, bool)
    err = np.zeros(B, bool)
    status = np.zeros(B, np.int32)
    stage_acc = np.full((L, B), -1, np.int32)
    margin = np.full((L, B), np.inf)
    draws = 0
    rows = np.arange(B)
    for k in range(L):
        s = L - k
        last = k == L - 1
        draft = levels[s][:, :gm]
        r = verify(levels[s - 1], draft, tok[:, :gm], uniforms[k], temperature, top_k, top_p,
                   gamma_per_row=n.astype(np.int32), threads=threads)
        a = r["accepted_len"].astype(np.int64)
        t = r["next_token"]
        live = ~err
        status[live] |= r["row_status"][live]
        bad = live & ((r["row_status"] & ERROR_MASK) != 0)
        err |= bad
        ok = live & ~bad
        stage_acc[k, live] = a[live]
        dg = r["diag"]
        m = np.minimum(np.minimum(dg["accept_margin"], dg["cdf_margin"]), dg["topp_margin"])
        margin[k, live] = m[live]
        draws += int(dg["n_tests"][live].sum() + dg["n_draws"][live].sum())
        rej = ok & (a < n)
        tok[rows[rej], a[rej]] = t[rej]
        n[rej] = a[rej] + 1
        resampled |= rej
        bonus = ok & (a == n) & (~resampled) & last
        tok[rows[bonus], n[bonus]] = t[bonus]
        n[bonus] += 1
    n[err] = 0
    out = np.full((B, gm + 1), -1, np.int32)
    for b in range(B):
        out[b, : n[b]] = tok[b, : n[b]]
    return {"out_tokens": out, "out_len": n.astype(np.int32), "stage_accepted": stage_acc,
            "row_status": status, "margin": margin, "draws": draws}
